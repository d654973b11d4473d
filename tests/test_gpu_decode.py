"""GPU parity of gdn_decode_step (through the C ABI) against the CPU oracle.

Tolerance: max |gpu - oracle| / max |oracle| <= 1e-4 for the fp32 state and for y computed with an
fp32 store; a bf16 y must equal the round-to-nearest-even of the oracle or a bf16 neighbour of it.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
import oracle
from gpu_util import dev, host, library, sample_heads
from parity import bf16_neighbours_ok, max_rel_err, max_rel_err_slices

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()


def _dev_token(t):
    return (dev(t["q"], torch.bfloat16), dev(t["k"], torch.bfloat16), dev(t["v"], torch.bfloat16),
            dev(t["g"], torch.float32), dev(t["beta"], torch.bfloat16))


def _gpu_step(S, t, scale, out=None, y_dtype=torch.float32):
    q, k, v, g, beta = _dev_token(t)
    return gdn.gdn_decode_step(S, q, k, v, g, beta, scale=scale, state_out=out, y_dtype=y_dtype)


def test_tiny_workload_warmed_by_oracle():
    # B=1, Hk=2, Hv=4, Dk=Dv=64: 16 oracle warm-up steps from zero, then one measured step.
    c = gi.GDN_DECODE_TINY
    B, Hk, Hv, Dk, Dv = c["B"], c["Hk"], c["Hv"], c["Dk"], c["Dv"]
    scale = Dk ** -0.5
    g = gi.rng(0)
    S = np.zeros((B, Hv, Dv, Dk))
    toks = []
    for _ in range(c["warmup"]):
        t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
        toks.append(t)
        S, _ = oracle.gdn_decode(S, t["q"], t["k"], t["v"], t["g"], t["beta"], scale)
        S = S.astype(np.float32).astype(np.float64)   # the state is stored in fp32
    t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
    ref_S, ref_y = oracle.gdn_decode(S, t["q"], t["k"], t["v"], t["g"], t["beta"], scale)

    Sd = dev(S, torch.float32)
    S1, y32 = _gpu_step(Sd, t, scale)
    assert max_rel_err(host(S1), ref_S) <= TOL
    assert max_rel_err(host(y32), ref_y) <= TOL
    assert max_rel_err_slices(host(S1), ref_S, 2) <= TOL   # per (batch row, value head)
    assert max_rel_err_slices(host(y32), ref_y, 2) <= TOL
    _, ybf = _gpu_step(Sd, t, scale, y_dtype=torch.bfloat16)
    assert bf16_neighbours_ok(host(ybf), ref_y)
    assert np.array_equal(host(Sd), S)   # functional: the input state is untouched

    # the whole 17-step chain on the GPU from zero
    Sg = torch.zeros((B, Hv, Dv, Dk), dtype=torch.float32, device="cuda")
    for tt in toks + [t]:
        Sg, yg = _gpu_step(Sg, tt, scale)
    assert max_rel_err(host(Sg), ref_S) <= TOL
    assert max_rel_err(host(yg), ref_y) <= TOL


def test_batched_workload_chain_sampled_heads():
    # B=64, Hk=16, Hv=32, Dk=Dv=128: the GPU runs 16 warm-up steps + the measured step from zero
    # over every head; the oracle runs the same chain for a sample of heads.  Then 100 steps that
    # reuse the last draw, state ping-ponged between two buffers as the benchmark times it.
    c = gi.GDN_DECODE_BATCHED
    B, Hk, Hv, Dk, Dv = c["B"], c["Hk"], c["Hv"], c["Dk"], c["Dv"]
    scale = Dk ** -0.5
    g = gi.rng(0)
    toks = [gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv) for _ in range(c["warmup"] + 1)]
    heads = sample_heads(np.random.default_rng(1), B, Hv, 24)

    bufs = [torch.zeros((B, Hv, Dv, Dk), dtype=torch.float32, device="cuda"),
            torch.empty((B, Hv, Dv, Dk), dtype=torch.float32, device="cuda")]
    y = torch.empty((B, Hv, Dv), dtype=torch.float32, device="cuda")
    cur = 0
    ref = {h: np.zeros((Dv, Dk)) for h in heads}

    def oracle_step(t):
        out = {}
        for (b, hv) in heads:
            hk = hv // (Hv // Hk)
            Sn, yh = oracle.gdn_decode(ref[(b, hv)][None, None], t["q"][b:b + 1, hk:hk + 1],
                                       t["k"][b:b + 1, hk:hk + 1], t["v"][b:b + 1, hv:hv + 1],
                                       t["g"][b:b + 1, hv:hv + 1], t["beta"][b:b + 1, hv:hv + 1],
                                       scale)
            ref[(b, hv)] = Sn[0, 0].astype(np.float32).astype(np.float64)
            out[(b, hv)] = yh[0, 0]
        return out

    for t in toks:
        gdn.gdn_decode_step(bufs[cur], *_dev_token(t), scale=scale, state_out=bufs[1 - cur], y=y)
        cur = 1 - cur
        ref_y = oracle_step(t)
    S_h, y_h = host(bufs[cur]), host(y)
    for h in heads:
        assert max_rel_err(S_h[h], ref[h]) <= TOL, h
        assert max_rel_err(y_h[h], ref_y[h]) <= TOL, h

    last = _dev_token(toks[-1])
    for _ in range(100):
        gdn.gdn_decode_step(bufs[cur], *last, scale=scale, state_out=bufs[1 - cur], y=y)
        cur = 1 - cur
        ref_y = oracle_step(toks[-1])
    S_h, y_h = host(bufs[cur]), host(y)
    for h in heads:
        assert max_rel_err(S_h[h], ref[h]) <= TOL, h
        assert max_rel_err(y_h[h], ref_y[h]) <= TOL, h
    # bf16 readout of the last step
    ybf = torch.empty((B, Hv, Dv), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(bufs[1 - cur], *last, scale=scale, state_out=bufs[cur], y=ybf)
    ybf_h = host(ybf)
    assert all(bf16_neighbours_ok(ybf_h[h], ref_y[h]) for h in heads)


@pytest.mark.parametrize("B,Hk,Hv,Dk,Dv", [(3, 2, 6, 128, 40), (2, 1, 3, 128, 200),
                                           (1, 4, 4, 64, 130), (5, 3, 3, 64, 7),
                                           (2, 2, 8, 128, 128)])
@pytest.mark.parametrize("in_place", [False, True])
def test_ragged_shapes_and_in_place(B, Hk, Hv, Dk, Dv, in_place):
    g = gi.rng(B * 1000 + Dv)
    S = (g.standard_normal((B, Hv, Dv, Dk)) * 0.3).astype(np.float32)
    t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
    scale = 0.37
    ref_S, ref_y = oracle.gdn_decode(S, t["q"], t["k"], t["v"], t["g"], t["beta"], scale)
    Sd = dev(S, torch.float32)
    S1, y = _gpu_step(Sd, t, scale, out=Sd if in_place else None)
    assert (S1.data_ptr() == Sd.data_ptr()) == in_place
    assert max_rel_err(host(S1), ref_S) <= TOL
    assert max_rel_err(host(y), ref_y) <= TOL


def test_empty_batch_is_a_no_op():
    S = torch.zeros((0, 4, 128, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    S1, y = gdn.gdn_decode_step(S, q, q, v, torch.zeros((0, 4), device="cuda"),
                                torch.zeros((0, 4), dtype=torch.bfloat16, device="cuda"))
    assert S1.shape == S.shape and y.shape == (0, 4, 128)


def test_rejects_indivisible_heads_without_writing():
    S = torch.zeros((1, 3, 128, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 3, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(S, 5.0)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_decode_step(S, q, q, v, torch.zeros((1, 3), device="cuda"),
                            torch.zeros((1, 3), dtype=torch.bfloat16, device="cuda"), state_out=out)
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    assert bool(torch.all(out == 5.0))


@pytest.mark.parametrize("B,Hk,Hv,Dv", [(3, 2, 4, 256), (2, 1, 2, 100)])
def test_head_dim_256(B, Hk, Hv, Dv):
    g = gi.rng(B + Dv)
    S = (g.standard_normal((B, Hv, Dv, 256)) * 0.2).astype(np.float32)
    t = gi.gdn_decode_token(g, B, Hk, Hv, 256, Dv)
    ref_S, ref_y = oracle.gdn_decode(S, t["q"], t["k"], t["v"], t["g"], t["beta"], 256 ** -0.5)
    S1, y = _gpu_step(dev(S, torch.float32), t, 256 ** -0.5)
    assert max_rel_err(host(S1), ref_S) <= TOL
    assert max_rel_err(host(y), ref_y) <= TOL


@pytest.mark.parametrize("Dk", [64, 128, 256])
def test_pooled_decode_gathers_and_scatters_its_slots(Dk):
    # batch row b updates pool slot cache_indices[b] in place; other slots stay bitwise untouched;
    # an out-of-range slot is flagged and its row skipped
    B, Hk, Hv, Dv, pool = 4, 2, 4, 64, 7
    g = gi.rng(40 + Dk)
    P = (g.standard_normal((pool, Hv, Dv, Dk)) * 0.2).astype(np.float32)
    t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
    idx = np.array([5, 0, 3, 9], dtype=np.int64)   # 9 is outside the pool
    scale = Dk ** -0.5
    Pd = dev(P, torch.float32)
    y = torch.full((B, Hv, Dv), -7.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v, gg, beta = _dev_token(t)
    gdn.gdn_decode_step_pooled(Pd, dev(idx, torch.int64), q, k, v, gg, beta, scale=scale, y=y,
                               dev_status=status)
    assert int(status.item()) & gdn.STATUS_BAD_CACHE_INDEX
    Ph, yh = host(Pd), host(y)
    for b, slot in enumerate(idx[:3]):
        ref_S, ref_y = oracle.gdn_decode(P[slot][None], t["q"][b:b + 1], t["k"][b:b + 1],
                                         t["v"][b:b + 1], t["g"][b:b + 1], t["beta"][b:b + 1], scale)
        assert max_rel_err(Ph[slot], ref_S[0]) <= TOL
        assert max_rel_err(yh[b], ref_y[0]) <= TOL
    assert np.all(yh[3] == -7.0)
    for s in (1, 2, 4, 6):
        assert np.array_equal(Ph[s], P[s].astype(np.float64))


@pytest.mark.parametrize("B,T,Hk,Hv,Dk,Dv", [(2, 1, 2, 4, 128, 128), (3, 37, 1, 2, 128, 100),
                                             (1, 16, 2, 2, 64, 64), (2, 9, 1, 1, 256, 40),
                                             (2, 33, 1, 2, 64, 48), (1, 20, 1, 1, 256, 72)])
@pytest.mark.parametrize("in_place", [False, True])
def test_multi_token_steps_equal_a_chain_of_steps(B, T, Hk, Hv, Dk, Dv, in_place):
    # [gated_delta.rs] mt_gated_delta_chunk: the decode recurrence wrapped in a loop over t
    g = gi.rng(B * 100 + T + Dk)
    S = (g.standard_normal((B, Hv, Dv, Dk)) * 0.2).astype(np.float32)
    toks = [gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv) for _ in range(T)]
    stack = {n: np.stack([t[n] for t in toks], axis=1) for n in ("q", "k", "v", "g", "beta")}
    scale = Dk ** -0.5
    ref = S.astype(np.float64)
    ys = []
    for t in toks:
        ref, y = oracle.gdn_decode(ref, t["q"], t["k"], t["v"], t["g"], t["beta"], scale)
        ys.append(y)
    ref_y = np.stack(ys, axis=1)
    Sd = dev(S, torch.float32)
    S1, y = gdn.gdn_decode_multi(Sd, dev(stack["q"], torch.bfloat16), dev(stack["k"], torch.bfloat16),
                                 dev(stack["v"], torch.bfloat16), dev(stack["g"], torch.float32),
                                 dev(stack["beta"], torch.bfloat16), scale=scale,
                                 state_out=Sd if in_place else None, y_dtype=torch.float32)
    assert max_rel_err(host(S1), ref) <= TOL
    assert max_rel_err(host(y), ref_y) <= TOL
