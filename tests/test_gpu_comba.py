"""GPU parity of comba_decode_step (through the C ABI) against the CPU oracle.

Tolerance: max |gpu - oracle| / max |oracle| <= 1e-4 for the fp32 state and for o with an fp32
store; a bf16 o must equal the round-to-nearest-even of the oracle or a bf16 neighbour of it.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
import oracle
from gpu_util import dev, host, library, sample_heads
from parity import bf16_neighbours_ok, max_rel_err, rel_frobenius

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()


def _dev_token(t):
    b16 = torch.bfloat16
    return (dev(t["q"], b16), dev(t["k"], b16), dev(t["v"], b16), dev(t["p"], b16),
            dev(t["beta"], b16), dev(t["g_log"], torch.float32))


def _oracle_chain(B, H, K, V, steps, seed):
    """16 warm-up steps from zero (state stored in fp32), then the measured step."""
    g = gi.rng(seed)
    scale = K ** -0.5
    S = np.zeros((B, H, K, V))
    toks = []
    for _ in range(steps):
        t = gi.comba_decode_token(g, B, H, K, V)
        toks.append(t)
        S, _ = oracle.comba_decode(S, t["q"], t["k"], t["v"], t["p"], t["beta"], t["g_log"], scale)
        S = S.astype(np.float32).astype(np.float64)
    t = gi.comba_decode_token(g, B, H, K, V)
    return S, toks, t


# The Comba spec's correctness shapes (B, H, K, V), with the full oracle.
@pytest.mark.parametrize("B,H,K,V", [(8, 4, 128, 128), (16, 2, 64, 128), (4, 8, 128, 64),
                                     (32, 4, 64, 64)])
def test_spec_correctness_shapes(B, H, K, V):
    scale = K ** -0.5
    S, _, t = _oracle_chain(B, H, K, V, 16, seed=B + H + K + V)
    ref_S, ref_o = oracle.comba_decode(S, t["q"], t["k"], t["v"], t["p"], t["beta"], t["g_log"],
                                       scale)
    Sd = dev(S, torch.float32)
    S1, o32 = gdn.comba_decode_step(Sd, *_dev_token(t), scale=scale, o_dtype=torch.float32)
    assert max_rel_err(host(S1), ref_S) <= TOL
    assert max_rel_err(host(o32), ref_o) <= TOL
    assert rel_frobenius(host(S1), ref_S) <= 1e-6
    _, obf = gdn.comba_decode_step(Sd, *_dev_token(t), scale=scale, o_dtype=torch.bfloat16)
    assert bf16_neighbours_ok(host(obf), ref_o)
    assert np.array_equal(host(Sd), S)   # functional: state untouched
    # in place
    S2, _ = gdn.comba_decode_step(Sd, *_dev_token(t), scale=scale, state_new=Sd)
    assert S2.data_ptr() == Sd.data_ptr()
    assert max_rel_err(host(Sd), ref_S) <= TOL


def test_full_workload_chain_sampled_heads():
    # B=256, H=32, K=V=128: the GPU runs the 17-step chain from zero over every head; the oracle
    # runs it for a sample of heads.
    c = gi.COMBA_DECODE
    B, H, K, V = c["B"], c["H"], c["K"], c["V"]
    scale = K ** -0.5
    g = gi.rng(0)
    toks = [gi.comba_decode_token(g, B, H, K, V) for _ in range(c["warmup"] + 1)]
    heads = sample_heads(np.random.default_rng(2), B, H, 24)
    bufs = [torch.zeros((B, H, K, V), dtype=torch.float32, device="cuda"),
            torch.empty((B, H, K, V), dtype=torch.float32, device="cuda")]
    o = torch.empty((B, H, V), dtype=torch.float32, device="cuda")
    cur = 0
    ref = {h: np.zeros((K, V)) for h in heads}
    ref_o = {}
    for t in toks:
        gdn.comba_decode_step(bufs[cur], *_dev_token(t), scale=scale, state_new=bufs[1 - cur], o=o)
        cur = 1 - cur
        for (b, h) in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            Sn, on = oracle.comba_decode(ref[(b, h)][None, None], t["q"][sl], t["k"][sl],
                                         t["v"][sl], t["p"][sl], t["beta"][sl], t["g_log"][sl],
                                         scale)
            ref[(b, h)] = Sn[0, 0].astype(np.float32).astype(np.float64)
            ref_o[(b, h)] = on[0, 0]
    S_h, o_h = host(bufs[cur]), host(o)
    for h in heads:
        assert max_rel_err(S_h[h], ref[h]) <= TOL, h
        assert max_rel_err(o_h[h], ref_o[h]) <= TOL, h


def test_empty_batch_is_a_no_op():
    S = torch.zeros((0, 2, 128, 128), dtype=torch.float32, device="cuda")
    q = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((0, 2), dtype=torch.bfloat16, device="cuda")
    S1, o = gdn.comba_decode_step(S, q, q, q, q, b, torch.zeros((0, 2), device="cuda"))
    assert S1.shape == S.shape and o.shape == (0, 2, 128)


# The Comba spec's quick measure shapes (B, H, K, V), including K = 64: the GPU runs the whole step,
# the oracle a sample of heads.
@pytest.mark.parametrize("B,H,K,V", [(256, 16, 128, 128), (128, 32, 128, 128), (512, 16, 64, 128)])
def test_spec_measure_shapes_sampled(B, H, K, V):
    scale = K ** -0.5
    g = gi.rng(B + H + K)
    S = (g.standard_normal((B, H, K, V)) * 0.1).astype(np.float32)
    t = gi.comba_decode_token(g, B, H, K, V)
    S1, o = gdn.comba_decode_step(dev(S, torch.float32), *_dev_token(t), scale=scale,
                                  o_dtype=torch.float32)
    S_h, o_h = host(S1), host(o)
    for (b, h) in sample_heads(np.random.default_rng(3), B, H, 16):
        sl = (slice(b, b + 1), slice(h, h + 1))
        Sn, on = oracle.comba_decode(S[sl], t["q"][sl], t["k"][sl], t["v"][sl], t["p"][sl],
                                     t["beta"][sl], t["g_log"][sl], scale)
        assert max_rel_err(S_h[b, h], Sn[0, 0]) <= TOL
        assert max_rel_err(o_h[b, h], on[0, 0]) <= TOL
