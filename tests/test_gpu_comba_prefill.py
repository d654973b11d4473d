"""GPU parity of comba_prefill_chunked (through the C ABI) against the sequential CPU oracle of the
Comba recurrence (oracle.comba_forward, one sequence at a time).

Tolerances (max |gpu - oracle| / max |oracle| per tensor): outputs (bf16) <= 5e-3, final state
<= 2e-3, as for the GDN prefill.  Pool slots that no sequence references stay bitwise untouched.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
import oracle
from gpu_util import dev, host, library
from parity import max_rel_err, max_rel_err_slices

pytestmark = pytest.mark.gpu
OUT_TOL, STATE_TOL = 5e-3, 2e-3
SENTINEL = -1000.0
H = 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()


def _to_dev(x):
    bf, f32, i64 = torch.bfloat16, torch.float32, torch.int64
    return {n: dev(x[n], dt) for n, dt in (("q", bf), ("k", bf), ("v", bf), ("p", bf), ("beta", bf),
                                           ("g_log", f32), ("state_pool", f32), ("cache_indices", i64),
                                           ("cu_seqlens", i64))}


def _gpu(d, scale, ws_bytes=None):
    T = d["v"].shape[0]
    out = torch.full((T, H, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None if ws_bytes is None else torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    gdn.comba_prefill_chunked(d["q"], d["k"], d["v"], d["p"], d["beta"], d["g_log"], d["state_pool"],
                              d["cache_indices"], d["cu_seqlens"], 64, scale=scale, out=out, workspace=ws,
                              dev_status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def _check_all(x, d, out, scale):
    pool = host(d["state_pool"])
    o = host(out)
    cu, ci = x["cu_seqlens"], [int(c) for c in x["cache_indices"]]
    for n, slot in enumerate(ci):
        a, b = int(cu[n]), int(cu[n + 1])
        if b == a:
            assert np.array_equal(pool[slot], x["state_pool"][slot].astype(np.float64)), n
            continue
        sl = slice(a, b)
        S, o_ref = oracle.comba_forward(x["state_pool"][slot][None], x["q"][None, sl], x["k"][None, sl],
                                        x["v"][None, sl], x["p"][None, sl], x["beta"][None, sl],
                                        x["g_log"][None, sl], scale)
        assert max_rel_err(o[sl], o_ref[0]) <= OUT_TOL, n
        assert max_rel_err(pool[slot], S[0]) <= STATE_TOL, n
        # and per head of the sequence
        assert max_rel_err_slices(np.moveaxis(o[sl], 1, 0), np.moveaxis(o_ref[0], 1, 0), 1) <= OUT_TOL, n
        assert max_rel_err_slices(pool[slot], S[0], 1) <= STATE_TOL, n
    for s in range(pool.shape[0]):
        if s not in ci:
            assert np.array_equal(pool[s], x["state_pool"][s].astype(np.float64)), s


def _split_scratch_bytes(N, T):
    cap = (T + 63) // 64 + N
    return (8 * 3 * H + (cap // 2) * H) * 65536


@pytest.mark.parametrize("mild", [False, True])
@pytest.mark.parametrize("seqlens", [[1], [63], [65, 100], [64, 0, 130, 1, 7]])
def test_small_varlen(seqlens, mild):
    x = gi.comba_prefill_inputs(gi.rng(700 + sum(seqlens) + mild), seqlens, H, 128, 128,
                                pool=len(seqlens) + 3, mild=mild)
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


@pytest.mark.parametrize("seqlens", [[1300 + 20, 900, 700, 40], [2000, 3], [64 * 8]])
def test_long_sequences_split_and_unsplit(seqlens):
    # the schedule splits the long sequences (their second halves run from a zero state and from the
    # identity and are combined by the fix-up kernel); without the split scratch nothing is split
    N = len(seqlens)
    x = gi.comba_prefill_inputs(gi.rng(800 + sum(seqlens)), seqlens, H, 128, 128, pool=N + 2, mild=True)
    scale = 128 ** -0.5
    full = gdn.gdn_prefill_workspace_size(N, x["T"], H, H, 128, 128, 64)
    outs, pools = [], []
    for ws_bytes in (full, full - _split_scratch_bytes(N, x["T"])):
        d = _to_dev(x)
        out, st = _gpu(d, scale, ws_bytes)
        assert st == 0
        _check_all(x, d, out, scale)
        outs.append(host(out))
        pools.append(host(d["state_pool"]))
    assert max_rel_err(outs[0], outs[1]) <= OUT_TOL
    assert max_rel_err(pools[0], pools[1]) <= STATE_TOL


@pytest.mark.parametrize("seqlens", [[150, 64], [700]])
@pytest.mark.parametrize("case", ["no_update", "no_decay", "full_decay"])
def test_gate_extremes(case, seqlens):
    # beta = 0: the state only decays; g = 0: no decay (gamma_L = 1 on every chunk); g = -100: the
    # chunk decay underflows to 0 in fp32 and the update overwrites the state
    x = gi.comba_prefill_inputs(gi.rng(900 + sum(seqlens)), seqlens, H, 128, 128, pool=2, mild=True)
    if case == "no_update":
        x["beta"][:] = 0.0
    elif case == "no_decay":
        x["g_log"][:] = 0.0
    else:
        x["g_log"][:] = -100.0
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


def test_read_key_equal_to_write_key_matches_the_gdn_step():
    # With p = k the Comba step is the GDN decode step on the transposed state (S^T, V x K) with
    # gate exp(g): the prefill is checked against the GDN oracle run token by token.
    seqlens = [200, 70]
    x = gi.comba_prefill_inputs(gi.rng(31), seqlens, H, 128, 128, pool=3, mild=True)
    x["p"] = x["k"].copy()
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    o, pool = host(out), host(d["state_pool"])
    cu = x["cu_seqlens"]
    for n, slot in enumerate(int(c) for c in x["cache_indices"]):
        S = x["state_pool"][slot].transpose(0, 2, 1)[None].astype(np.float64)  # [1, H, V, K]
        ys = []
        for t in range(int(cu[n]), int(cu[n + 1])):
            S, y = oracle.gdn_decode(S, x["q"][t][None], x["k"][t][None], x["v"][t][None],
                                     np.exp(x["g_log"][t].astype(np.float64))[None], x["beta"][t][None], scale)
            ys.append(y[0])
        assert max_rel_err(o[int(cu[n]):int(cu[n + 1])], np.stack(ys)) <= OUT_TOL, n
        assert max_rel_err(pool[slot], S[0].transpose(0, 2, 1)) <= STATE_TOL, n


def test_bad_slot_is_flagged_and_skipped():
    x = gi.comba_prefill_inputs(gi.rng(41), [70, 30], H, 128, 128, pool=3)
    x["cache_indices"] = np.array([5, 1], dtype=np.int64)  # 5 is outside the pool of 3
    d = _to_dev(x)
    out, st = _gpu(d, 128 ** -0.5)
    assert st & gdn.STATUS_BAD_CACHE_INDEX
    assert np.all(host(out)[:70] == SENTINEL)
    pool = host(d["state_pool"])
    for s in (0, 2):
        assert np.array_equal(pool[s], x["state_pool"][s].astype(np.float64))
