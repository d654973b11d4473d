"""gdn_prefill_chunked_noalloc: the prefill for callers that cannot allocate device memory (their
device memory belongs to another allocator, or allocation is not allowed where they run).  It uses
the library's fixed 64 MiB device scratch instead of a caller-owned workspace.

The GPU tests run calls in a row through the C ABI, each with a different batch so that whatever an
earlier call left in the shared scratch would show if it were read.  Every call is checked against
the oracle (per sequence, the prefill tolerances) and against gdn_prefill_chunked given a workspace
of exactly 64 MiB: with the same workspace size both take the same split decision and run the same
kernels, so their outputs and pools must agree bit for bit.  One batch has a long sequence that is
split inside the 64 MiB; another is too large for the split scratch but not for the records, so it
runs unsplit.  This file is named to be collected last: it needs nothing from the other tests and
passes alone in a fresh process as well as after them.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
import oracle
from parity import max_rel_err

OUT_TOL, STATE_TOL = 5e-3, 2e-3
SCRATCH = 64 << 20
SCALE = 128 ** -0.5


def _dev(x):
    b16, f32, i64 = torch.bfloat16, torch.float32, torch.int64
    return {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(dt).to("cuda")
            for n, dt in (("q", b16), ("k", b16), ("v", b16), ("a", b16), ("b", b16),
                          ("A_log", f32), ("dt_bias", f32), ("cache_indices", i64),
                          ("cu_seqlens", i64))}


def _run(fn, d, pool, **kw):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fn(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], pool,
             d["cache_indices"], d["cu_seqlens"], 64, scale=SCALE, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def _check_oracle(x, pool_before, out, pool_after):
    """Per sequence: outputs and the final state against the oracle run from pool_before; slots no
    sequence references unchanged bit for bit."""
    pool_ref, out_ref, st = oracle.gdn_prefill(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                                               x["dt_bias"], pool_before, x["cache_indices"],
                                               x["cu_seqlens"], SCALE)
    assert st == 0
    o = out.float().cpu().numpy().astype(np.float64)
    pool = pool_after.cpu().numpy().astype(np.float64)
    cu, ci = x["cu_seqlens"], [int(c) for c in x["cache_indices"]]
    for n, slot in enumerate(ci):
        if cu[n + 1] > cu[n]:
            assert max_rel_err(o[cu[n]:cu[n + 1]], out_ref[cu[n]:cu[n + 1]]) <= OUT_TOL, n
            assert max_rel_err(pool[slot], pool_ref[slot]) <= STATE_TOL, n
    for s in range(pool.shape[0]):
        if s not in ci:
            assert np.array_equal(pool[s], pool_before[s].astype(np.float64)), s


def _both(x, pool_na, pool_ws):
    """One call of each entry point on the same inputs and equal pools; returns the no-alloc
    output after checking it against the oracle and, bit for bit, against the 64 MiB workspace."""
    d = _dev(x)
    before = pool_na.cpu().numpy()
    assert torch.equal(pool_na, pool_ws)
    ws = torch.empty(SCRATCH, dtype=torch.uint8, device="cuda")
    ref = _run(gdn.gdn_prefill_chunked, d, pool_ws, workspace=ws)
    got = _run(gdn.gdn_prefill_chunked_noalloc, d, pool_na)
    _check_oracle(x, before, got, pool_na)
    assert torch.equal(got, ref)
    assert torch.equal(pool_na, pool_ws)
    return got


@pytest.mark.gpu
def test_noalloc_on_calls_in_a_row_matches_the_oracle_and_the_workspace_entry_point():
    gdn.load()
    Hk, Hv, pool_size = 2, 4, 6
    g = gi.rng(2024)
    # call 1: the 1000-token sequence (16 chunks) dominates and is split; its whole workspace,
    # split scratch included, fits the 64 MiB
    x1 = gi.gdn_prefill_inputs(g, [300, 64, 1000, 17], Hk, Hv, 128, 128, pool=pool_size, mild_gates=True)
    # call 2 continues slots 1 and 3 with another batch
    x2 = gi.gdn_prefill_inputs(g, [17, 1000, 130], Hk, Hv, 128, 128, pool=pool_size)
    x2["cache_indices"] = np.array([4, 1, 3], dtype=np.int64)
    assert gdn.gdn_prefill_workspace_size(4, x1["T"], Hk, Hv, 128, 128, 64) <= SCRATCH
    assert gdn.gdn_prefill_workspace_size(3, x2["T"], Hk, Hv, 128, 128, 64) <= SCRATCH
    pool_na = torch.from_numpy(x1["state_pool"]).float().cuda()
    pool_ws = pool_na.clone()
    for x in (x1, x2):
        _both(x, pool_na, pool_ws)


@pytest.mark.gpu
def test_noalloc_runs_unsplit_when_only_the_records_fit():
    gdn.load()
    # one 2944-token sequence with Hv = 16: its records fit the 64 MiB, its split scratch does not
    Hk, Hv = 8, 16
    x = gi.gdn_prefill_inputs(gi.rng(77), [2944], Hk, Hv, 128, 128, pool=2, mild_gates=True)
    lay_full = gdn.gdn_prefill_workspace_size(1, x["T"], Hk, Hv, 128, 128, 64)
    assert lay_full > SCRATCH
    pool_na = torch.from_numpy(x["state_pool"]).float().cuda()
    pool_ws = pool_na.clone()
    _both(x, pool_na, pool_ws)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = gdn.load()
    P = ctypes.c_void_p(1 << 20)
    # T = 65,536 tokens with Hv = 32 needs about 3.4 GB of workspace: rejected before any CUDA call
    need = gdn.gdn_prefill_workspace_size(4, 65536, 16, 32, 128, 128, 64)
    assert need > SCRATCH
    st = lib.gdn_prefill_chunked_noalloc(P, P, P, P, P, P, P, ctypes.c_void_p(1 << 30), 4, P, P, 4, 65536,
                                         16, 32, 128, 128, 64, 0.08, ctypes.c_void_p(1 << 40), P, None)
    assert st == gdn.GDN_ERR_UNSUPPORTED
    assert str(need) in gdn.last_error() and "gdn_prefill_chunked" in gdn.last_error()
    # no sequences: a no-op that touches nothing
    assert lib.gdn_prefill_chunked_noalloc(None, None, None, None, None, None, None, None, 0, None, None,
                                           0, 0, 1, 1, 128, 128, 64, 0.08, None, None, None) == gdn.GDN_OK
