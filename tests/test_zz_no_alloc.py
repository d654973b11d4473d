"""gdn_prefill_chunked_noalloc: the prefill for callers that cannot allocate device memory (their
device memory belongs to another allocator, or allocation is not allowed where they run).  It uses
the library's fixed 64 MiB device scratch instead of a caller-owned workspace.

The GPU test runs two calls in a row through the C ABI, the second with a different batch so that
whatever the first left in the shared scratch would show if it were read, and compares outputs and
final states with gdn_prefill_chunked's on the same inputs, within the prefill parity tolerances.
This file is named to be collected last: it needs nothing from the other tests and passes alone in a
fresh process as well as after them.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
from parity import max_rel_err

OUT_TOL, STATE_TOL = 5e-3, 2e-3
SCRATCH = 64 << 20


def _dev(x):
    b16, f32, i64 = torch.bfloat16, torch.float32, torch.int64
    return {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(dt).to("cuda")
            for n, dt in (("q", b16), ("k", b16), ("v", b16), ("a", b16), ("b", b16),
                          ("A_log", f32), ("dt_bias", f32), ("cache_indices", i64),
                          ("cu_seqlens", i64))}


def _run(fn, d, pool, **kw):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fn(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], pool,
             d["cache_indices"], d["cu_seqlens"], 64, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.float().cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    gdn.load()
    Hk, Hv, pool_size = 2, 4, 6
    g = gi.rng(2024)
    x1 = gi.gdn_prefill_inputs(g, [300, 64, 1000, 17], Hk, Hv, 128, 128, pool=pool_size)
    x2 = gi.gdn_prefill_inputs(g, [17, 1000, 130], Hk, Hv, 128, 128, pool=pool_size)
    x2["cache_indices"] = np.array([4, 1, 3], dtype=np.int64)  # the second call continues slots 1 and 3
    assert gdn.gdn_prefill_workspace_size(4, x1["T"], Hk, Hv, 128, 128, 64) <= SCRATCH
    assert gdn.gdn_prefill_workspace_size(3, x2["T"], Hk, Hv, 128, 128, 64) <= SCRATCH
    pool_ref = torch.from_numpy(x1["state_pool"]).float().cuda()
    pool_na = pool_ref.clone()
    d1, d2 = _dev(x1), _dev(x2)
    for d in (d1, d2):
        ref = _run(gdn.gdn_prefill_chunked, d, pool_ref)
        got = _run(gdn.gdn_prefill_chunked_noalloc, d, pool_na)
        assert max_rel_err(got, ref) <= OUT_TOL
        assert max_rel_err(pool_na.cpu().numpy(), pool_ref.cpu().numpy()) <= STATE_TOL


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
