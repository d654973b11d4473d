"""The prefill's bounded device-side waits, made to run out on purpose (through the C ABI).

Every mbarrier wait of the prefill kernels gives up after a bounded number of polls, sets
GDN_STATUS_TIMEOUT in dev_status and stops its CTA after draining the copies and products it has in
flight.  gdn_prefill_set_wait_limit(1) makes those limits small enough to run out on a healthy GPU:
the call must return, report the timeout, and leave the device usable -- the next call on the same
stream, with the built-in limits restored, must match the oracle.  No fault, trap or hang is
involved: the kernels stop by themselves.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
import oracle
from gpu_util import dev, host, library
from parity import max_rel_err

pytestmark = pytest.mark.gpu
OUT_TOL, STATE_TOL = 5e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()
    yield
    gdn.set_prefill_wait_limit(0)


def _call(x):
    tok, f32, i64 = torch.bfloat16, torch.float32, torch.int64
    d = {n: dev(x[n], dt) for n, dt in (("q", tok), ("k", tok), ("v", tok), ("a", tok), ("b", tok),
                                        ("A_log", f32), ("dt_bias", f32), ("state_pool", f32),
                                        ("cache_indices", i64), ("cu_seqlens", i64))}
    T, Hv = x["T"], x["v"].shape[1]
    out = torch.zeros((T, Hv, 128), dtype=tok, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                            d["state_pool"], d["cache_indices"], d["cu_seqlens"], 64,
                            scale=128 ** -0.5, out=out, dev_status=status)
    torch.cuda.synchronize()
    return d, out, int(status.item())


def test_a_wait_that_runs_out_reports_and_the_next_call_is_exact():
    # one sequence of 300 tokens (5 chunks: no split), one key head, two value heads
    x = gi.gdn_prefill_inputs(gi.rng(41), [300], 1, 2, 128, 128, pool=3, mild_gates=True)
    try:
        gdn.set_prefill_wait_limit(1)
        _, _, st = _call(x)
    finally:
        gdn.set_prefill_wait_limit(0)
    assert st & gdn.STATUS_TIMEOUT, st

    d, out, st = _call(x)  # the same stream, the built-in limits
    assert st == 0
    pool_ref, out_ref, rst = oracle.gdn_prefill(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                                                x["dt_bias"], x["state_pool"], x["cache_indices"],
                                                x["cu_seqlens"], 128 ** -0.5)
    assert rst == 0
    slot = int(x["cache_indices"][0])
    assert max_rel_err(host(out), out_ref) <= OUT_TOL
    assert max_rel_err(host(d["state_pool"])[slot], pool_ref[slot]) <= STATE_TOL
    for s in range(x["state_pool"].shape[0]):
        if s != slot:
            assert np.array_equal(host(d["state_pool"])[s], x["state_pool"][s].astype(np.float64))
