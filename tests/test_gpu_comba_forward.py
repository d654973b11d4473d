"""GPU parity of comba_forward (the Comba recurrence over T tokens, through the C ABI) against the
CPU oracle (oracle.comba_forward, T chained Comba steps).

Tolerance: max |gpu - oracle| / max |oracle| <= 1e-4 for the final fp32 state and for o with an
fp32 store, per head; a bf16 o must equal the round-to-nearest-even of the oracle or a bf16
neighbour of it.  The state is carried in fp32 on the GPU and in fp64 in the oracle.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import gated_deltanet_delta_gb300 as gdn
import oracle
from gpu_util import dev, host, library
from parity import bf16_neighbours_ok, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()


def _dev(x):
    b16, f32 = torch.bfloat16, torch.float32
    return {n: dev(x[n], dt) for n, dt in (("q", b16), ("k", b16), ("v", b16), ("p", b16),
                                           ("beta", b16), ("g_log", f32), ("state", f32))}


def _run(d, scale, o_dtype):
    state = d["state"].clone()
    o = gdn.comba_forward(state, d["q"], d["k"], d["v"], d["p"], d["beta"], d["g_log"], scale=scale,
                          o_dtype=o_dtype)
    torch.cuda.synchronize()
    return host(state), host(o)


@pytest.mark.parametrize("B,T,H,K,V", [(2, 5, 3, 128, 128), (3, 7, 2, 64, 128), (2, 4, 2, 128, 64),
                                       (4, 3, 2, 64, 64), (1, 33, 2, 128, 128)])
def test_small_shapes(B, T, H, K, V):
    x = gi.comba_forward_inputs(gi.rng(B * 100 + T + K + V), B, T, H, K, V)
    scale = K ** -0.5
    ref_S, ref_o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["p"], x["beta"],
                                        x["g_log"], scale)
    d = _dev(x)
    S, o32 = _run(d, scale, torch.float32)
    for b in range(B):
        for h in range(H):
            assert max_rel_err(S[b, h], ref_S[b, h]) <= TOL, (b, h)
            assert max_rel_err(o32[b, :, h], ref_o[b, :, h]) <= TOL, (b, h)
    S2, obf = _run(d, scale, torch.bfloat16)
    assert np.array_equal(S, S2)
    assert bf16_neighbours_ok(obf, ref_o)


def test_no_tokens_keeps_the_state():
    x = gi.comba_forward_inputs(gi.rng(7), 2, 0, 2, 128, 128)
    d = _dev(x)
    S, o = _run(d, 128 ** -0.5, torch.float32)
    assert o.shape == (2, 0, 2, 128) and np.array_equal(S, x["state"].astype(np.float64))


def test_one_token_matches_the_decode_step():
    x = gi.comba_forward_inputs(gi.rng(8), 4, 1, 4, 128, 128)
    d = _dev(x)
    scale = 128 ** -0.5
    S, o = _run(d, scale, torch.float32)
    S1, o1 = gdn.comba_decode_step(d["state"], d["q"][:, 0].contiguous(), d["k"][:, 0].contiguous(),
                                   d["v"][:, 0].contiguous(), d["p"][:, 0].contiguous(),
                                   d["beta"][:, 0].contiguous(), d["g_log"][:, 0].contiguous(),
                                   scale=scale, o_dtype=torch.float32)
    assert max_rel_err(S, host(S1)) <= 1e-6 and max_rel_err(o[:, 0], host(o1)) <= 1e-6


def test_benchmark_workload_sampled_heads():
    # B=256, T=8, H=32, K=V=128: the whole call on the GPU, the oracle on sampled heads
    c = gi.COMBA_FORWARD
    B, T, H, K, V = c["B"], c["T"], c["H"], c["K"], c["V"]
    x = gi.comba_forward_inputs(gi.rng(0), B, T, H, K, V)
    scale = K ** -0.5
    d = _dev(x)
    S, o = _run(d, scale, torch.float32)
    for b, h in [(0, 0), (17, 5), (128, 31), (255, 16), (255, 31)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ref_S, ref_o = oracle.comba_forward(x["state"][b:b + 1, h:h + 1], x["q"][sl], x["k"][sl],
                                            x["v"][sl], x["p"][sl], x["beta"][sl], x["g_log"][sl], scale)
        assert max_rel_err(S[b, h], ref_S[0, 0]) <= TOL, (b, h)
        assert max_rel_err(o[b, :, h], ref_o[0, :, 0]) <= TOL, (b, h)


def test_gate_extremes():
    # g = -inf (the state wiped at that token), g = 0 (no decay), beta = 0 and beta = 1, over three
    # chunks of tokens with a ragged tail
    B, T, H, K, V = 2, 19, 3, 128, 128
    x = gi.comba_forward_inputs(gi.rng(11), B, T, H, K, V)
    x["g_log"][:, 3, 0] = -np.inf
    x["g_log"][:, 9:12, 1] = -np.inf
    x["g_log"][:, :, 2] = 0.0
    x["beta"][0, 5:9, :] = 0.0
    x["beta"][1, 12:, :] = 1.0
    scale = K ** -0.5
    ref_S, ref_o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["p"], x["beta"],
                                        x["g_log"], scale)
    assert np.isfinite(ref_S).all() and np.isfinite(ref_o).all()
    S, o = _run(_dev(x), scale, torch.float32)
    assert np.isfinite(S).all() and np.isfinite(o).all()
    for b in range(B):
        for h in range(H):
            assert max_rel_err(S[b, h], ref_S[b, h]) <= TOL, (b, h)
            assert max_rel_err(o[b, :, h], ref_o[b, :, h]) <= TOL, (b, h)
