"""GPU parity of gdn_window_fused (through the C ABI) against the CPU oracle.

Tolerance: max |gpu - oracle| / max |oracle| <= 1e-4 for y and the committed state; the committed
conv history is a copy of inputs and must match bit for bit; verify mode must leave state and
hist_out bitwise untouched; a partial commit 0x100|k must equal, bitwise, a k-token commit.
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
TOL = 1e-4
f32 = torch.float32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()


def _dev(x):
    return {k: dev(v, f32) for k, v in x.items()}


def _gpu(d, h_k, commit, hist_out=None, state=None):
    state = d["state"].clone() if state is None else state
    hist_out = torch.full_like(d["hist"], -7.5) if hist_out is None else hist_out
    y = gdn.gdn_window_fused(state, d["hist"], hist_out, d["qkv"], d["alpha"], d["beta"], d["z"],
                             d["conv_w"], d["dt"], d["ssm_a"], d["gamma"], h_k, commit)
    return state, hist_out, y


def _oracle(x, h_k, commit):
    return oracle.gdn_window(x["state"], x["hist"], x["qkv"], x["alpha"], x["beta"], x["z"],
                             x["conv_w"], x["dt"], x["ssm_a"], x["gamma"], h_k, commit,
                             hist_out=np.full(x["hist"].shape, -7.5))


@pytest.mark.parametrize("commit", [0, 1])
def test_full_workload(commit):
    # N=32 sequences, h_k=16, h_v=48, head dim 128, ntok=8: verify and commit.
    c = gi.GDN_WINDOW
    x = gi.gdn_window_inputs(gi.rng(0), c["N"], c["h_k"], c["h_v"], c["D"], c["ntok"])
    d = _dev(x)
    S, ho, y = _gpu(d, c["h_k"], commit)
    rS, rho, ry = _oracle(x, c["h_k"], commit)
    assert max_rel_err(host(y), ry) <= TOL
    # and per (sequence, value head): y [N, ntok, h_v, D], state [N, D, h_v, D]
    assert max_rel_err_slices(np.moveaxis(host(y), 2, 1), np.moveaxis(ry, 2, 1), 2) <= TOL
    if commit:
        assert max_rel_err(host(S), rS) <= TOL
        assert max_rel_err_slices(np.moveaxis(host(S), 2, 1), np.moveaxis(rS, 2, 1), 2) <= TOL
        assert np.array_equal(host(ho), rho)
    else:
        assert np.array_equal(host(S), x["state"].astype(np.float64))
        assert bool(torch.all(ho == -7.5))


@pytest.mark.parametrize("k", [1, 3, 8])
def test_partial_commit_is_bitwise_a_k_token_commit(k):
    N, h_k, h_v, ntok = 3, 2, 6, 8
    x = gi.gdn_window_inputs(gi.rng(10 + k), N, h_k, h_v, 128, ntok)
    d = _dev(x)
    S_p, ho_p, y_p = _gpu(d, h_k, 0x100 | k)
    rS, rho, ry = _oracle(x, h_k, 0x100 | k)
    assert max_rel_err(host(y_p), ry) <= TOL
    assert max_rel_err(host(S_p), rS) <= TOL
    assert np.array_equal(host(ho_p), rho)
    dk = dict(d, qkv=d["qkv"][:, :k].contiguous(), alpha=d["alpha"][:, :k].contiguous(),
              beta=d["beta"][:, :k].contiguous(), z=d["z"][:, :k].contiguous())
    S_k, ho_k, y_k = _gpu(dk, h_k, 1)
    assert torch.equal(S_p, S_k) and torch.equal(ho_p, ho_k)
    assert torch.equal(y_p[:, :k], y_k)


@pytest.mark.parametrize("N,h_k,h_v,ntok,commit", [(1, 1, 1, 1, 1), (2, 2, 5, 3, 1),
                                                   (1, 3, 3, 7, 0x105), (4, 1, 2, 2, 0)])
def test_small_shapes(N, h_k, h_v, ntok, commit):
    x = gi.gdn_window_inputs(gi.rng(N * 100 + h_v * 10 + ntok), N, h_k, h_v, 128, ntok)
    d = _dev(x)
    S, ho, y = _gpu(d, h_k, commit)
    rS, rho, ry = _oracle(x, h_k, commit)
    assert max_rel_err(host(y), ry) <= TOL
    assert max_rel_err(host(S), rS) <= TOL
    assert np.array_equal(host(ho), rho)


def test_chained_windows_track_the_oracle():
    # four committed windows in a row, history ping-ponged as the page's host does
    N, h_k, h_v, ntok = 2, 2, 4, 4
    g = gi.rng(77)
    x = gi.gdn_window_inputs(g, N, h_k, h_v, 128, ntok)
    d = _dev(x)
    S = d["state"].clone()
    h_in, h_out = d["hist"].clone(), torch.empty_like(d["hist"])
    rS, rh = x["state"].astype(np.float64), x["hist"].astype(np.float64)
    for w in range(4):
        nx = gi.gdn_window_inputs(g, N, h_k, h_v, 128, ntok)
        for key in ("qkv", "alpha", "beta", "z"):
            d[key] = dev(nx[key], f32)
            x[key] = nx[key]
        d["hist"] = h_in
        _gpu(d, h_k, 1, hist_out=h_out, state=S)
        h_in, h_out = h_out, h_in
        rS, rh, ry = oracle.gdn_window(rS, rh, x["qkv"], x["alpha"], x["beta"], x["z"],
                                       x["conv_w"], x["dt"], x["ssm_a"], x["gamma"], h_k, 1)
    assert max_rel_err(host(S), rS) <= TOL
    assert np.array_equal(host(h_in), rh)


def test_rejections_write_nothing():
    x = gi.gdn_window_inputs(gi.rng(5), 1, 2, 2, 128, 2)
    d = _dev(x)
    y = torch.full((1, 2, 2, 128), 3.0, device="cuda")
    for kwargs, status in ((dict(h_k=2, commit=0x103), gdn.GDN_ERR_INVALID_ARG),
                           (dict(h_k=2, commit=2), gdn.GDN_ERR_INVALID_ARG)):
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_window_fused(d["state"], d["hist"], torch.empty_like(d["hist"]), d["qkv"],
                                 d["alpha"], d["beta"], d["z"], d["conv_w"], d["dt"], d["ssm_a"],
                                 d["gamma"], y=y, **kwargs)
        assert e.value.status == status
    with pytest.raises(gdn.GdnError) as e:   # hist_out aliasing hist
        gdn.gdn_window_fused(d["state"], d["hist"], d["hist"], d["qkv"], d["alpha"], d["beta"],
                             d["z"], d["conv_w"], d["dt"], d["ssm_a"], d["gamma"], 2, 1, y=y)
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    assert bool(torch.all(y == 3.0))
    assert np.array_equal(host(d["state"]), x["state"].astype(np.float64))


@pytest.mark.parametrize("commit", [1, 0x105])
def test_gate_extremes(commit):
    # gates that saturate: alpha = +60 drives the decay to exp(-60 * |ssm_a|) = 0 (the state wiped at
    # that token), alpha = -60 to exp(0) = 1 (no decay); beta_raw = -60 / +60 give beta = 0 / 1
    N, h_k, h_v, ntok = 2, 2, 4, 8
    x = gi.gdn_window_inputs(gi.rng(31), N, h_k, h_v, 128, ntok)
    x["alpha"][:, 2, 0] = 60.0
    x["alpha"][:, 5:7, 1] = 60.0
    x["alpha"][:, :, 2] = -60.0
    x["beta"][0, 3:6, :] = -60.0
    x["beta"][1, :, 3] = 60.0
    S, ho, y = _gpu(_dev(x), h_k, commit)
    rS, rho, ry = _oracle(x, h_k, commit)
    assert np.isfinite(ry).all() and np.isfinite(rS).all()
    assert max_rel_err(host(y), ry) <= TOL
    assert max_rel_err(host(S), rS) <= TOL
    assert np.array_equal(host(ho), rho)
