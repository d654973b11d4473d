"""Pins of the oracle's fused decode window (regolith gdn.metal): conv tap order, the gate's closed
forms, the key-head map h % h_k, reduction of one token to the Comba step, the output norm's RMS,
and the commit / verify / partial-commit semantics of GdnArgs.  CPU only."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle


def _inputs(seed, N=1, h_k=1, h_v=1, D=8, ntok=1):
    return gi.gdn_window_inputs(gi.rng(seed), N, h_k, h_v, D, ntok)


def _run(x, h_k, commit, hist_out=None, **over):
    y = dict(x, **over)
    return oracle.gdn_window(y["state"], y["hist"], y["qkv"], y["alpha"], y["beta"], y["z"],
                             y["conv_w"], y["dt"], y["ssm_a"], y["gamma"], h_k, commit,
                             hist_out=hist_out)


def _silu(s):
    return s / (1.0 + np.exp(-s))


def _sig(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, np.float64)))


def test_conv_taps_read_history_oldest_first():
    # With a zero state the output is y_j = c v_j / rms(v) * gamma_j sigmoid(z_j) (c = +-1 up to
    # eps), so y reveals the v channels' conv output.  A one-hot tap m must select vals[m] of
    # (h0, h1, h2, x_t), oldest first.
    D = 8
    x = _inputs(1, D=D)
    x["state"][:] = 0.0
    C = 3 * D
    hist = x["hist"][0].astype(np.float64)
    xt = x["qkv"][0, 0].astype(np.float64)
    vals = [hist[:, 0], hist[:, 1], hist[:, 2], xt]
    for m in range(4):
        w = np.zeros((C, 4), np.float32)
        w[:, m] = 1.0
        _, _, y = _run(x, 1, 0, conv_w=w)
        r = y[0, 0, 0] / (x["gamma"] * _sig(x["z"][0, 0, 0]))
        want = _silu(vals[m][2 * D:3 * D])
        cos = np.dot(r, want) / (np.linalg.norm(r) * np.linalg.norm(want))
        assert abs(abs(cos) - 1.0) < 1e-12, (m, cos)
        for other in range(4):
            if other != m:
                alt = _silu(vals[other][2 * D:3 * D])
                c2 = np.dot(r, alt) / (np.linalg.norm(r) * np.linalg.norm(alt))
                assert abs(abs(c2) - 1.0) > 1e-3


def test_gate_closed_forms():
    # beta_raw -> -inf makes beta = 0, so a committed token leaves S <- gate S.
    # alpha + dt = 0: softplus = ln 2, gate = 2^ssm_a;  alpha + dt = 30 (> 20): gate = e^(30 ssm_a).
    x = _inputs(2, D=4)
    x["beta"][:] = -1e4
    for a_val, ssm, want in [(0.0, -1.0, 0.5), (0.0, -3.0, 0.125), (30.0, -0.5, np.exp(-15.0))]:
        x["alpha"][:] = a_val - x["dt"][0]
        S, _, _ = _run(x, 1, 1, ssm_a=np.array([ssm], np.float32))
        np.testing.assert_allclose(S, want * x["state"].astype(np.float64), rtol=1e-6, atol=0)


def test_one_token_is_conv_then_comba_step_then_gated_rmsnorm():
    # With identity taps (0,0,0,1) the conv output is SiLU(x_t).  One token of the window is then
    # the Comba step with p = k = k^, q = q^, log-decay log(gate) and scale 1/sqrt(D), followed by
    # the gated RMSNorm.  Value head h reads key head h % h_k.
    D, h_k, h_v = 8, 2, 6
    x = _inputs(3, N=2, h_k=h_k, h_v=h_v, D=D)
    C = (2 * h_k + h_v) * D
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0
    S_after, hist_out, y = _run(x, h_k, 1, conv_w=w)
    eps = 1e-6
    for n in range(2):
        act = _silu(x["qkv"][n, 0].astype(np.float64))
        for h in range(h_v):
            hk = h % h_k
            q = act[hk * D:(hk + 1) * D]
            k = act[(h_k + hk) * D:(h_k + hk + 1) * D]
            v = act[(2 * h_k + h) * D:(2 * h_k + h + 1) * D]
            qn = q / np.sqrt(q @ q + eps)
            kn = k / np.sqrt(k @ k + eps)
            a = x["alpha"][n, 0, h] + np.float64(x["dt"][h])
            gate = np.exp(np.log1p(np.exp(a)) * np.float64(x["ssm_a"][h]))
            beta = _sig(x["beta"][n, 0, h])
            S0 = x["state"][n, :, h, :].astype(np.float64)[None, None]   # [1,1,K=i,V=j]
            Sn, o = oracle.comba_decode(S0, qn[None, None], kn[None, None], v[None, None],
                                        kn[None, None], [[beta]], [[np.log(gate)]], D ** -0.5)
            np.testing.assert_allclose(S_after[n, :, h, :], Sn[0, 0], rtol=0, atol=1e-12)
            o = o[0, 0]
            want = o / np.sqrt(np.mean(o * o) + eps) * x["gamma"] * _sig(x["z"][n, 0, h])
            np.testing.assert_allclose(y[n, 0, h], want, rtol=0, atol=1e-11)


def test_value_head_reads_key_head_modulo():
    D, h_k, h_v = 4, 2, 6
    x = _inputs(4, h_k=h_k, h_v=h_v, D=D, ntok=3)
    S_all, _, y_all = _run(x, h_k, 1)
    for h in range(h_v):
        for hk, expect_equal in [(h % h_k, True), (h // 3, h // 3 == h % h_k)]:
            ch = np.r_[hk * D:(hk + 1) * D, (h_k + hk) * D:(h_k + hk + 1) * D,
                       (2 * h_k + h) * D:(2 * h_k + h + 1) * D]
            one = dict(state=x["state"][:, :, h:h + 1, :], hist=x["hist"][:, ch],
                       qkv=x["qkv"][:, :, ch], alpha=x["alpha"][:, :, h:h + 1],
                       beta=x["beta"][:, :, h:h + 1], z=x["z"][:, :, h:h + 1],
                       conv_w=x["conv_w"][ch], dt=x["dt"][h:h + 1], ssm_a=x["ssm_a"][h:h + 1],
                       gamma=x["gamma"])
            S1, _, y1 = _run(one, 1, 1)
            same = np.array_equal(y1[:, :, 0], y_all[:, :, h]) and \
                np.array_equal(S1[:, :, 0], S_all[:, :, h])
            assert same == expect_equal, (h, hk)


def test_output_norm_has_unit_rms():
    # y / (gamma sigmoid(z)) = o / sqrt(mean(o^2) + eps): its RMS is sqrt(ms / (ms + eps)), which is
    # 1 when eps vanishes and below 1 otherwise.
    x = _inputs(5, N=2, h_k=2, h_v=4, D=16, ntok=4)
    for eps, lo, hi in [(1e-30, 1 - 1e-12, 1 + 1e-12), (1e-6, 0.0, 1.0)]:
        y = oracle.gdn_window(x["state"], x["hist"], x["qkv"], x["alpha"], x["beta"], x["z"],
                              x["conv_w"], x["dt"], x["ssm_a"], x["gamma"], 2, 0, eps=eps)[2]
        r = y / (x["gamma"][None, None, None] * _sig(x["z"]))
        rms = np.sqrt(np.mean(r * r, axis=-1))
        assert np.all(rms >= lo) and np.all(rms <= hi), (eps, rms.min(), rms.max())


def test_verify_writes_nothing():
    x = _inputs(6, N=2, h_k=2, h_v=4, D=8, ntok=5)
    sentinel = np.full_like(x["hist"], 7.25, dtype=np.float64)
    S, ho, _ = _run(x, 2, 0, hist_out=sentinel)
    assert np.array_equal(S, x["state"].astype(np.float64))
    assert np.array_equal(ho, sentinel)


def test_committed_history_is_the_last_three_inputs():
    x = _inputs(7, N=2, h_k=1, h_v=2, D=4, ntok=5)
    full = np.concatenate([x["hist"], np.swapaxes(x["qkv"], 1, 2)], axis=2)   # [N, C, 3+ntok]
    for commit, k in [(1, 5), (0x101, 1), (0x102, 2), (0x105, 5)]:
        _, ho, _ = _run(x, 1, commit)
        assert np.array_equal(ho, full[:, :, k:k + 3].astype(np.float64)), commit


@pytest.mark.parametrize("k", [1, 3, 7])
def test_partial_commit_is_bitwise_a_k_token_commit(k):
    # GdnArgs: commit 0x100|k writes state and history after token k, in place, while every token's
    # y is still computed - bitwise the commit of a k-token step.
    x = _inputs(8, N=2, h_k=2, h_v=4, D=8, ntok=8)
    S_p, ho_p, y_p = _run(x, 2, 0x100 | k)
    xk = dict(x, qkv=x["qkv"][:, :k], alpha=x["alpha"][:, :k], beta=x["beta"][:, :k],
              z=x["z"][:, :k])
    S_k, ho_k, y_k = _run(xk, 2, 1)
    assert np.array_equal(S_p, S_k) and np.array_equal(ho_p, ho_k)
    assert np.array_equal(y_p[:, :k], y_k)
    _, _, y_v = _run(x, 2, 0)
    assert np.array_equal(y_p, y_v)   # y does not depend on the commit point


def test_window_equals_chain_of_single_token_commits():
    x = _inputs(9, N=1, h_k=2, h_v=2, D=8, ntok=4)
    S_w, ho_w, y_w = _run(x, 2, 1)
    S, hist = x["state"], x["hist"]
    for t in range(4):
        xt = dict(x, state=S, hist=hist, qkv=x["qkv"][:, t:t + 1], alpha=x["alpha"][:, t:t + 1],
                  beta=x["beta"][:, t:t + 1], z=x["z"][:, t:t + 1])
        S, hist, y = _run(xt, 2, 1)
        assert np.array_equal(y[:, 0], y_w[:, t])
    assert np.array_equal(S, S_w) and np.array_equal(hist, ho_w)


def test_bad_commit_codes_are_rejected():
    x = _inputs(10, ntok=3)
    for bad in (2, 0x100, 0x104, 0x200 | 1):
        with pytest.raises(ValueError):
            _run(x, 1, bad)


def test_silu_and_the_l2_norm_eps_against_hand_values():
    # Two channels per head (D = 2), identity taps, a zero state and beta_raw = 0 (beta = 1/2): one
    # committed token leaves S[i][j] = k^_i * beta * v_j with v = SiLU(x_v) and k^ = k / sqrt(|k|^2
    # + eps), k = SiLU(x_k).  The values are worked out by hand, not by the oracle's formulas:
    #   SiLU(1) = sigma(1) = 0.7310585786300049,  SiLU(-2) = -2 sigma(-2) = -0.2384058440442351,
    #   SiLU(-30) = -30 / (1 + e^30) = -30 * 9.357622968840175e-14.
    # x_k = -30 makes |k|^2 ~ 1.6e-23, far below eps = 1e-6, so k^ = k / sqrt(eps) = 1000 k: a norm
    # without eps (unit k^) or with eps / 128 (k^ larger by sqrt(128)) misses by orders of magnitude.
    D = 2
    x = _inputs(6, D=D)
    x["state"][:] = 0.0
    x["beta"][:] = 0.0
    w = np.zeros((3 * D, 4), np.float32)
    w[:, 3] = 1.0
    x["qkv"][0, 0] = np.array([0.5, 0.25, -30.0, -30.0, 1.0, -2.0], np.float32)
    S, _, _ = _run(x, 1, 1, conv_w=w)
    v = np.array([0.7310585786300049, -0.2384058440442351])
    k = -30.0 * 9.357622968840175e-14
    k_hat = k / np.sqrt(2 * k * k + 1e-6)
    assert abs(k_hat / (1000.0 * k) - 1.0) < 1e-15
    want = np.array([[k_hat * 0.5 * v[0], k_hat * 0.5 * v[1]]] * 2)  # rows i (key), columns j
    np.testing.assert_allclose(S[0, :, 0, :], want, rtol=1e-12, atol=0)
