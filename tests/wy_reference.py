"""Chunkwise WY form of the gated delta rule in float64 numpy (test-only).

This restates the algorithm of the pymllm gdn_chunkwise page (module doc, steps 1-3) as matrix
algebra so that tests can check, by brute force on small shapes, that it reproduces the sequential
recurrence of the oracle.  It is the algebra the CUDA prefill kernel follows, written in the plainest
way; it shares nothing with that kernel.

Readings of the page used here:
  - step 1's w recursion is read as w_i = beta_i k_i - W_{<i} (K_{<i}^T (beta_i k_i)) (the printed
    form has W and K swapped, which agrees only for the first two rows);
  - the state update's "U~^T K" is read as U~ K^T = sum_i u~_i k_i^T, in the [V, K] state layout;
  - "triu" is the causal mask including the diagonal, and "gamma ." scales output column t by the
    inclusive cumulative gate gamma_t; gamma_C is the product over the whole (possibly short) chunk;
  - every exponential is taken as exp(G_t - G_s) with s <= t (the ratio form), which equals the
    page's beta_i / gamma_i form in exact arithmetic but cannot overflow.
"""
import numpy as np


def derive_gates(a, b, A_log_h, dt_bias_h):
    """log g = -exp(A_log) softplus(a + dt_bias) (threshold 20), beta = sigmoid(b)."""
    x = np.asarray(a, np.float64) + dt_bias_h
    sp = np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))
    log_g = -np.exp(A_log_h) * sp
    beta = 1.0 / (1.0 + np.exp(-np.asarray(b, np.float64)))
    return log_g, beta


def l2n(x, eps=1e-6):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def wy_chunk(S0, Kh, Qh, V, log_g, beta):
    """One chunk.  S0 [Vd, Kd]; Kh, Qh [L, Kd] (normalised keys, scaled normalised queries);
    V [L, Vd]; log_g, beta [L].  Returns (O [L, Vd], S_new [Vd, Kd])."""
    L = len(log_g)
    G = np.cumsum(log_g)
    gam = np.exp(G)
    D = np.tril(np.exp(np.minimum(G[:, None] - G[None, :], 0.0)))   # D_ts, s <= t
    A = Kh @ Kh.T
    Tinv = np.linalg.inv(np.eye(L) + np.tril(beta[:, None] * A * D, -1))
    Wbar = Tinv @ ((beta * gam)[:, None] * Kh)
    U = Tinv @ (beta[:, None] * V)
    Delta = U - Wbar @ S0.T
    O = gam[:, None] * (Qh @ S0.T) + np.tril((Qh @ Kh.T) * D) @ Delta
    S_new = gam[-1] * S0 + (Delta * D[-1][:, None]).T @ Kh
    return O, S_new


def wy_chunk_page_form(S0, Kh, Qh, V, log_g, beta, printed_w=False):
    """The page's own form (steps 1-3 with 1/gamma_i inside u~), with the w recursion either as
    read (printed_w=False) or as printed (printed_w=True).  Overflows for strong decay."""
    L, Kd = Kh.shape
    G = np.cumsum(log_g)
    gam = np.exp(G)
    W = np.zeros((Kd, L))      # columns w_i
    Ut = np.zeros((V.shape[1], L))  # columns u~_i
    Kc = Kh.T                  # columns k_i
    for i in range(L):
        bk = beta[i] * Kc[:, i]
        if printed_w:
            W[:, i] = bk - Kc[:, :i] @ (W[:, :i].T @ bk)
        else:
            W[:, i] = bk - W[:, :i] @ (Kc[:, :i].T @ bk)
        Ut[:, i] = (beta[i] / gam[i]) * V[i] - Ut[:, :i] @ (Kc[:, :i].T @ bk)
    KQ = np.triu(Kc.T @ Qh.T)  # [s, t], s <= t
    S0W = S0 @ W
    O = gam[None, :] * (S0 @ Qh.T - S0W @ KQ + Ut @ KQ)   # [Vd, L]
    S_new = gam[-1] * (S0 - S0W @ Kc.T + Ut @ Kc.T)
    return O.T, S_new


def wy_sequence(S0, q, k, v, a, b, A_log_h, dt_bias_h, chunk, scale, eps=1e-6, form="ratio"):
    """One (sequence, value head): q, k [T, Kd]; v [T, Vd]; a, b [T].  Returns (out, S)."""
    log_g, beta = derive_gates(a, b, A_log_h, dt_bias_h)
    Kh = l2n(k, eps)
    Qh = scale * l2n(q, eps)
    T = len(a)
    out = np.zeros((T, v.shape[1]))
    S = np.array(S0, np.float64)
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        sl = slice(c0, c1)
        if form == "ratio":
            O, S = wy_chunk(S, Kh[sl], Qh[sl], np.asarray(v[sl], np.float64), log_g[sl], beta[sl])
        else:
            O, S = wy_chunk_page_form(S, Kh[sl], Qh[sl], np.asarray(v[sl], np.float64),
                                      log_g[sl], beta[sl], printed_w=(form == "printed"))
        out[sl] = O
    return out, S
