"""Pins of oracle.comba_forward, the Comba recurrence over T tokens (KBench comba_decode_step
spec, spec_md: the decode step is the comba-forward task's recurrence run for one token, and
running the step T times reproduces that task).

- one token equals one oracle.comba_decode step, on every head;
- T tokens equal T chained oracle.comba_decode steps, token by token, state and outputs bitwise
  (the [B, T, H] token layout and the carried state);
- with the read key equal to the write key, on the transposed state, it equals a chain of
  oracle.gdn_decode steps with the linear gate exp(g) (the GDN recurrence, pinned on its own);
- with beta = 0 the state only decays: S_T = exp(sum g) S_0 and o_t = scale q_t^T S_t (closed form);
- T = 0 returns the state unchanged.
"""
import numpy as np

import gdn_inputs as gi
import oracle


def _chain(x, scale):
    S = x["state"].astype(np.float64)
    outs = []
    for t in range(x["q"].shape[1]):
        S, o = oracle.comba_decode(S, x["q"][:, t], x["k"][:, t], x["v"][:, t], x["p"][:, t],
                                   x["beta"][:, t], x["g_log"][:, t], scale)
        outs.append(o)
    return S, np.stack(outs, axis=1)


def test_one_token_is_one_decode_step():
    x = gi.comba_forward_inputs(gi.rng(1), 2, 1, 3, 8, 4)
    S, o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["p"], x["beta"], x["g_log"], 0.3)
    S1, o1 = oracle.comba_decode(x["state"], x["q"][:, 0], x["k"][:, 0], x["v"][:, 0], x["p"][:, 0],
                                 x["beta"][:, 0], x["g_log"][:, 0], 0.3)
    assert np.array_equal(S, S1) and np.array_equal(o[:, 0], o1)


def test_tokens_equal_chained_decode_steps():
    x = gi.comba_forward_inputs(gi.rng(2), 3, 5, 2, 16, 8)
    S, o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["p"], x["beta"], x["g_log"], 0.25)
    Sc, oc = _chain(x, 0.25)
    assert np.array_equal(S, Sc) and np.array_equal(o, oc)


def test_read_key_equal_write_key_is_the_gdn_recurrence():
    B, T, H, K, V = 2, 4, 3, 8, 8
    x = gi.comba_forward_inputs(gi.rng(3), B, T, H, K, V)
    S, o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["k"], x["beta"], x["g_log"], 0.5)
    Sg = np.swapaxes(x["state"].astype(np.float64), -1, -2)   # GDN state is [V][K]
    for t in range(T):
        Sg, y = oracle.gdn_decode(Sg, x["q"][:, t], x["k"][:, t], x["v"][:, t],
                                  np.exp(x["g_log"][:, t].astype(np.float64)), x["beta"][:, t], 0.5)
        assert np.allclose(y, o[:, t], rtol=1e-12, atol=1e-12)
    assert np.allclose(np.swapaxes(Sg, -1, -2), S, rtol=1e-12, atol=1e-12)


def test_zero_beta_only_decays():
    B, T, H, K, V = 1, 3, 2, 4, 6
    x = gi.comba_forward_inputs(gi.rng(4), B, T, H, K, V)
    beta = np.zeros_like(x["beta"])
    S, o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["p"], beta, x["g_log"], 0.7)
    S0 = x["state"].astype(np.float64)
    G = np.cumsum(x["g_log"].astype(np.float64), axis=1)           # [B, T, H]
    assert np.allclose(S, np.exp(G[:, -1])[:, :, None, None] * S0, rtol=1e-13, atol=0)
    for t in range(T):
        St = np.exp(G[:, t])[:, :, None, None] * S0
        ref = np.einsum("bhk,bhkv->bhv", 0.7 * x["q"][:, t].astype(np.float64), St)
        assert np.allclose(o[:, t], ref, rtol=1e-12, atol=1e-14)


def test_no_tokens_keeps_the_state():
    x = gi.comba_forward_inputs(gi.rng(5), 2, 0, 2, 4, 4)
    S, o = oracle.comba_forward(x["state"], x["q"], x["k"], x["v"], x["p"], x["beta"], x["g_log"], 1.0)
    assert o.shape == (2, 0, 2, 4) and np.array_equal(S, x["state"].astype(np.float64))
