"""Pins of the oracle's decode steps (GDN and Comba) to facts fixed outside the oracle itself:
hand-worked examples, closed forms of special gates, the recall property of the delta rule, the
key-sharing map, the Comba/GDN reduction, and the error magnitudes of wrong variants that the Comba
spec prints.  CPU only."""
import os

import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from parity import rel_frobenius

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gdn_case(seed, B=2, Hk=2, Hv=4, Dk=8, Dv=6):
    g = gi.rng(seed)
    S = g.standard_normal((B, Hv, Dv, Dk))
    t = gi.gdn_decode_token(g, B, Hk, Hv, Dk, Dv)
    return S, t


# ---------------------------------------------------------------------------------------------
# Hand-worked examples (every number below is derived by hand in the comments)
# ---------------------------------------------------------------------------------------------
def test_gdn_hand_example_2x2():
    # metaltile-std gated_delta.rs, module doc "Recurrence per step", with Dk = Dv = 2:
    # S = [[1,2],[3,4]] (rows = Dv, cols = Dk), g = 0.8, beta = 0.25, k = [0.6, 0.8], q = [1, -2],
    # v = [1, -1], scale = 0.5.
    #   S' = g S = [[0.8, 1.6], [2.4, 3.2]]
    #   kv = S' k = [0.48 + 1.28, 1.44 + 2.56] = [1.76, 4.0]
    #   delta = (v - kv) beta = [-0.19, -1.25]
    #   S_new = S' + delta k^T = [[0.686, 1.448], [1.65, 2.2]]
    #   y = scale S_new q = 0.5 [0.686 - 2.896, 1.65 - 4.4] = [-1.105, -1.375]
    S = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    q = np.array([[[1.0, -2.0]]])
    k = np.array([[[0.6, 0.8]]])
    v = np.array([[[1.0, -1.0]]])
    Sn, y = oracle.gdn_decode(S, q, k, v, np.array([[0.8]]), np.array([[0.25]]), 0.5)
    np.testing.assert_allclose(Sn[0, 0], [[0.686, 1.448], [1.65, 2.2]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(y[0, 0], [-1.105, -1.375], rtol=0, atol=1e-14)


def test_comba_hand_example_2x2():
    # KBench comba_decode_step spec_md, elementwise form, K = V = 2 (rows i = K, cols j = V):
    # state = [[1,2],[3,4]], g = ln 0.5, p = [1,0], k = [0,1], v = [1,1], beta = 0.5, q = [1,1],
    # scale = 1.
    #   S = 0.5 state = [[0.5, 1], [1.5, 2]]
    #   u_j = beta (v_j - sum_i p_i S_ij) = 0.5 [1 - 0.5, 1 - 1] = [0.25, 0]
    #   S_new = S + k u^T = [[0.5, 1], [1.75, 2]]
    #   o_j = sum_i q_i S_new_ij = [2.25, 3]
    S = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    Sn, o = oracle.comba_decode(S, [[[1.0, 1.0]]], [[[0.0, 1.0]]], [[[1.0, 1.0]]],
                                [[[1.0, 0.0]]], [[0.5]], [[np.log(0.5)]], 1.0)
    np.testing.assert_allclose(Sn[0, 0], [[0.5, 1.0], [1.75, 2.0]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[0, 0], [2.25, 3.0], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Closed forms and invariants
# ---------------------------------------------------------------------------------------------
def test_gate_one_beta_zero_leaves_state_unchanged():
    S, t = _gdn_case(1)
    B, Hv = S.shape[:2]
    Sn, y = oracle.gdn_decode(S, t["q"], t["k"], t["v"], np.ones((B, Hv)), np.zeros((B, Hv)), 0.3)
    assert np.array_equal(Sn, S)  # bitwise
    qe = np.repeat(t["q"].astype(np.float64), Hv // t["q"].shape[1], axis=1)
    np.testing.assert_allclose(y, 0.3 * np.einsum("bhrc,bhc->bhr", S, qe), rtol=1e-13, atol=1e-13)


def test_gate_zero_forgets_prior_state():
    S, t = _gdn_case(2)
    B, Hv = S.shape[:2]
    Hk = t["k"].shape[1]
    beta = t["beta"].astype(np.float64)
    Sn, y = oracle.gdn_decode(S, t["q"], t["k"], t["v"], np.zeros((B, Hv)), beta, 0.7)
    ke = np.repeat(t["k"].astype(np.float64), Hv // Hk, axis=1)
    qe = np.repeat(t["q"].astype(np.float64), Hv // Hk, axis=1)
    v = t["v"].astype(np.float64)
    want = beta[..., None, None] * v[..., :, None] * ke[..., None, :]
    np.testing.assert_allclose(Sn, want, rtol=1e-15, atol=1e-15)
    want_y = 0.7 * beta[..., None] * np.sum(ke * qe, -1)[..., None] * v
    np.testing.assert_allclose(y, want_y, rtol=1e-13, atol=1e-13)


def test_unit_key_full_step_recalls_value():
    # beta = 1 and |k| = 1: S_new k = g S k + (v - g S k) (k.k) = v.
    S, t = _gdn_case(3, Dk=16, Dv=16)
    B, Hv = S.shape[:2]
    Hk = t["k"].shape[1]
    k = np.random.default_rng(5).standard_normal(t["k"].shape)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    Sn, _ = oracle.gdn_decode(S, t["q"], k, t["v"], t["g"], np.ones((B, Hv)), 1.0)
    ke = np.repeat(k, Hv // Hk, axis=1)
    np.testing.assert_allclose(np.einsum("bhrc,bhc->bhr", Sn, ke), t["v"], rtol=0, atol=1e-12)


def test_key_sharing_map_is_division():
    # Hv = 6 value heads over Hk = 2 key heads: value head hv reads key head hv // 3.
    S, t = _gdn_case(4, B=1, Hk=2, Hv=6, Dk=8, Dv=8)
    Sn, y = oracle.gdn_decode(S, t["q"], t["k"], t["v"], t["g"], t["beta"], 0.5)
    for hv in range(6):
        hk = hv // 3
        s1, y1 = oracle.gdn_decode(S[:, hv:hv + 1], t["q"][:, hk:hk + 1], t["k"][:, hk:hk + 1],
                                   t["v"][:, hv:hv + 1], t["g"][:, hv:hv + 1],
                                   t["beta"][:, hv:hv + 1], 0.5)
        assert np.array_equal(s1[:, 0], Sn[:, hv])
        assert np.array_equal(y1[:, 0], y[:, hv])
        if hv % 2 != hk:  # the modulo map would read another, distinct key head
            s2, _ = oracle.gdn_decode(S[:, hv:hv + 1], t["q"][:, hv % 2:hv % 2 + 1],
                                      t["k"][:, hv % 2:hv % 2 + 1], t["v"][:, hv:hv + 1],
                                      t["g"][:, hv:hv + 1], t["beta"][:, hv:hv + 1], 0.5)
            assert not np.allclose(s2[:, 0], Sn[:, hv])


def test_key_sharing_rejects_indivisible_heads():
    S, t = _gdn_case(5, Hk=2, Hv=4)
    with pytest.raises(ValueError):
        oracle.gdn_decode(S[:, :3], t["q"], t["k"], t["v"][:, :3], t["g"][:, :3],
                          t["beta"][:, :3], 1.0)


def test_comba_with_read_key_equal_write_key_is_gdn():
    # The Comba spec: in DeltaNet the read and write keys are the same vector.  Comba's state is
    # (K, V); GDN's is (Dv, Dk), so the two agree on the transposed state, with g_log = log g.
    S, t = _gdn_case(6, B=2, Hk=3, Hv=3, Dk=8, Dv=5)
    Sg, yg = oracle.gdn_decode(S, t["q"], t["k"], t["v"], t["g"], t["beta"], 0.25)
    Sc, oc = oracle.comba_decode(np.swapaxes(S, -1, -2), t["q"], t["k"], t["v"], t["k"],
                                 t["beta"], np.log(t["g"].astype(np.float64)), 0.25)
    np.testing.assert_allclose(np.swapaxes(Sc, -1, -2), Sg, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oc, yg, rtol=1e-12, atol=1e-12)


def test_decode_steps_chain_equals_prefill_recurrence():
    # The Comba spec (spec_md): running the step T times reproduces the multi-token forward.  Here
    # the GDN decode step, fed the prefill's derived gates and normalised keys, must reproduce the
    # oracle's sequential prefill of the same tokens.
    g = gi.rng(7)
    T, Hk, Hv, K, V = 9, 1, 2, 8, 8
    x = gi.gdn_prefill_inputs(g, [T], Hk, Hv, K, V, pool=1, mild_gates=True)
    scale = K ** -0.5
    pool, out, st = oracle.gdn_prefill(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                                       x["dt_bias"], x["state_pool"], [0], [0, T], scale)
    assert st == 0
    S = x["state_pool"][0].astype(np.float64)[None]  # [1, Hv, V, K]
    for t in range(T):
        a = x["a"][t].astype(np.float64) + x["dt_bias"]
        sp = np.where(a > 20, a, np.log1p(np.exp(a)))
        gate = np.exp(-np.exp(x["A_log"].astype(np.float64)) * sp)[None]
        beta = (1 / (1 + np.exp(-x["b"][t].astype(np.float64))))[None]
        k = x["k"][t].astype(np.float64)
        q = x["q"][t].astype(np.float64)
        kn = k / np.sqrt(np.sum(k * k, -1, keepdims=True) + 1e-6)
        qn = q / np.sqrt(np.sum(q * q, -1, keepdims=True) + 1e-6)
        S, y = oracle.gdn_decode(S, qn[None], kn[None], x["v"][t][None], gate, beta, scale)
        np.testing.assert_allclose(y[0], out[t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0], pool[0], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# Error calibration of wrong variants, printed by the Comba spec (precision_md)
# ---------------------------------------------------------------------------------------------
def _golden_mutants():
    vals = {}
    with open(os.path.join(GOLDEN, "comba_mutant_errors.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, val = line.split()
                vals[name] = float(val)
    return vals


def test_wrong_variants_land_where_the_spec_says():
    want = _golden_mutants()
    B, H, K, V = 16, 8, 128, 128
    scale = K ** -0.5
    g = gi.rng(0)
    S = np.zeros((B, H, K, V))
    for _ in range(16):  # make_inputs_src: 16 warm-up steps from a zero state
        t = gi.comba_decode_token(g, B, H, K, V)
        S, _ = oracle.comba_decode(S, t["q"], t["k"], t["v"], t["p"], t["beta"], t["g_log"], scale)
        S = S.astype(np.float32).astype(np.float64)  # the state is stored in fp32 between steps
    t = gi.comba_decode_token(g, B, H, K, V)
    ref_S, ref_o = oracle.comba_decode(S, t["q"], t["k"], t["v"], t["p"], t["beta"], t["g_log"],
                                       scale)

    def worst(Sn, o):
        return max(rel_frobenius(Sn, ref_S), rel_frobenius(o, ref_o))

    got = {}
    # the new state stored in bf16 (o read out of that state)
    Sb = gi.bf16_round(ref_S.astype(np.float32)).astype(np.float64)
    got["bf16_state"] = worst(Sb, np.einsum("bhij,bhi->bhj", Sb, t["q"] * scale))
    # forget gate dropped: exp(g) replaced by 1
    got["dropped_gate"] = worst(*oracle.comba_decode(S, t["q"], t["k"], t["v"], t["p"], t["beta"],
                                                     np.zeros_like(t["g_log"]), scale))
    # correction read with the write key
    got["k_instead_of_p"] = worst(*oracle.comba_decode(S, t["q"], t["k"], t["v"], t["k"],
                                                       t["beta"], t["g_log"], scale))
    # correction "- S^T p" dropped: a zero read key removes exactly that term
    got["dropped_correction"] = worst(*oracle.comba_decode(S, t["q"], t["k"], t["v"],
                                                           np.zeros_like(t["p"]), t["beta"],
                                                           t["g_log"], scale))
    for name, ref in want.items():
        ratio = got[name] / ref
        assert 0.75 <= ratio <= 1.35, (name, got[name], ref)
