"""Pins of the oracle's varlen prefill: brute-force agreement with the chunkwise WY algebra of the
pymllm gdn_chunkwise page on small shapes, closed forms of the derived gates, sequence splitting,
segmentation and the pool's slot handling.  CPU only."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from wy_reference import wy_sequence


def _inputs(seed, seqlens, Hk=1, Hv=2, K=8, V=8, pool=4, mild=True):
    return gi.gdn_prefill_inputs(gi.rng(seed), seqlens, Hk, Hv, K, V, pool, mild_gates=mild)


def _run(x, scale, **kw):
    return oracle.gdn_prefill(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                              x["state_pool"], x["cache_indices"], x["cu_seqlens"], scale, **kw)


@pytest.mark.parametrize("KV", [4, 8])
@pytest.mark.parametrize("C", [2, 4, 8, 64])
@pytest.mark.parametrize("mild", [True, False])
def test_wy_chunkwise_equals_sequential(KV, C, mild):
    T = 3 * C + 1
    x = _inputs(10 + KV + C, [T], Hk=1, Hv=2, K=KV, V=KV, pool=2, mild=mild)
    scale = KV ** -0.5
    pool, out, st = _run(x, scale)
    assert st == 0
    slot = int(x["cache_indices"][0])
    for h in range(2):
        o_wy, S_wy = wy_sequence(x["state_pool"][slot, h], x["q"][:, 0], x["k"][:, 0],
                                 x["v"][:, h], x["a"][:, h], x["b"][:, h], float(x["A_log"][h]),
                                 float(x["dt_bias"][h]), C, scale)
        ref = max(1.0, np.max(np.abs(out[:, h])))
        assert np.max(np.abs(o_wy - out[:, h])) <= 1e-10 * ref
        assert np.max(np.abs(S_wy - pool[slot, h])) <= 1e-10 * max(1.0, np.max(np.abs(S_wy)))


def test_page_form_agrees_when_w_is_read_untransposed():
    # Mild gates keep 1/gamma finite, so the page's own form can be evaluated.  With the w
    # recursion read as W_{<i}(K_{<i}^T .) it matches the sequential oracle; as printed
    # (K_{<i}(W_{<i}^T .)) it does not, once a chunk has three or more tokens.
    C, T, KV = 8, 17, 6
    x = _inputs(3, [T], K=KV, V=KV, pool=1, mild=True)
    scale = KV ** -0.5
    pool, out, _ = _run(x, scale)
    args = (x["state_pool"][0, 0], x["q"][:, 0], x["k"][:, 0], x["v"][:, 0], x["a"][:, 0],
            x["b"][:, 0], float(x["A_log"][0]), float(x["dt_bias"][0]), C, scale)
    o_read, S_read = wy_sequence(*args, form="page")
    o_printed, _ = wy_sequence(*args, form="printed")
    np.testing.assert_allclose(o_read, out[:, 0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(S_read, pool[0, 0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(o_printed[:2], out[:2, 0], rtol=0, atol=1e-10)
    assert np.max(np.abs(o_printed - out[:, 0])) > 1e-3


def test_gate_closed_forms():
    # With beta -> 0 (b = -1e4 gives sigmoid exactly 0 in double) the step is S <- g S, so the gate
    # can be read off the state.  a + dt_bias = 0 gives softplus = ln 2, so g = 2^(-exp(A_log));
    # a + dt_bias = 30 (> 20, the softplus threshold) gives g = exp(-exp(A_log) * 30).
    K = V = 4
    S0 = np.arange(1, 1 + V * K, dtype=np.float64).reshape(1, 1, V, K)
    q = np.ones((1, 1, K))
    k = np.ones((1, 1, K))
    v = np.ones((1, 1, V))
    for a_val, A_log, want in [(0.0, 0.0, 0.5), (0.0, np.log(3.0), 0.125),
                               (30.0, 0.0, np.exp(-30.0)), (-1e4, 2.0, 1.0)]:
        pool, _, _ = oracle.gdn_prefill(q, k, v, [[a_val]], [[-1e4]], [A_log], [0.0], S0, [0],
                                        [0, 1], 1.0)
        np.testing.assert_allclose(pool[0, 0], want * S0[0, 0], rtol=1e-14, atol=0)
    # b = 0 gives beta = 1/2; with g -> 0 (a = 1e4) the prior state is forgotten:
    # S_new = beta v k^^T with k^^ = k / sqrt(|k|^2 + eps).
    pool, _, _ = oracle.gdn_prefill(q, k, v, [[1e4]], [[0.0]], [0.0], [0.0], S0, [0], [0, 1], 1.0)
    np.testing.assert_allclose(pool[0, 0], 0.5 / np.sqrt(4.0 + 1e-6) * np.ones((V, K)), rtol=1e-14)


def test_no_decay_no_update_reads_initial_state():
    # a -> -inf (g = 1) and b -> -inf (beta = 0): the state is unchanged and out_t = S0 q^_t.
    x = _inputs(4, [5], K=8, V=8, pool=2)
    x["a"][:] = -1e4
    x["b"][:] = -1e4
    scale = 0.125
    pool, out, _ = _run(x, scale)
    slot = int(x["cache_indices"][0])
    assert np.array_equal(pool, x["state_pool"].astype(np.float64))
    q = x["q"][:, 0].astype(np.float64)
    qn = scale * q / np.sqrt(np.sum(q * q, -1, keepdims=True) + 1e-6)
    for h in range(2):
        np.testing.assert_allclose(out[:, h], qn @ x["state_pool"][slot, h].T.astype(np.float64),
                                   rtol=1e-13, atol=1e-13)


def test_split_sequence_carries_state_through_pool():
    x = _inputs(5, [13], K=8, V=8, pool=3)
    scale = 8 ** -0.5
    pool_full, out_full, _ = _run(x, scale)
    ci = x["cache_indices"]
    y1 = dict(x, cu_seqlens=np.array([0, 6]))
    pool_1, out_1, _ = _run(y1, scale)
    pool_2, out_2, _ = oracle.gdn_prefill(x["q"][6:], x["k"][6:], x["v"][6:], x["a"][6:],
                                          x["b"][6:], x["A_log"], x["dt_bias"], pool_1, ci,
                                          [0, 7], scale)
    np.testing.assert_allclose(pool_2, pool_full, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out_1[:6], out_full[:6], rtol=0, atol=1e-13)
    np.testing.assert_allclose(out_2, out_full[6:], rtol=0, atol=1e-13)


def test_segmentation_slots_and_key_sharing():
    # Three sequences (one empty), Hv = 4 over Hk = 2.  Outputs of a sequence depend only on its own
    # tokens and its own slot; slots not referenced stay bitwise unchanged; an empty sequence leaves
    # its slot unchanged.
    seqlens = [7, 0, 5]
    x = _inputs(6, seqlens, Hk=2, Hv=4, K=8, V=8, pool=6)
    scale = 8 ** -0.5
    pool, out, st = _run(x, scale)
    assert st == 0
    ci = [int(c) for c in x["cache_indices"]]
    for s in range(6):
        if s not in ci or s == ci[1]:
            assert np.array_equal(pool[s], x["state_pool"][s].astype(np.float64))
    # perturb sequence 2's tokens: sequence 0's outputs and slot are bitwise unchanged
    x2 = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in x.items()}
    x2["v"][7:] += 1.0
    pool2, out2, _ = _run(x2, scale)
    assert np.array_equal(out2[:7], out[:7]) and np.array_equal(pool2[ci[0]], pool[ci[0]])
    assert not np.allclose(out2[7:], out[7:])
    # each value head uses key head h // 2: compare with single-head units
    for h in range(4):
        S, o = oracle.gdn_prefill_unit(x["q"][:7], x["k"][:7], x["v"][:7], x["a"][:7],
                                       x["b"][:7], x["A_log"][h], x["dt_bias"][h],
                                       x["state_pool"][ci[0], h], h, scale)
        assert np.array_equal(o, out[:7, h]) and np.array_equal(S, pool[ci[0], h])


def test_bad_slots_and_bounds_are_flagged_and_skipped():
    x = _inputs(7, [4, 4], K=4, V=4, pool=3)
    scale = 0.5
    x["cache_indices"] = np.array([3, 0])   # 3 is outside the pool of 3
    pool, out, st = _run(x, scale)
    assert st & oracle.STATUS_BAD_CACHE_INDEX
    assert np.array_equal(out[:4], np.zeros_like(out[:4]))
    assert np.array_equal(pool[1:], x["state_pool"][1:].astype(np.float64))
    assert not np.array_equal(pool[0], x["state_pool"][0].astype(np.float64))
    x["cache_indices"] = np.array([1, 0])
    x["cu_seqlens"] = np.array([0, 5, 4])   # decreasing bound
    pool, out, st = _run(x, scale)
    assert st & oracle.STATUS_BAD_SEQLENS
