"""GPU parity of gdn_prefill_chunked (through the C ABI) against the sequential CPU oracle.

Tolerances (max |gpu - oracle| / max |oracle| per tensor): outputs (bf16) <= 5e-3, final state
<= 2e-3.  Integer behaviour is bit-exact: cache_indices gather and scatter, cu_seqlens segmentation,
and pool slots that no sequence references stay bitwise untouched.
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
OUT_TOL, STATE_TOL = 5e-3, 2e-3
SENTINEL = -1000.0  # exactly representable in bf16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    library()


def _to_dev(x, tok=torch.bfloat16):
    f32, i64 = torch.float32, torch.int64
    return {n: dev(x[n], dt) for n, dt in (("q", tok), ("k", tok), ("v", tok), ("a", tok),
                                           ("b", tok), ("A_log", f32), ("dt_bias", f32),
                                           ("state_pool", f32), ("cache_indices", i64),
                                           ("cu_seqlens", i64))}


def _gpu(d, scale, out_fill=SENTINEL, chunk_size=64):
    T, Hv = d["v"].shape[0], d["v"].shape[1]
    out = torch.full((T, Hv, 128), out_fill, dtype=d["v"].dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                            d["state_pool"], d["cache_indices"], d["cu_seqlens"], chunk_size,
                            scale=scale, out=out, dev_status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


def _check_all(x, d, out, scale):
    pool_ref, out_ref, st = oracle.gdn_prefill(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                                               x["dt_bias"], x["state_pool"], x["cache_indices"],
                                               x["cu_seqlens"], scale)
    assert st == 0
    pool = host(d["state_pool"])
    ci = [int(c) for c in x["cache_indices"]]
    cu = x["cu_seqlens"]
    o = host(out)
    for n, slot in enumerate(ci):
        if cu[n + 1] > cu[n]:
            assert max_rel_err(o[cu[n]:cu[n + 1]], out_ref[cu[n]:cu[n + 1]]) <= OUT_TOL, n
            assert max_rel_err(pool[slot], pool_ref[slot]) <= STATE_TOL, n
            # and per value head of the sequence
            o_h = np.moveaxis(o[cu[n]:cu[n + 1]], 1, 0)
            r_h = np.moveaxis(out_ref[cu[n]:cu[n + 1]], 1, 0)
            assert max_rel_err_slices(o_h, r_h, 1) <= OUT_TOL, n
            assert max_rel_err_slices(pool[slot], pool_ref[slot], 1) <= STATE_TOL, n
        else:
            assert np.array_equal(pool[slot], x["state_pool"][slot].astype(np.float64))
    for s in range(pool.shape[0]):
        if s not in ci:
            assert np.array_equal(pool[s], x["state_pool"][s].astype(np.float64)), s


@pytest.mark.parametrize("mild", [False, True])
@pytest.mark.parametrize("seqlens", [[1], [63], [65, 100], [64, 0, 130, 1, 7]])
def test_small_varlen(seqlens, mild):
    x = gi.gdn_prefill_inputs(gi.rng(sum(seqlens) + mild), seqlens, 2, 4, 128, 128,
                              pool=len(seqlens) + 3, mild_gates=mild)
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


def test_long_mild_sequence_carries_the_state():
    # 40 chunks with slow decay: the carried state matters for every chunk
    x = gi.gdn_prefill_inputs(gi.rng(3), [2560 + 17], 1, 2, 128, 128, pool=2, mild_gates=True)
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


def test_full_workload_sampled_units():
    # T = 15360 over 4096 + 2048 + 1024 + 8192 tokens, Hk=16, Hv=32: the whole call on the GPU,
    # the oracle on a sample of (sequence, value head) units, including the 8192-token sequence.
    c = gi.GDN_PREFILL
    x = gi.gdn_prefill_inputs(gi.rng(0), c["seqlens"], c["Hk"], c["Hv"], c["K"], c["V"],
                              c["pool"])
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    o, pool = host(out), host(d["state_pool"])
    cu, ci = x["cu_seqlens"], x["cache_indices"]
    for (n, h) in [(0, 0), (1, 17), (2, 31), (3, 0), (3, 5), (3, 31)]:
        sl = slice(cu[n], cu[n + 1])
        S, o_ref = oracle.gdn_prefill_unit(x["q"][sl], x["k"][sl], x["v"][sl], x["a"][sl],
                                           x["b"][sl], x["A_log"][h], x["dt_bias"][h],
                                           x["state_pool"][ci[n], h], h, scale)
        assert max_rel_err(o[sl, h], o_ref) <= OUT_TOL, (n, h)
        assert max_rel_err(pool[ci[n], h], S) <= STATE_TOL, (n, h)
    for s in range(c["pool"]):
        if s not in set(int(i) for i in ci):
            assert np.array_equal(pool[s], x["state_pool"][s].astype(np.float64))


def test_full_workload_mild_gates_every_head_of_the_split_sequence():
    # the benchmark's lengths (4096 + 2048 + 1024 + 8192) and heads with slow decay, so that the
    # state carried across chunks -- and across the split of the 8192-token sequence into two
    # halves that the fix-up recombines -- matters: all 32 heads of that sequence, and a sample of
    # the others, against the oracle (run over the heads in parallel)
    import os
    from concurrent.futures import ThreadPoolExecutor
    c = gi.GDN_PREFILL
    x = gi.gdn_prefill_inputs(gi.rng(9), c["seqlens"], c["Hk"], c["Hv"], c["K"], c["V"], c["pool"],
                              mild_gates=True)
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    o, pool = host(out), host(d["state_pool"])
    cu, ci = x["cu_seqlens"], x["cache_indices"]
    seq = {n: {k: np.ascontiguousarray(x[k][cu[n]:cu[n + 1]], dtype=np.float64)
               for k in ("q", "k", "v", "a", "b")} for n in range(len(c["seqlens"]))}
    units = [(3, h) for h in range(c["Hv"])] + [(0, 0), (1, 17), (2, 31)]

    def ref(unit):
        n, h = unit
        z = seq[n]
        return oracle.gdn_prefill_unit(z["q"], z["k"], z["v"], z["a"], z["b"], x["A_log"][h],
                                       x["dt_bias"][h], x["state_pool"][ci[n], h], h, scale)

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        refs = list(ex.map(ref, units))
    for (n, h), (S, o_ref) in zip(units, refs):
        sl = slice(cu[n], cu[n + 1])
        assert max_rel_err(o[sl, h], o_ref) <= OUT_TOL, (n, h)
        assert max_rel_err(pool[ci[n], h], S) <= STATE_TOL, (n, h)


@pytest.mark.parametrize("Hk,Hv", [(3, 3), (1, 4)])
def test_key_head_sharing_ratios(Hk, Hv):
    # Hv / Hk = 1 (no sharing) and 4, over several chunks and a short tail
    seqlens = [70, 129]
    x = gi.gdn_prefill_inputs(gi.rng(100 + Hk * Hv), seqlens, Hk, Hv, 128, 128, pool=4, mild_gates=True)
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


@pytest.mark.parametrize("mild", [False, True])
@pytest.mark.parametrize("seqlens", [[1], [65, 100], [64, 0, 130, 1, 7], [300, 20]])
def test_fp16_inputs(seqlens, mild):
    # q, k, v, a, b and out in IEEE binary16 (gdn_prefill_chunked_f16), with a ratio-2 head sharing
    x = gi.gdn_prefill_inputs(gi.rng(500 + sum(seqlens) + mild), seqlens, 2, 4, 128, 128,
                              pool=len(seqlens) + 2, mild_gates=mild, dtype="f16")
    d = _to_dev(x, torch.float16)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert out.dtype == torch.float16 and st == 0
    _check_all(x, d, out, scale)


def test_fp16_long_mild_sequence_carries_the_state():
    x = gi.gdn_prefill_inputs(gi.rng(4), [1280 + 33], 1, 2, 128, 128, pool=2, mild_gates=True,
                              dtype="f16")
    d = _to_dev(x, torch.float16)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


def test_chunk_size_128_gives_the_same_call():
    # chunk size 128 (the page's batched default) selects the same 64-token computation
    x = gi.gdn_prefill_inputs(gi.rng(9), [200, 64, 3], 2, 4, 128, 128, pool=4, mild_gates=True)
    scale = 128 ** -0.5
    d64, d128 = _to_dev(x), _to_dev(x)
    out64, st64 = _gpu(d64, scale)
    out128, st128 = _gpu(d128, scale, chunk_size=128)
    assert st64 == 0 and st128 == 0
    assert torch.equal(out64, out128) and torch.equal(d64["state_pool"], d128["state_pool"])
    _check_all(x, d128, out128, scale)


def test_zero_key_and_query_rows():
    # k = 0 gives k^ = 0 (rk = 1/sqrt(eps) = 1000 multiplies a zero row): the token updates nothing;
    # q = 0 gives a zero output row
    x = gi.gdn_prefill_inputs(gi.rng(31), [70, 5], 1, 2, 128, 128, pool=2, mild_gates=True)
    x["k"][[0, 3, 63, 64, 69, 71]] = 0.0
    x["q"][[1, 64, 72]] = 0.0
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)
    assert not host(out)[[1, 64, 72]].any()


@pytest.mark.parametrize("seqlens", [[150, 64], [700]])
@pytest.mark.parametrize("case", ["no_update", "no_decay", "full_decay"])
def test_gate_extremes(case, seqlens):
    # b -> -inf: beta = 0, the state only decays; a -> -inf: the log-gate is 0 (no decay), so the
    # state carries unchanged in scale and gamma_L = 1 on every chunk; a -> +inf: the chunk decay
    # gamma_L underflows to 0 in fp32 and the update overwrites the state.  700 tokens (11 chunks)
    # with Hv = 2 is a sequence the schedule cuts in two.
    x = gi.gdn_prefill_inputs(gi.rng(41), seqlens, 1, 2, 128, 128, pool=2, mild_gates=True)
    if case == "no_update":
        x["b"][:] = -60.0
    elif case == "no_decay":
        x["a"][:] = -60.0
    else:
        x["a"][:] = 40.0
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


def _split_scratch_bytes(N, T, Hv):
    # the optional tail of the workspace: 3 states per split (8 splits) and one row per scratch
    # chunk (cap // 2), 64 KB each per value head
    cap = (T + 63) // 64 + N
    return (8 * 3 * Hv + (cap // 2) * Hv) * 65536


def _gpu_ws(d, scale, ws_bytes):
    T, Hv = d["v"].shape[0], d["v"].shape[1]
    out = torch.full((T, Hv, 128), SENTINEL, dtype=d["v"].dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                            d["state_pool"], d["cache_indices"], d["cu_seqlens"], 64, scale=scale,
                            out=out, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


@pytest.mark.parametrize("mild", [False, True])
@pytest.mark.parametrize("seqlens", [[1300 + 20, 900, 700, 40], [2000, 3], [64 * 8]])
def test_long_sequences_split_in_two(seqlens, mild):
    # Sequences of 8 or more chunks that set the call's length are cut in two: the second half runs
    # from a zero state and from the identity (v = 0) next to the first half, and the fix-up kernel
    # combines them with the first half's end state.  The first case splits two sequences (21 and 15
    # chunks; 11 chunks would not shorten the call), the second one, the third exactly 8 chunks.
    # With a workspace that lacks the split scratch nothing is split.  Both match the oracle, and
    # each other within the output tolerance.
    N = len(seqlens)
    x = gi.gdn_prefill_inputs(gi.rng(600 + sum(seqlens) + mild), seqlens, 1, 2, 128, 128, pool=N + 2,
                              mild_gates=mild)
    scale = 128 ** -0.5
    full = gdn.gdn_prefill_workspace_size(N, x["T"], 1, 2, 128, 128, 64)
    outs, pools = [], []
    for ws_bytes in (full, full - _split_scratch_bytes(N, x["T"], 2)):
        d = _to_dev(x)
        out, st = _gpu_ws(d, scale, ws_bytes)
        assert st == 0
        _check_all(x, d, out, scale)
        outs.append(host(out))
        pools.append(host(d["state_pool"]))
    assert max_rel_err(outs[0], outs[1]) <= OUT_TOL
    assert max_rel_err(pools[0], pools[1]) <= STATE_TOL


def test_all_sequences_empty():
    # num_seqs > 0 but every sequence is empty (T = 0): nothing is written, the pool is untouched
    x = gi.gdn_prefill_inputs(gi.rng(51), [0, 0, 0], 1, 2, 128, 128, pool=4)
    d = _to_dev(x)
    out, st = _gpu(d, 128 ** -0.5)
    assert st == 0 and out.numel() == 0
    assert np.array_equal(host(d["state_pool"]), x["state_pool"].astype(np.float64))


def test_many_short_sequences():
    # 1100 sequences of 0 to 3 tokens: the chunk offsets are scanned in tiles of 1024 sequences, and
    # every chunk is a short one
    g = gi.rng(77)
    seqlens = [int(v) for v in g.integers(0, 4, size=1100)]
    x = gi.gdn_prefill_inputs(g, seqlens, 1, 2, 128, 128, pool=1100)
    d = _to_dev(x)
    scale = 128 ** -0.5
    out, st = _gpu(d, scale)
    assert st == 0
    _check_all(x, d, out, scale)


def test_workspace_reused_by_two_calls():
    # one workspace, two different batches: nothing of the first call leaks into the second
    scale = 128 ** -0.5
    xa = gi.gdn_prefill_inputs(gi.rng(21), [300, 20], 1, 2, 128, 128, pool=2)
    xb = gi.gdn_prefill_inputs(gi.rng(22), [40, 190, 64], 1, 2, 128, 128, pool=3)
    ws_bytes = max(gdn.gdn_prefill_workspace_size(2, xa["T"], 1, 2, 128, 128, 64),
                   gdn.gdn_prefill_workspace_size(3, xb["T"], 1, 2, 128, 128, 64))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for x in (xa, xb):
        d = _to_dev(x)
        T, Hv = d["v"].shape[0], d["v"].shape[1]
        out = torch.full((T, Hv, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                d["state_pool"], d["cache_indices"], d["cu_seqlens"], 64, scale=scale,
                                out=out, workspace=ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _check_all(x, d, out, scale)


def test_split_call_equals_one_call():
    # one sequence as one call, and as two calls that carry the state through the pool
    x = gi.gdn_prefill_inputs(gi.rng(9), [200], 1, 2, 128, 128, pool=1, mild_gates=True)
    scale = 128 ** -0.5
    d1 = _to_dev(x)
    out1, _ = _gpu(d1, scale)
    d2 = _to_dev(x)
    first = dict(d2, cu_seqlens=dev(np.array([0, 128]), torch.int64))
    outa, _ = _gpu(first, scale)
    second = {k: (v[128:].contiguous() if k in ("q", "k", "v", "a", "b") else v) for k, v in d2.items()}
    second["cu_seqlens"] = dev(np.array([0, 72]), torch.int64)
    outb, _ = _gpu(second, scale)
    both = torch.cat([outa[:128], outb], dim=0)
    o1, o2 = host(out1), host(both)
    assert max_rel_err(o2, o1) <= OUT_TOL
    assert max_rel_err(host(d2["state_pool"]), host(d1["state_pool"])) <= STATE_TOL


def test_bad_slots_and_bounds_are_flagged_and_skipped():
    x = gi.gdn_prefill_inputs(gi.rng(11), [70, 30], 1, 2, 128, 128, pool=3)
    scale = 128 ** -0.5
    x["cache_indices"] = np.array([5, 1], dtype=np.int64)   # 5 is outside the pool of 3
    d = _to_dev(x)
    out, st = _gpu(d, scale)
    assert st & gdn.STATUS_BAD_CACHE_INDEX
    o = host(out)
    assert np.all(o[:70] == SENTINEL)              # skipped sequence: out not written
    pool = host(d["state_pool"])
    assert np.array_equal(pool[0], x["state_pool"][0].astype(np.float64))
    assert np.array_equal(pool[2], x["state_pool"][2].astype(np.float64))
    pool_ref, out_ref, _ = oracle.gdn_prefill(x["q"], x["k"], x["v"], x["a"], x["b"], x["A_log"],
                                              x["dt_bias"], x["state_pool"], x["cache_indices"],
                                              x["cu_seqlens"], scale)
    assert max_rel_err(o[70:], out_ref[70:]) <= OUT_TOL
    assert max_rel_err(pool[1], pool_ref[1]) <= STATE_TOL
    x["cache_indices"] = np.array([0, 1], dtype=np.int64)
    x["cu_seqlens"] = np.array([0, 80, 60], dtype=np.int64)  # decreasing bound
    d = _to_dev(x)
    _, st = _gpu(d, scale)
    assert st & gdn.STATUS_BAD_SEQLENS


def test_rejections():
    x = gi.gdn_prefill_inputs(gi.rng(12), [10], 1, 2, 128, 128, pool=1)
    d = _to_dev(x)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                d["state_pool"], d["cache_indices"], d["cu_seqlens"], 96)
    assert e.value.status == gdn.GDN_ERR_UNSUPPORTED  # chunk sizes other than 64 and 128


def _plan(ws, N, T):
    # the schedule in the workspace header (layout in gdn.h): after the chunk offsets (8 bytes per
    # sequence + 1, padded to 16) and the chunk table (16 bytes per chunk of cap), the plan
    # (int ntask, int nsplit, int64 nscr), num_seqs + 16 tasks (int4) and 8 splits (int4:
    # sequence, first-part chunks, first scratch chunk)
    cap = (T + 63) // 64 + N
    off = (8 * (N + 1) + 15) // 16 * 16 + 16 * cap
    raw = ws.cpu().numpy()
    ntask, nsplit = (int(v) for v in raw[off:off + 8].view(np.int32))
    nscr = int(raw[off + 8:off + 16].view(np.int64)[0])
    tasks = raw[off + 16:off + 16 + 16 * (N + 16)].view(np.int32).reshape(-1, 4)[:ntask, :3]
    so = off + 16 + 16 * (N + 16)
    splits = raw[so:so + 16 * 8].view(np.int32).reshape(-1, 4)[:nsplit, :3]
    return ntask, nsplit, nscr, tasks.tolist(), splits.tolist()


@pytest.mark.parametrize("seqlens,Hv,expect", [
    # 21, 15, 11 and 1 chunks, 2 value heads: cut 21 -> 11 + 10 and 15 -> 8 + 7; cutting 11 would
    # not shorten the longest chain (11) by 10 %
    ([1300 + 20, 900, 700, 40], 2, [[0, 11, 0], [1, 8, 10]]),
    # the benchmark's lengths with 32 value heads: only the 8192-token sequence (128 chunks) is cut
    ([4096, 2048, 1024, 8192], 32, [[3, 64, 0]]),
    # 7 chunks: below the 8-chunk minimum
    ([448], 2, []),
])
def test_split_schedule(seqlens, Hv, expect):
    N = len(seqlens)
    x = gi.gdn_prefill_inputs(gi.rng(3), seqlens, 1, Hv, 128, 128, pool=N + 1, mild_gates=True)
    d = _to_dev(x)
    T = x["T"]
    ws = torch.empty(gdn.gdn_prefill_workspace_size(N, T, 1, Hv, 128, 128, 64), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["state_pool"],
                            d["cache_indices"], d["cu_seqlens"], 64, out=None, workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ntask, nsplit, nscr, tasks, splits = _plan(ws, N, T)
    assert splits == expect
    assert nsplit == len(expect) and ntask == N + 2 * nsplit
    assert nscr == sum((seqlens[s] + 63) // 64 - n1 for s, n1, _ in expect)
    # tasks: the split sequences' three chains first (first part, zero start, identity start), then
    # the other sequences in order; every sequence appears
    split_seqs = [s for s, _, _ in expect]
    want = [[s, kind, j] for j, s in enumerate(split_seqs) for kind in (1, 2, 3)]
    want += [[n, 0, 0] for n in range(N) if n not in split_seqs]
    assert tasks == want


def test_split_with_more_fixup_jobs_than_sms():
    # One 200-chunk sequence over 80 value heads: the schedule splits it 100 + 100, and the fix-up's
    # jobs (a state job and a chunk job per head, 160) outnumber its one-CTA-per-SM grid, so some
    # CTAs run two jobs (fresh barriers for the second).  The oracle runs on sampled heads.
    Hk, Hv = 8, 80
    seqlens = [200 * 64 - 5]
    x = gi.gdn_prefill_inputs(gi.rng(77), seqlens, Hk, Hv, 128, 128, pool=2, mild_gates=True)
    d = _to_dev(x)
    scale = 128 ** -0.5
    T = x["T"]
    ws = torch.empty(gdn.gdn_prefill_workspace_size(1, T, Hk, Hv, 128, 128, 64), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                  d["state_pool"], d["cache_indices"], d["cu_seqlens"], 64, scale=scale,
                                  workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ntask, nsplit, nscr, tasks, splits = _plan(ws, 1, T)
    assert splits == [[0, 100, 0]] and nscr == 100
    o, pool = host(out), host(d["state_pool"])
    slot = int(x["cache_indices"][0])
    for h in (0, 41, 79):  # the unit oracle on the one key head and value head involved
        hk = h // (Hv // Hk)
        S, o_ref = oracle.gdn_prefill_unit(x["q"][:, hk:hk + 1], x["k"][:, hk:hk + 1], x["v"][:, h:h + 1],
                                           x["a"][:, h:h + 1], x["b"][:, h:h + 1], x["A_log"][h], x["dt_bias"][h],
                                           x["state_pool"][slot, h], 0, scale)
        assert max_rel_err(o[:, h], o_ref) <= OUT_TOL, h
        assert max_rel_err(pool[slot, h], S) <= STATE_TOL, h
