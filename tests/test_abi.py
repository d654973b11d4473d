"""The C ABI without a GPU: libgdn.so builds, loads and exports every function include/gdn.h
declares, and host-side validation rejects bad arguments before anything is launched (these calls
return before the first CUDA call, so they run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_delta_gb300 as gdn
from gated_deltanet_delta_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdn.load()


def _declared():
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(\w+)\s*\(", text)) - {"defined"}


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert declared == set(gdn.ABI_SYMBOLS), declared ^ set(gdn.ABI_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(5):
        assert gdn.status_string(s)


N = None
P = ctypes.c_void_p(16)  # a non-null, 16-byte aligned dummy (never dereferenced by these calls)


def test_decode_validation(lib):
    f = lib.gdn_decode_step
    # Hv not a multiple of Hk
    assert f(P, P, P, P, P, P, P, P, 0, 1, 3, 4, 128, 128, 1.0, N) == gdn.GDN_ERR_INVALID_ARG
    assert "multiple" in gdn.last_error()
    # unsupported Dk
    assert f(P, P, P, P, P, P, P, P, 0, 1, 1, 1, 96, 128, 1.0, N) == gdn.GDN_ERR_UNSUPPORTED
    # null pointer
    assert f(N, P, P, P, P, P, P, P, 0, 1, 1, 1, 128, 128, 1.0, N) == gdn.GDN_ERR_INVALID_ARG
    # bad output dtype code
    assert f(P, P, P, P, P, P, P, P, 7, 1, 1, 1, 128, 128, 1.0, N) == gdn.GDN_ERR_INVALID_ARG
    # partially overlapping state buffers
    assert f(ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 512), P, P, P, P, P, P, 0, 1, 1, 1,
             128, 128, 1.0, N) == gdn.GDN_ERR_INVALID_ARG
    # misaligned state
    assert f(ctypes.c_void_p(4100), ctypes.c_void_p(4100), P, P, P, P, P, P, 0, 1, 1, 1, 128, 128,
             1.0, N) == gdn.GDN_ERR_INVALID_ARG
    # B = 0 is a no-op even with null pointers
    assert f(N, N, N, N, N, N, N, N, 0, 0, 1, 1, 128, 128, 1.0, N) == gdn.GDN_OK


def test_comba_validation(lib):
    f = lib.comba_decode_step
    assert f(P, P, P, P, P, P, P, P, P, 0, 1, 1, 96, 128, 1.0, N) == gdn.GDN_ERR_UNSUPPORTED
    assert f(P, P, P, P, P, P, P, P, N, 0, 1, 1, 128, 128, 1.0, N) == gdn.GDN_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 64), P, P, P, P, P, P, P, 0, 1,
             1, 128, 128, 1.0, N) == gdn.GDN_ERR_INVALID_ARG
    assert f(N, N, N, N, N, N, N, N, N, 0, 0, 4, 128, 128, 1.0, N) == gdn.GDN_OK


def test_window_validation(lib):
    f = lib.gdn_window_fused
    args = [P] * 12
    assert f(*args, 1, 2, 4, 9, 1, 1e-6, N) == gdn.GDN_ERR_UNSUPPORTED     # ntok > 8
    assert f(*args, 1, 4, 2, 2, 1, 1e-6, N) == gdn.GDN_ERR_UNSUPPORTED     # h_k > h_v
    assert f(*args, 1, 2, 4, 3, 0x104, 1e-6, N) == gdn.GDN_ERR_INVALID_ARG  # commit after token 4 of 3
    assert f(*args, 1, 2, 4, 3, 2, 1e-6, N) == gdn.GDN_ERR_INVALID_ARG      # unknown commit code
    assert f(*([N] * 12), 0, 2, 4, 3, 1, 1e-6, N) == gdn.GDN_OK            # N = 0
    # hist_out aliasing hist
    h = ctypes.c_void_p(1 << 24)
    a = [P, h, h] + [P] * 9
    assert f(*a, 1, 2, 4, 3, 1, 1e-6, N) == gdn.GDN_ERR_INVALID_ARG


def test_prefill_workspace_size(lib):
    # header: chunk offsets (8 bytes per sequence + 1, padded to 16), the chunk table (16 bytes per
    # chunk), the schedule (16 bytes, then 16 per task for num_seqs + 16 tasks, 16 per split for 8
    # splits, 16 per scratch chunk), padded to 1 KB; one 66,560-byte record per (chunk, value head)
    # for up to cap = ceil(T / 64) + num_seqs chunks; then the split scratch: 3 states of 64 KB per
    # split (8) and value head, one 64 KB row per scratch chunk (cap // 2) and value head
    def size(n, T, Hv):
        cap = (T + 63) // 64 + n
        cap2 = cap // 2
        head = (8 * (n + 1) + 15) // 16 * 16 + 16 * cap + 16 + 16 * (n + 16) + 16 * 8 + 16 * cap2
        head = (head + 1023) // 1024 * 1024
        return head + cap * Hv * 66560 + 8 * 3 * Hv * 65536 + cap2 * Hv * 65536
    assert size(4, 15360, 32) == 7168 + 244 * 32 * 66560 + 24 * 32 * 65536 + 122 * 32 * 65536
    assert gdn.gdn_prefill_workspace_size(4, 15360, 16, 32, 128, 128, 64) == size(4, 15360, 32)
    assert gdn.gdn_prefill_workspace_size(200, 65, 1, 2, 128, 128, 64) == size(200, 65, 2)
    assert gdn.gdn_prefill_workspace_size(0, 100, 1, 1, 128, 128, 64) == 0
    assert gdn.gdn_prefill_workspace_size(1, 100, 1, 1, 64, 128, 64) == 0    # unsupported K
    assert gdn.gdn_prefill_workspace_size(1, 100, 2, 3, 128, 128, 64) == 0   # Hv % Hk != 0
    # chunk size 128 (the page's batched default) runs the same 64-token chunks: same workspace
    assert gdn.gdn_prefill_workspace_size(4, 15360, 16, 32, 128, 128, 128) == \
        gdn.gdn_prefill_workspace_size(4, 15360, 16, 32, 128, 128, 64)
    assert gdn.gdn_prefill_workspace_size(4, 15360, 16, 32, 128, 128, 96) == 0


@pytest.mark.parametrize("name", ["gdn_prefill_chunked", "gdn_prefill_chunked_f16"])
def test_prefill_validation(lib, name):
    f = getattr(lib, name)
    pool, out = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 40)
    need = gdn.gdn_prefill_workspace_size(2, 100, 1, 2, 128, 128, 64)

    def call(ws, ws_bytes, chunk=64, num_seqs=2, K=128):
        return f(P, P, P, P, P, P, P, pool, 4, P, P, num_seqs, 100, 1, 2, K, 128, chunk, 1.0, out,
                 ws, ws_bytes, P, N)
    ws = ctypes.c_void_p(1 << 44)
    assert call(N, 0) == gdn.GDN_ERR_INVALID_ARG and "workspace" in gdn.last_error()
    # the header and the records are required; the split scratch (3 states per split for 8 splits,
    # one row per scratch chunk, cap // 2 = 2 of them, 64 KB each per value head) is optional
    need_min = need - (8 * 3 * 2 + 2 * 2) * 65536
    assert call(ws, need_min - 1) == gdn.GDN_ERR_INVALID_ARG and "needed" in gdn.last_error()
    assert str(need_min) in gdn.last_error()
    assert gdn.last_error().startswith(name + ":")
    assert call(ctypes.c_void_p((1 << 44) + 16), need) == gdn.GDN_ERR_INVALID_ARG   # misaligned
    assert call(ctypes.c_void_p((1 << 40) - 256), need) == gdn.GDN_ERR_INVALID_ARG  # overlaps out
    assert call(ws, need, chunk=32) == gdn.GDN_ERR_UNSUPPORTED and "64 or 128" in gdn.last_error()
    assert call(ws, need, K=64) == gdn.GDN_ERR_UNSUPPORTED
    assert call(N, 0, num_seqs=0) == gdn.GDN_OK


def test_comba_prefill_validation(lib):
    f = lib.comba_prefill_chunked
    pool, out = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 40)
    need = gdn.gdn_prefill_workspace_size(2, 100, 2, 2, 128, 128, 64)
    ws = ctypes.c_void_p(1 << 44)

    def call(ws=ws, ws_bytes=need, chunk=64, num_seqs=2, K=128, p=P, g=P, beta=P):
        # (q, k, v, p, beta, g, state_pool, pool_size, cache_indices, cu_seqlens, num_seqs, T, H, K, V,
        #  chunk_size, scale, out, workspace, workspace_bytes, dev_status, stream)
        return f(P, P, P, p, beta, g, pool, 4, P, P, num_seqs, 100, 2, K, 128, chunk, 1.0, out, ws, ws_bytes, P, N)
    assert call(ws=N, ws_bytes=0) == gdn.GDN_ERR_INVALID_ARG and "workspace" in gdn.last_error()
    assert gdn.last_error().startswith("comba_prefill_chunked:")
    assert call(p=N) == gdn.GDN_ERR_INVALID_ARG and "null token pointer" in gdn.last_error()
    assert call(p=ctypes.c_void_p(24)) == gdn.GDN_ERR_INVALID_ARG   # p must be 16-byte aligned
    assert call(g=ctypes.c_void_p(18)) == gdn.GDN_ERR_INVALID_ARG   # g must be 4-byte aligned
    assert call(chunk=32) == gdn.GDN_ERR_UNSUPPORTED and "64 or 128" in gdn.last_error()
    assert call(K=64) == gdn.GDN_ERR_UNSUPPORTED
    assert call(ws=N, ws_bytes=0, num_seqs=0) == gdn.GDN_OK


def test_comba_forward_validation(lib):
    f = lib.comba_forward
    st, o = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 40)

    def call(state=st, K=128, V=128, o_dtype=gdn.GDN_BF16, B=2, T=4, ptr=P, out=o):
        return f(state, ptr, ptr, ptr, ptr, ptr, ptr, out, o_dtype, B, T, 2, K, V, 0.1, N)
    assert call(K=96) == gdn.GDN_ERR_UNSUPPORTED and "64 or 128" in gdn.last_error()
    assert call(o_dtype=7) == gdn.GDN_ERR_INVALID_ARG
    assert call(state=N) == gdn.GDN_ERR_INVALID_ARG
    assert call(ptr=N) == gdn.GDN_ERR_INVALID_ARG
    assert call(state=ctypes.c_void_p((1 << 20) + 4)) == gdn.GDN_ERR_INVALID_ARG      # misaligned
    assert call(out=ctypes.c_void_p((1 << 20) + 64)) == gdn.GDN_ERR_INVALID_ARG       # o overlaps state
    assert call(B=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(B=0, state=N, ptr=N, out=N) == gdn.GDN_OK                               # no heads: no-op


def test_prefill_wait_limit_is_a_host_setting(lib):
    # a process-wide host value read at launch: setting and restoring it needs no GPU
    gdn.set_prefill_wait_limit(1)
    gdn.set_prefill_wait_limit(1 << 30)
    gdn.set_prefill_wait_limit(0)
    lib.gdn_prefill_set_wait_limit(ctypes.c_uint32(0xFFFFFFFF))
    lib.gdn_prefill_set_wait_limit(ctypes.c_uint32(0))
