"""Python binding of libgdn, the GB300 (sm_103a) gated delta-rule library.

Argument marshalling only: every function checks dtypes, shapes and contiguity of torch CUDA
tensors, allocates outputs the caller did not provide, and calls the C ABI (include/gdn.h) with raw
device pointers on the current CUDA stream.  Every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if libgdn.so is missing or cannot be loaded, the first call
raises.

Build the library with ``python -m gated_deltanet_delta_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_TIMEOUT = range(5)
GDN_BF16, GDN_F32 = 0, 1
STATUS_BAD_CACHE_INDEX = 1
STATUS_BAD_SEQLENS = 2
STATUS_TIMEOUT = 4

# Every symbol that include/gdn.h declares.
ABI_SYMBOLS = ("gdn_decode_step", "gdn_decode_multi", "gdn_decode_step_pooled", "comba_decode_step", "comba_forward",
               "gdn_prefill_workspace_size",
               "gdn_prefill_chunked", "gdn_prefill_chunked_f16", "gdn_prefill_chunked_noalloc",
               "comba_prefill_chunked", "gdn_window_fused", "gdn_prefill_set_wait_limit",
               "gdn_status_string", "gdn_last_error")


class GdnError(RuntimeError):
    """A libgdn call returned a status other than GDN_OK."""

    def __init__(self, status: int, what: str, detail: str):
        super().__init__(f"{what}: {detail or 'status ' + str(status)}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so (once) and declare the C signatures.  Raises OSError if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise OSError(f"{path} is not built: run `python -m gated_deltanet_delta_gb300.build` "
                          "(the CUDA library is required; there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, I, F, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint
        I64, SZ = ctypes.c_int64, ctypes.c_size_t
        lib.gdn_decode_step.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.gdn_decode_step.restype = I
        lib.gdn_decode_multi.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.gdn_decode_multi.restype = I
        lib.gdn_decode_step_pooled.argtypes = [P, I, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P]
        lib.gdn_decode_step_pooled.restype = I
        lib.comba_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
        lib.comba_decode_step.restype = I
        lib.comba_forward.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.comba_forward.restype = I
        lib.gdn_prefill_workspace_size.argtypes = [I, I64, I, I, I, I, I]
        lib.gdn_prefill_workspace_size.restype = SZ
        lib.gdn_prefill_chunked.argtypes = [P, P, P, P, P, P, P, P, I, P, P, I, I64, I, I, I, I, I,
                                            F, P, P, SZ, P, P]
        lib.gdn_prefill_chunked.restype = I
        lib.gdn_prefill_chunked_f16.argtypes = lib.gdn_prefill_chunked.argtypes
        lib.gdn_prefill_chunked_f16.restype = I
        lib.comba_prefill_chunked.argtypes = [P, P, P, P, P, P, P, I, P, P, I, I64, I, I, I, I, F, P, P, SZ,
                                              P, P]
        lib.comba_prefill_chunked.restype = I
        lib.gdn_prefill_chunked_noalloc.argtypes = [P, P, P, P, P, P, P, P, I, P, P, I, I64, I, I, I,
                                                    I, I, F, P, P, P]
        lib.gdn_prefill_chunked_noalloc.restype = I
        lib.gdn_window_fused.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, U, F, P]
        lib.gdn_window_fused.restype = I
        lib.gdn_prefill_set_wait_limit.argtypes = [ctypes.c_uint32]
        lib.gdn_prefill_set_wait_limit.restype = None
        lib.gdn_status_string.argtypes = [I]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def set_prefill_wait_limit(polls: int) -> None:
    """Bound every device-side wait of the prefill kernels to `polls` mbarrier polls (0: the
    built-in limits).  A wait that runs out sets STATUS_TIMEOUT in the call's dev_status."""
    load().gdn_prefill_set_wait_limit(int(polls))


def last_error() -> str:
    return load().gdn_last_error().decode()


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != GDN_OK:
        raise GdnError(status, what, last_error())


# ------------------------------------------------------------------------------------------------
# torch marshalling helpers (torch is imported lazily so that the ABI can be loaded without it)
# ------------------------------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def _want(t, name: str, dtype, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _out_code(dtype) -> int:
    torch = _torch()
    if dtype == torch.bfloat16:
        return GDN_BF16
    if dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"output dtype must be torch.bfloat16 or torch.float32, got {dtype}")


# ------------------------------------------------------------------------------------------------
# Operations
# ------------------------------------------------------------------------------------------------
def gdn_decode_step(state_in, q, k, v, g, beta, scale=None, state_out=None, y=None,
                    y_dtype=None):
    """One GDN decode step.  state_in f32 [B,Hv,Dv,Dk]; q,k bf16 [B,Hk,Dk]; v bf16 [B,Hv,Dv];
    g f32 [B,Hv] (linear gate); beta bf16 [B,Hv].  Returns (state_out, y).  state_out may be
    state_in (in place).  scale defaults to Dk^-0.5."""
    torch = _torch()
    B, Hv, Dv, Dk = state_in.shape
    Hk = q.shape[1]
    _want(state_in, "state_in", torch.float32)
    _want(q, "q", torch.bfloat16, (B, Hk, Dk))
    _want(k, "k", torch.bfloat16, (B, Hk, Dk))
    _want(v, "v", torch.bfloat16, (B, Hv, Dv))
    _want(g, "g", torch.float32, (B, Hv))
    _want(beta, "beta", torch.bfloat16, (B, Hv))
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _want(state_out, "state_out", torch.float32, state_in.shape)
    if y is None:
        y = torch.empty((B, Hv, Dv), dtype=y_dtype or torch.bfloat16, device=state_in.device)
    _want(y, "y", y.dtype, (B, Hv, Dv))
    scale = Dk ** -0.5 if scale is None else float(scale)
    _check(load().gdn_decode_step(_ptr(state_in), _ptr(state_out), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(g), _ptr(beta), _ptr(y), _out_code(y.dtype), B, Hk, Hv, Dk,
                                  Dv, scale, _stream(state_in.device)), "gdn_decode_step")
    return state_out, y


def gdn_decode_multi(state_in, q, k, v, g, beta, scale=None, state_out=None, y=None, y_dtype=None):
    """T consecutive GDN decode steps.  state_in f32 [B,Hv,Dv,Dk]; q,k bf16 [B,T,Hk,Dk];
    v bf16 [B,T,Hv,Dv]; g f32 [B,T,Hv]; beta bf16 [B,T,Hv].  Returns (state_out, y [B,T,Hv,Dv])."""
    torch = _torch()
    B, Hv, Dv, Dk = state_in.shape
    T, Hk = q.shape[1], q.shape[2]
    _want(state_in, "state_in", torch.float32)
    _want(q, "q", torch.bfloat16, (B, T, Hk, Dk))
    _want(k, "k", torch.bfloat16, (B, T, Hk, Dk))
    _want(v, "v", torch.bfloat16, (B, T, Hv, Dv))
    _want(g, "g", torch.float32, (B, T, Hv))
    _want(beta, "beta", torch.bfloat16, (B, T, Hv))
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _want(state_out, "state_out", torch.float32, state_in.shape)
    if y is None:
        y = torch.empty((B, T, Hv, Dv), dtype=y_dtype or torch.bfloat16, device=state_in.device)
    _want(y, "y", y.dtype, (B, T, Hv, Dv))
    scale = Dk ** -0.5 if scale is None else float(scale)
    _check(load().gdn_decode_multi(_ptr(state_in), _ptr(state_out), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(g), _ptr(beta), _ptr(y), _out_code(y.dtype), B, T, Hk, Hv,
                                   Dk, Dv, scale, _stream(state_in.device)), "gdn_decode_multi")
    return state_out, y


def gdn_decode_step_pooled(state_pool, cache_indices, q, k, v, g, beta, scale=None, y=None,
                           y_dtype=None, dev_status=None):
    """One GDN decode step on a pooled state, in place: batch row b uses slot cache_indices[b] of
    state_pool f32 [pool,Hv,Dv,Dk].  q,k bf16 [B,Hk,Dk]; v bf16 [B,Hv,Dv]; g f32 [B,Hv];
    beta bf16 [B,Hv].  Returns y.  dev_status (int32 [1], zeroed) receives STATUS_BAD_CACHE_INDEX."""
    torch = _torch()
    _want(state_pool, "state_pool", torch.float32)
    pool, Hv, Dv, Dk = state_pool.shape
    B, Hk = q.shape[0], q.shape[1]
    _want(cache_indices, "cache_indices", torch.int64, (B,))
    _want(q, "q", torch.bfloat16, (B, Hk, Dk))
    _want(k, "k", torch.bfloat16, (B, Hk, Dk))
    _want(v, "v", torch.bfloat16, (B, Hv, Dv))
    _want(g, "g", torch.float32, (B, Hv))
    _want(beta, "beta", torch.bfloat16, (B, Hv))
    if y is None:
        y = torch.empty((B, Hv, Dv), dtype=y_dtype or torch.bfloat16, device=state_pool.device)
    _want(y, "y", y.dtype, (B, Hv, Dv))
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=state_pool.device)
    _want(dev_status, "dev_status", torch.int32, (1,))
    scale = Dk ** -0.5 if scale is None else float(scale)
    _check(load().gdn_decode_step_pooled(_ptr(state_pool), pool, _ptr(cache_indices), _ptr(q),
                                         _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(y),
                                         _out_code(y.dtype), B, Hk, Hv, Dk, Dv, scale,
                                         _ptr(dev_status), _stream(state_pool.device)),
           "gdn_decode_step_pooled")
    return y


def comba_decode_step(state, q, k, v, p, beta, g, scale=None, state_new=None, o=None,
                      o_dtype=None):
    """One Comba decode step.  state f32 [B,H,K,V]; q,k,p bf16 [B,H,K]; v bf16 [B,H,V];
    beta bf16 [B,H]; g f32 [B,H] (log-decay).  Returns (state_new, o).  state_new may be state
    (in place).  scale defaults to K^-0.5."""
    torch = _torch()
    B, H, K, V = state.shape
    _want(state, "state", torch.float32)
    for name, t in (("q", q), ("k", k), ("p", p)):
        _want(t, name, torch.bfloat16, (B, H, K))
    _want(v, "v", torch.bfloat16, (B, H, V))
    _want(beta, "beta", torch.bfloat16, (B, H))
    _want(g, "g", torch.float32, (B, H))
    if state_new is None:
        state_new = torch.empty_like(state)
    _want(state_new, "state_new", torch.float32, state.shape)
    if o is None:
        o = torch.empty((B, H, V), dtype=o_dtype or torch.bfloat16, device=state.device)
    _want(o, "o", o.dtype, (B, H, V))
    scale = K ** -0.5 if scale is None else float(scale)
    _check(load().comba_decode_step(_ptr(state), _ptr(state_new), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(p), _ptr(beta), _ptr(g), _ptr(o), _out_code(o.dtype), B, H,
                                    K, V, scale, _stream(state.device)), "comba_decode_step")
    return state_new, o


def comba_forward(state, q, k, v, p, beta, g, scale=None, o=None, o_dtype=None):
    """The Comba recurrence over T tokens.  state f32 [B,H,K,V] (updated in place); q,k,p bf16
    [B,T,H,K]; v bf16 [B,T,H,V]; beta bf16 [B,T,H]; g f32 [B,T,H] (log-decay).  Returns o
    [B,T,H,V] (bf16 unless o / o_dtype say float32); scale defaults to K^-0.5."""
    torch = _torch()
    B, H, K, V = state.shape
    T = q.shape[1]
    _want(state, "state", torch.float32)
    _want(q, "q", torch.bfloat16, (B, T, H, K))
    _want(k, "k", torch.bfloat16, (B, T, H, K))
    _want(p, "p", torch.bfloat16, (B, T, H, K))
    _want(v, "v", torch.bfloat16, (B, T, H, V))
    _want(beta, "beta", torch.bfloat16, (B, T, H))
    _want(g, "g", torch.float32, (B, T, H))
    if o is None:
        o = torch.empty((B, T, H, V), dtype=o_dtype or torch.bfloat16, device=state.device)
    _want(o, "o", o.dtype, (B, T, H, V))
    scale = K ** -0.5 if scale is None else float(scale)
    _check(load().comba_forward(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(p), _ptr(beta), _ptr(g),
                                _ptr(o), _out_code(o.dtype), B, T, H, K, V, scale,
                                _stream(state.device)), "comba_forward")
    return o


def gdn_prefill_workspace_size(num_seqs: int, T: int, Hk: int, Hv: int, K: int, V: int,
                               chunk_size: int = 64) -> int:
    return int(load().gdn_prefill_workspace_size(num_seqs, T, Hk, Hv, K, V, chunk_size))


def gdn_prefill_chunked(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens,
                        chunk_size: int = 64, scale=None, out=None, workspace=None,
                        dev_status=None):
    """Varlen chunkwise prefill.  q,k [T,Hk,K]; v [T,Hv,V]; a,b [T,Hv], all bf16 or all float16
    (q's dtype selects gdn_prefill_chunked or gdn_prefill_chunked_f16); A_log, dt_bias f32 [Hv];
    state_pool f32 [pool,Hv,V,K] (updated in place); cache_indices int64 [N]; cu_seqlens int64
    [N+1].  Returns out [T,Hv,V] in q's dtype.  dev_status (int32 [1], zeroed by the caller)
    receives STATUS_* bits for skipped sequences; scale defaults to K^-0.5."""
    torch = _torch()
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cache_indices.shape[0]
    dt = q.dtype if q.dtype == torch.float16 else torch.bfloat16
    _want(q, "q", dt)
    _want(k, "k", dt, (T, Hk, K))
    _want(v, "v", dt, (T, Hv, V))
    _want(a, "a", dt, (T, Hv))
    _want(b, "b", dt, (T, Hv))
    _want(A_log, "A_log", torch.float32, (Hv,))
    _want(dt_bias, "dt_bias", torch.float32, (Hv,))
    _want(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (Hv, V, K):
        raise ValueError(f"state_pool must be [pool,{Hv},{V},{K}], got {tuple(state_pool.shape)}")
    _want(cache_indices, "cache_indices", torch.int64, (N,))
    _want(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,))
    if out is None:
        out = torch.empty((T, Hv, V), dtype=dt, device=q.device)
    _want(out, "out", dt, (T, Hv, V))
    ws_bytes = gdn_prefill_workspace_size(N, T, Hk, Hv, K, V, chunk_size)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    _want(dev_status, "dev_status", torch.int32, (1,))
    scale = K ** -0.5 if scale is None else float(scale)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    name = "gdn_prefill_chunked_f16" if dt == torch.float16 else "gdn_prefill_chunked"
    _check(getattr(load(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                                 _ptr(dt_bias), _ptr(state_pool), state_pool.shape[0],
                                 _ptr(cache_indices), _ptr(cu_seqlens), N, T, Hk, Hv, K, V,
                                 int(chunk_size), scale, _ptr(out), _ptr(workspace), wsz,
                                 _ptr(dev_status), _stream(q.device)), name)
    return out


def comba_prefill_chunked(q, k, v, p, beta, g, state_pool, cache_indices, cu_seqlens, chunk_size: int = 64,
                          scale=None, out=None, workspace=None, dev_status=None):
    """Varlen chunkwise prefill of the Comba recurrence.  q, k, p [T,H,K] and v [T,H,V] bf16; beta
    bf16 [T,H]; g f32 [T,H] (log decay); state_pool f32 [pool,H,K,V] (updated in place);
    cache_indices int64 [N]; cu_seqlens int64 [N+1].  Returns out bf16 [T,H,V]; scale defaults to
    K^-0.5."""
    torch = _torch()
    T, H, K = q.shape
    V = v.shape[2]
    N = cache_indices.shape[0]
    bf = torch.bfloat16
    _want(q, "q", bf)
    _want(k, "k", bf, (T, H, K))
    _want(p, "p", bf, (T, H, K))
    _want(v, "v", bf, (T, H, V))
    _want(beta, "beta", bf, (T, H))
    _want(g, "g", torch.float32, (T, H))
    _want(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, K, V):
        raise ValueError(f"state_pool must be [pool,{H},{K},{V}], got {tuple(state_pool.shape)}")
    _want(cache_indices, "cache_indices", torch.int64, (N,))
    _want(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,))
    if out is None:
        out = torch.empty((T, H, V), dtype=bf, device=q.device)
    _want(out, "out", bf, (T, H, V))
    ws_bytes = gdn_prefill_workspace_size(N, T, H, H, K, V, chunk_size)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    _want(dev_status, "dev_status", torch.int32, (1,))
    scale = K ** -0.5 if scale is None else float(scale)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().comba_prefill_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(p), _ptr(beta), _ptr(g), _ptr(state_pool),
                                        state_pool.shape[0], _ptr(cache_indices), _ptr(cu_seqlens), N, T, H, K, V,
                                        int(chunk_size), scale, _ptr(out), _ptr(workspace), wsz, _ptr(dev_status),
                                        _stream(q.device)), "comba_prefill_chunked")
    return out


def gdn_prefill_chunked_noalloc(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens,
                                chunk_size: int = 64, scale=None, out=None, dev_status=None):
    """gdn_prefill_chunked for callers that cannot allocate device memory: the same arguments and
    results without a workspace; the library's own fixed 64 MiB device scratch serves instead.
    Workloads needing more than that raise GdnError (GDN_ERR_UNSUPPORTED).  Calls on one device
    share the scratch, so calls that run concurrently on the GPU race: order them on one stream.
    This wrapper allocates out and dev_status only when they are not given."""
    torch = _torch()
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    N = cache_indices.shape[0]
    _want(q, "q", torch.bfloat16)
    _want(k, "k", torch.bfloat16, (T, Hk, K))
    _want(v, "v", torch.bfloat16, (T, Hv, V))
    _want(a, "a", torch.bfloat16, (T, Hv))
    _want(b, "b", torch.bfloat16, (T, Hv))
    _want(A_log, "A_log", torch.float32, (Hv,))
    _want(dt_bias, "dt_bias", torch.float32, (Hv,))
    _want(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (Hv, V, K):
        raise ValueError(f"state_pool must be [pool,{Hv},{V},{K}], got {tuple(state_pool.shape)}")
    _want(cache_indices, "cache_indices", torch.int64, (N,))
    _want(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,))
    if out is None:
        out = torch.empty((T, Hv, V), dtype=torch.bfloat16, device=q.device)
    _want(out, "out", torch.bfloat16, (T, Hv, V))
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    _want(dev_status, "dev_status", torch.int32, (1,))
    scale = K ** -0.5 if scale is None else float(scale)
    _check(load().gdn_prefill_chunked_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                                              _ptr(dt_bias), _ptr(state_pool), state_pool.shape[0],
                                              _ptr(cache_indices), _ptr(cu_seqlens), N, T, Hk, Hv, K, V,
                                              int(chunk_size), scale, _ptr(out), _ptr(dev_status),
                                              _stream(q.device)), "gdn_prefill_chunked_noalloc")
    return out


def gdn_window_fused(state, hist, hist_out, qkv, alpha, beta, z, conv_w, dt, ssm_a, gamma,
                     h_k: int, commit: int, eps: float = 1e-6, y=None):
    """Fused decode window.  state f32 [N,128,h_v,128] (written in place when committing);
    hist, hist_out f32 [N,C,3]; qkv f32 [N,ntok,C]; alpha, beta f32 [N,ntok,h_v];
    z f32 [N,ntok,h_v,128]; conv_w f32 [C,4]; dt, ssm_a f32 [h_v]; gamma f32 [128].
    commit: 0 verify, 1 commit after the last token, 0x100|k commit after token k.  Returns y."""
    torch = _torch()
    N, D, h_v, _ = state.shape
    if D != 128:
        raise ValueError(f"gdn_window_fused: the head dim is 128, got state of shape {tuple(state.shape)}")
    ntok = qkv.shape[1]
    C = (2 * h_k + h_v) * D
    f32 = torch.float32
    _want(state, "state", f32, (N, D, h_v, D))
    _want(hist, "hist", f32, (N, C, 3))
    _want(hist_out, "hist_out", f32, (N, C, 3))
    _want(qkv, "qkv", f32, (N, ntok, C))
    _want(alpha, "alpha", f32, (N, ntok, h_v))
    _want(beta, "beta", f32, (N, ntok, h_v))
    _want(z, "z", f32, (N, ntok, h_v, D))
    _want(conv_w, "conv_w", f32, (C, 4))
    _want(dt, "dt", f32, (h_v,))
    _want(ssm_a, "ssm_a", f32, (h_v,))
    _want(gamma, "gamma", f32, (D,))
    if y is None:
        y = torch.empty((N, ntok, h_v, D), dtype=f32, device=state.device)
    _want(y, "y", f32, (N, ntok, h_v, D))
    _check(load().gdn_window_fused(_ptr(state), _ptr(hist), _ptr(hist_out), _ptr(qkv),
                                   _ptr(alpha), _ptr(beta), _ptr(z), _ptr(conv_w), _ptr(dt),
                                   _ptr(ssm_a), _ptr(gamma), _ptr(y), N, h_k, h_v, ntok,
                                   int(commit), float(eps), _stream(state.device)),
           "gdn_window_fused")
    return y
