"""Plain CPU oracle of the gated delta-rule recurrence (test infrastructure only).

The arithmetic lives in ``gdn_oracle.c`` (IEEE double, no fused multiply-add, one head and one
token at a time).  This module only marshals numpy arrays to it through ctypes.  It is imported by the
tests, by the smoke check and by the CPU-baseline leg of the benchmark; the CUDA library and its
Python binding never import it, and it imports nothing from them.

Every function takes arrays of any real dtype (bf16 values must already be widened to float32 or
float64, which is exact) and returns float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_HDR = os.path.join(_HERE, "gdn_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

STATUS_BAD_CACHE_INDEX = 1
STATUS_BAD_SEQLENS = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into _build/liboracle.so with gcc (strict IEEE: no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            D = ctypes.POINTER(ctypes.c_double)
            I64 = ctypes.POINTER(ctypes.c_int64)
            I32 = ctypes.POINTER(ctypes.c_int32)
            i, l, d, u = ctypes.c_int, ctypes.c_long, ctypes.c_double, ctypes.c_uint
            lib.oracle_gdn_decode_head.argtypes = [i, i, D, D, D, D, d, d, d, D, D]
            lib.oracle_gdn_decode_head.restype = None
            lib.oracle_gdn_decode.argtypes = [i, i, i, i, i, D, D, D, D, D, D, d, D, D]
            lib.oracle_gdn_decode.restype = i
            lib.oracle_comba_decode_head.argtypes = [i, i, D, D, D, D, D, d, d, d, D, D]
            lib.oracle_comba_decode_head.restype = None
            lib.oracle_comba_decode.argtypes = [i, i, i, i, D, D, D, D, D, D, D, d, D, D]
            lib.oracle_comba_decode.restype = i
            lib.oracle_comba_forward.argtypes = [i, i, i, i, i, D, D, D, D, D, D, D, d, D, D]
            lib.oracle_comba_forward.restype = i
            lib.oracle_gdn_prefill_unit.argtypes = [l, i, i, i, i, i, D, D, D, D, D, d, d, d, d, D, D]
            lib.oracle_gdn_prefill_unit.restype = None
            lib.oracle_gdn_prefill.argtypes = [i, I64, I64, i, l, i, i, i, i, D, D, D, D, D, D, D,
                                               d, d, D, D, I32]
            lib.oracle_gdn_prefill.restype = i
            lib.oracle_gdn_window_seq.argtypes = [i, i, i, i, u, d, D, D, D, D, D, D, D, D, D, D,
                                                  D, D]
            lib.oracle_gdn_window_seq.restype = i
            lib.oracle_gdn_window.argtypes = [i, i, i, i, i, u, d, D, D, D, D, D, D, D, D, D, D,
                                              D, D]
            lib.oracle_gdn_window.restype = i
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments of {what} (code {rc})")


# ------------------------------------------------------------------------------------------------
# GDN decode step: state [B,Hv,Dv,Dk], q,k [B,Hk,Dk], v [B,Hv,Dv], g (linear gate), beta [B,Hv]
# ------------------------------------------------------------------------------------------------
def gdn_decode(state, q, k, v, g, beta, scale: float):
    state, q, k, v, g, beta = map(_f64, (state, q, k, v, g, beta))
    B, Hv, Dv, Dk = state.shape
    Hk = q.shape[1]
    state_new = np.empty_like(state)
    y = np.empty((B, Hv, Dv))
    _check(_load().oracle_gdn_decode(B, Hk, Hv, Dk, Dv, _p(state), _p(q), _p(k), _p(v), _p(g),
                                     _p(beta), float(scale), _p(state_new), _p(y)), "gdn_decode")
    return state_new, y


# ------------------------------------------------------------------------------------------------
# Comba decode step: state [B,H,K,V], q,k,p [B,H,K], v [B,H,V], beta, g_log [B,H]
# ------------------------------------------------------------------------------------------------
def comba_decode(state, q, k, v, p, beta, g_log, scale: float):
    state, q, k, v, p, beta, g_log = map(_f64, (state, q, k, v, p, beta, g_log))
    B, H, K, V = state.shape
    state_new = np.empty_like(state)
    o = np.empty((B, H, V))
    _check(_load().oracle_comba_decode(B, H, K, V, _p(state), _p(q), _p(k), _p(v), _p(p),
                                       _p(beta), _p(g_log), float(scale), _p(state_new), _p(o)),
           "comba_decode")
    return state_new, o


def comba_forward(state, q, k, v, p, beta, g_log, scale: float):
    """T Comba steps per head: state [B,H,K,V]; q,k,p [B,T,H,K]; v [B,T,H,V]; beta,g_log [B,T,H].
    Returns (final state [B,H,K,V], o [B,T,H,V])."""
    state, q, k, v, p, beta, g_log = map(_f64, (state, q, k, v, p, beta, g_log))
    B, H, K, V = state.shape
    T = q.shape[1]
    state_out = np.empty_like(state)
    o = np.empty((B, T, H, V))
    _check(_load().oracle_comba_forward(B, T, H, K, V, _p(state), _p(q), _p(k), _p(v), _p(p),
                                        _p(beta), _p(g_log), float(scale), _p(state_out), _p(o)),
           "comba_forward")
    return state_out, o


# ------------------------------------------------------------------------------------------------
# Prefill (sequential recurrence): q,k [T,Hk,K], v [T,Hv,V], a,b [T,Hv], A_log,dt_bias [Hv],
# state_pool [pool,Hv,V,K] (a float64 copy is updated and returned), out [T,Hv,V]
# ------------------------------------------------------------------------------------------------
def gdn_prefill(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens,
                scale: float, eps: float = 1e-6, out=None):
    q, k, v, a, b, A_log, dt_bias = map(_f64, (q, k, v, a, b, A_log, dt_bias))
    pool = _f64(state_pool).copy()
    ci = np.ascontiguousarray(np.asarray(cache_indices, dtype=np.int64))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    T, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    out = np.zeros((T, Hv, V)) if out is None else _f64(out).copy()
    status = ctypes.c_int32(0)
    I64 = ctypes.POINTER(ctypes.c_int64)
    _check(_load().oracle_gdn_prefill(len(ci), cu.ctypes.data_as(I64), ci.ctypes.data_as(I64),
                                      pool.shape[0], T, Hk, Hv, K, V, _p(q), _p(k), _p(v), _p(a),
                                      _p(b), _p(A_log), _p(dt_bias), float(eps), float(scale),
                                      _p(pool), _p(out), ctypes.byref(status)), "gdn_prefill")
    return pool, out, int(status.value)


def gdn_prefill_unit(q, k, v, a, b, A_log_h: float, dt_bias_h: float, S0, h: int, scale: float,
                     eps: float = 1e-6):
    """One (sequence, value head): q,k [T_n,Hk,K], v [T_n,Hv,V], a,b [T_n,Hv], S0 [V,K].
    Returns (S_final [V,K], out [T_n,V])."""
    q, k, v, a, b = map(_f64, (q, k, v, a, b))
    T_n, Hk, K = q.shape
    Hv, V = v.shape[1], v.shape[2]
    S = _f64(S0).copy()
    out = np.zeros((T_n, Hv, V))
    _load().oracle_gdn_prefill_unit(T_n, Hk, Hv, K, V, h, _p(q), _p(k), _p(v), _p(a), _p(b),
                                    float(A_log_h), float(dt_bias_h), float(eps), float(scale),
                                    _p(S), _p(out))
    return S, out[:, h, :]


# ------------------------------------------------------------------------------------------------
# Fused decode window, N sequences: state [N,D,h_v,D], hist [N,C,3], qkv [N,ntok,C],
# alpha,beta [N,ntok,h_v], z [N,ntok,h_v,D], conv_w [C,4], dt,ssm_a [h_v], gamma [D]
# ------------------------------------------------------------------------------------------------
def gdn_window(state, hist, qkv, alpha, beta, z, conv_w, dt, ssm_a, gamma, h_k: int,
               commit: int, eps: float = 1e-6, hist_out=None):
    """Returns (state_after [N,D,h_v,D], hist_out [N,C,3], y [N,ntok,h_v,D]).  The input state and
    hist_out are copied; in verify mode the returned state equals the input and hist_out is the
    given hist_out (zeros if None)."""
    state = _f64(state).copy()
    hist, qkv, alpha, beta, z, conv_w, dt, ssm_a, gamma = map(
        _f64, (hist, qkv, alpha, beta, z, conv_w, dt, ssm_a, gamma))
    N, D, h_v, _ = state.shape
    ntok = qkv.shape[1]
    hist_out = np.zeros_like(hist) if hist_out is None else _f64(hist_out).copy()
    y = np.empty((N, ntok, h_v, D))
    _check(_load().oracle_gdn_window(N, D, h_k, h_v, ntok, int(commit), float(eps), _p(state),
                                     _p(hist), _p(hist_out), _p(qkv), _p(alpha), _p(beta), _p(z),
                                     _p(conv_w), _p(dt), _p(ssm_a), _p(gamma), _p(y)),
           "gdn_window")
    return state, hist_out, y
