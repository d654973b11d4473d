"""Seeded synthetic inputs for the gated delta-rule workloads.

This module is shared by the tests, the benchmark and the smoke check, and is the only code that
both the CUDA path and the CPU oracle are fed from.  It holds none of the method's arithmetic: it
draws random numbers (numpy PCG64, seeded) in the shapes, dtypes and distributions of the workloads,
and rounds values to bfloat16 (round-to-nearest-even) where a workload says bf16.  bf16 values are
returned as float32 arrays whose values are exactly representable in bf16, so that widening them to
float32 or float64 on either side is exact.

Distributions follow the workload descriptions:
  - decode (GDN): q ~ randn; k = L2-normalised randn; v ~ randn; beta = sigmoid(U(0,1)), all bf16;
    gate g = exp(logsigmoid(randn) / 4) fp32 (a linear gate, as the decode step takes it);
  - Comba: the same with a read key p = L2-normalised randn (bf16) and the log-decay
    g = logsigmoid(randn) / 4 fp32 (KBench specs/comba_decode_step.py, make_inputs_src);
  - prefill: q, k, v, a, b ~ randn bf16; A_log = log(U(1,16)); dt_bias = U(-1,1); state pool
    randn * 0.05; distinct random cache slots;
  - window: conv_w ~ 0.5 randn; alpha ~ randn; dt ~ U(-1,1); ssm_a = -U(0.5,8); beta ~ randn;
    gamma ~ 1 + 0.1 randn; z ~ randn; qkv, hist ~ randn; state randn * 0.05 (all fp32).
"""
from __future__ import annotations

import numpy as np

# ------------------------------------------------------------------------------------------------
# Named workloads (sizes only)
# ------------------------------------------------------------------------------------------------
GDN_DECODE_TINY = dict(name="gdn decode B1 Hk2 Hv4 D64", B=1, Hk=2, Hv=4, Dk=64, Dv=64, warmup=16)
GDN_DECODE_BATCHED = dict(name="gdn decode B64 Hk16 Hv32 D128", B=64, Hk=16, Hv=32, Dk=128, Dv=128,
                          warmup=16, steps=100)
COMBA_DECODE = dict(name="comba decode B256 H32 K128 V128", B=256, H=32, K=128, V=128, warmup=16)
# the Comba forward over T tokens per call on the decode workload's heads
COMBA_FORWARD = dict(name="comba forward B256 T8 H32 K128 V128", B=256, T=8, H=32, K=128, V=128)
GDN_PREFILL = dict(name="gdn chunked prefill T15360 (4096+2048+1024+8192) Hk16 Hv32 K128 V128 C64",
                   seqlens=(4096, 2048, 1024, 8192), Hk=16, Hv=32, K=128, V=128, pool=16, chunk=64)
GDN_WINDOW = dict(name="gdn fused window N32 h_k16 h_v48 D128 ntok8", N=32, h_k=16, h_v=48, D=128,
                  ntok=8)


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returned as float32."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(a.shape)


def f16_round(x) -> np.ndarray:
    """Round float32 values to the nearest IEEE binary16 (ties to even); returned as float32."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def _randn(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(shape, dtype=np.float32)


def _unit(g: np.random.Generator, shape) -> np.ndarray:
    x = _randn(g, shape)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return x / np.maximum(n, np.float32(1e-12))


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    return (-np.logaddexp(np.float32(0), -x)).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


# ------------------------------------------------------------------------------------------------
# Decode tokens
# ------------------------------------------------------------------------------------------------
def gdn_decode_token(g: np.random.Generator, B: int, Hk: int, Hv: int, Dk: int, Dv: int) -> dict:
    """One token of GDN decode inputs: q,k [B,Hk,Dk] bf16; v [B,Hv,Dv] bf16; beta [B,Hv] bf16;
    g [B,Hv] fp32 linear gate."""
    q = bf16_round(_randn(g, (B, Hk, Dk)))
    k = bf16_round(_unit(g, (B, Hk, Dk)))
    v = bf16_round(_randn(g, (B, Hv, Dv)))
    beta = bf16_round(_sigmoid(g.random((B, Hv), dtype=np.float32)))
    gate = np.exp(_logsigmoid(_randn(g, (B, Hv))) / np.float32(4.0)).astype(np.float32)
    return dict(q=q, k=k, v=v, g=gate, beta=beta)


def comba_decode_token(g: np.random.Generator, B: int, H: int, K: int, V: int) -> dict:
    """One token of Comba inputs: q,k,p [B,H,K] bf16; v [B,H,V] bf16; beta [B,H] bf16;
    g_log [B,H] fp32 log-decay (<= 0)."""
    q = bf16_round(_randn(g, (B, H, K)))
    k = bf16_round(_unit(g, (B, H, K)))
    v = bf16_round(_randn(g, (B, H, V)))
    p = bf16_round(_unit(g, (B, H, K)))
    beta = bf16_round(_sigmoid(g.random((B, H), dtype=np.float32)))
    g_log = (_logsigmoid(_randn(g, (B, H))) / np.float32(4.0)).astype(np.float32)
    return dict(q=q, k=k, v=v, p=p, beta=beta, g_log=g_log)


def comba_forward_inputs(g: np.random.Generator, B: int, T: int, H: int, K: int, V: int) -> dict:
    """T tokens of Comba inputs per sequence (each token drawn as comba_decode_token draws one) and
    an initial state: q,k,p [B,T,H,K] bf16; v [B,T,H,V] bf16; beta, g_log [B,T,H];
    state [B,H,K,V] fp32 = 0.05 randn."""
    toks = [comba_decode_token(g, B, H, K, V) for _ in range(T)]
    x = {n: np.ascontiguousarray(np.stack([t[n] for t in toks], axis=1)) for n in toks[0]} if T else \
        dict(q=np.zeros((B, 0, H, K), np.float32), k=np.zeros((B, 0, H, K), np.float32),
             v=np.zeros((B, 0, H, V), np.float32), p=np.zeros((B, 0, H, K), np.float32),
             beta=np.zeros((B, 0, H), np.float32), g_log=np.zeros((B, 0, H), np.float32))
    x["state"] = (_randn(g, (B, H, K, V)) * np.float32(0.05)).astype(np.float32)
    return x


# ------------------------------------------------------------------------------------------------
# Prefill
# ------------------------------------------------------------------------------------------------
def comba_prefill_inputs(g: np.random.Generator, seqlens, H: int, K: int, V: int, pool: int,
                         mild: bool = False) -> dict:
    """Varlen Comba prefill inputs, every token drawn as comba_decode_token draws one: q, k, p
    [T,H,K] bf16; v [T,H,V] bf16; beta bf16, g_log fp32 [T,H]; state_pool [pool,H,K,V] fp32 =
    0.05 randn; distinct cache_indices.  mild divides the log decays by 25, so that the state
    carried from chunk to chunk is not wiped out."""
    seqlens = [int(s) for s in seqlens]
    T = int(sum(seqlens))
    cu = np.zeros(len(seqlens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seqlens)
    x = comba_decode_token(g, T, H, K, V)
    if mild:
        x["g_log"] = (x["g_log"] / np.float32(25.0)).astype(np.float32)
    x["state_pool"] = (_randn(g, (pool, H, K, V)) * np.float32(0.05)).astype(np.float32)
    x["cache_indices"] = g.choice(pool, size=len(seqlens), replace=False).astype(np.int64)
    x["cu_seqlens"] = cu
    x["T"] = T
    return x


def gdn_prefill_inputs(g: np.random.Generator, seqlens, Hk: int, Hv: int, K: int, V: int,
                       pool: int, mild_gates: bool = False, dtype: str = "bf16") -> dict:
    """Varlen prefill inputs.  mild_gates draws A_log = log(U(0.01, 0.1)) instead of
    log(U(1, 16)), so that the state carried between chunks is not wiped out by the decay.
    dtype ("bf16" or "f16") is the type q, k, v, a and b are rounded to (the same draws)."""
    rnd = {"bf16": bf16_round, "f16": f16_round}[dtype]
    seqlens = [int(s) for s in seqlens]
    T = int(sum(seqlens))
    cu = np.zeros(len(seqlens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seqlens)
    q = rnd(_randn(g, (T, Hk, K)))
    k = rnd(_randn(g, (T, Hk, K)))
    v = rnd(_randn(g, (T, Hv, V)))
    a = rnd(_randn(g, (T, Hv)))
    b = rnd(_randn(g, (T, Hv)))
    lo, hi = (0.01, 0.1) if mild_gates else (1.0, 16.0)
    A_log = np.log(g.uniform(lo, hi, Hv)).astype(np.float32)
    dt_bias = g.uniform(-1.0, 1.0, Hv).astype(np.float32)
    state_pool = (_randn(g, (pool, Hv, V, K)) * np.float32(0.05)).astype(np.float32)
    cache_indices = g.choice(pool, size=len(seqlens), replace=False).astype(np.int64)
    return dict(q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state_pool=state_pool,
                cache_indices=cache_indices, cu_seqlens=cu, T=T)


# ------------------------------------------------------------------------------------------------
# Fused decode window
# ------------------------------------------------------------------------------------------------
def gdn_window_inputs(g: np.random.Generator, N: int, h_k: int, h_v: int, D: int,
                      ntok: int) -> dict:
    C = (2 * h_k + h_v) * D
    state = (_randn(g, (N, D, h_v, D)) * np.float32(0.05)).astype(np.float32)
    hist = _randn(g, (N, C, 3))
    qkv = _randn(g, (N, ntok, C))
    alpha = _randn(g, (N, ntok, h_v))
    beta = _randn(g, (N, ntok, h_v))
    z = _randn(g, (N, ntok, h_v, D))
    conv_w = (_randn(g, (C, 4)) * np.float32(0.5)).astype(np.float32)
    dt = g.uniform(-1.0, 1.0, h_v).astype(np.float32)
    ssm_a = (-g.uniform(0.5, 8.0, h_v)).astype(np.float32)
    gamma = (1.0 + 0.1 * _randn(g, (D,))).astype(np.float32)
    return dict(state=state, hist=hist, qkv=qkv, alpha=alpha, beta=beta, z=z, conv_w=conv_w,
                dt=dt, ssm_a=ssm_a, gamma=gamma)
