"""Comparators used by the parity tests.

max_rel_err is the tolerance metric: max |x - ref| / max |ref| over a whole tensor (an elementwise
relative error is ill-posed where the reference crosses zero).  max_rel_err_slices applies the same
metric to every slice along the leading axes (per head, per sequence and head) and returns the
worst, so that a head whose outputs are small beside the tensor's largest cannot hide its error.
rel_frobenius is the metric of the KBench Comba spec (correctness_md): |x - ref|_F / |ref|_F.
"""
import numpy as np


def max_rel_err(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    den = float(np.max(np.abs(ref)))
    num = float(np.max(np.abs(x - ref)))
    if den == 0.0:
        return num
    return num / den


def max_rel_err_slices(x, ref, lead: int) -> float:
    """The worst max_rel_err over the slices x[i0, .., i_{lead-1}] (the first `lead` axes index the
    slices, the rest is compared as one tensor)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    n = int(np.prod(x.shape[:lead])) if lead else 1
    xs, rs = x.reshape(n, -1), ref.reshape(n, -1)
    return max((max_rel_err(xs[i], rs[i]) for i in range(n)), default=0.0)


def rel_frobenius(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.linalg.norm(ref.ravel()))
    num = float(np.linalg.norm((x - ref).ravel()))
    return num / den if den else num


def bf16_neighbours_ok(x_bf16_as_f32, ref) -> bool:
    """True when every bf16 value equals the round-to-nearest-even bf16 of the fp64 reference, or
    one of its two bf16 neighbours (a pre-rounding difference of ~1e-7 may flip a rounding)."""
    x = np.asarray(x_bf16_as_f32, dtype=np.float32)
    r = np.asarray(ref, dtype=np.float64).astype(np.float32)
    u = r.view(np.uint32).astype(np.uint64)
    rn = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.int64)   # RNE bf16 bits of ref
    rn = np.where(rn >= 0x8000, -(rn - 0x8000), rn)                  # signed-magnitude -> ordered
    xb = (x.view(np.uint32) >> 16).astype(np.int64)
    xb = np.where(xb >= 0x8000, -(xb - 0x8000), xb)
    return bool(np.all(np.abs(xb - rn) <= 1))
