"""Helpers of the GPU parity tests: moving seeded numpy inputs to the device and back."""
import numpy as np


def dev(x, dtype):
    """numpy -> CUDA tensor of `dtype`.  bf16 inputs from gdn_inputs are exactly representable, so
    the conversion is exact."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()


def host(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def library():
    """Build (if stale) and load libgdn.so."""
    import gated_deltanet_delta_gb300 as gdn
    from gated_deltanet_delta_gb300 import build
    build.build()
    return gdn.load()


def sample_heads(rng, n_b, n_h, count):
    """A reproducible sample of (b, h) pairs that always includes the first and the last head."""
    picks = {(0, 0), (n_b - 1, n_h - 1)}
    while len(picks) < min(count, n_b * n_h):
        picks.add((int(rng.integers(n_b)), int(rng.integers(n_h))))
    return sorted(picks)
