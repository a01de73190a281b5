"""Seeded synthetic rank buffers for the allreduce tests and benchmark.

This module only draws inputs; it holds none of the allreduce's arithmetic and
is shared by the CPU oracle's tests, the GPU parity tests and ``bench.py``.

Recipe (one generator per call, ranks drawn in order 0..P-1, seed 0 unless
stated):
  uniform_int   int32 uniform on [-1000, 1000]            (NumPy PCG64)
  small_int     int32 uniform on [-3, 3] (products that stay interesting)
  normal        N(0, sigma^2) drawn in float64, stored as fp32; bf16 buffers
                are that fp32 value rounded to nearest even by torch's
                float32 -> bfloat16 conversion, then viewed as uint16
Device buffers (large sweeps) are drawn by ``torch.randn`` on the device from
a ``torch.Generator`` seeded the same way; they are not bit-identical to the
host draws and are checked against the oracle on sampled elements.
"""

import numpy as np


def _to_bf16_bits(x32):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def rank_inputs(P, n, dtype, dist="normal", sigma=1.0, seed=0):
    """P host buffers of n elements: int32 / float32 arrays, or uint16 bit
    patterns for bfloat16."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(P):
        if dist == "uniform_int":
            a = rng.integers(-1000, 1001, size=n, dtype=np.int64).astype(np.int32)
        elif dist == "small_int":
            a = rng.integers(-3, 4, size=n, dtype=np.int64).astype(np.int32)
        elif dist == "normal":
            x = (rng.standard_normal(n) * sigma).astype(np.float32)
            a = _to_bf16_bits(x) if dtype == "bfloat16" else x
        else:
            raise ValueError(dist)
        if dtype == "int32" and a.dtype != np.int32:
            raise ValueError("int32 buffers need an integer distribution")
        if dtype == "float32" and a.dtype != np.float32:
            a = a.astype(np.float32)
        out.append(a)
    return out


def device_inputs(P, n, dtype, sigma=1.0, seed=0, device="cuda"):
    """P device tensors of n elements drawn N(0, sigma^2) on the device."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    tdt = {"float32": torch.float32, "bfloat16": torch.bfloat16}[dtype]
    out = []
    for _ in range(P):
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        x.mul_(sigma)
        out.append(x.to(tdt))
    return out
