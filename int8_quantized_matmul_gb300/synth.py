"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no packing, no quantization, no matmul). Both the GPU path
and the CPU oracle receive the arrays it returns and each packs/quantizes them
with its own code.

Distributions follow the workloads of the I2_S / I8_S pages:
  * ternary codes {0,1,2} i.i.d. with P = (0.3, 0.4, 0.3);
  * F32 activations ~ N(0, 1), optionally with 1% outliers scaled by 20
    (prefill shape);
  * int8 weights ~ round(N(0, 40)) clamped to +-127 (I8_S encoder FC);
  * per-tensor weight scales ~ U(0.01, 0.1) for the decoder projection set.
"""

from __future__ import annotations

import numpy as np

CODE_P = (0.3, 0.4, 0.3)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def codes(N: int, K: int, seed: int, p=CODE_P) -> np.ndarray:
    """N x K ternary codes in {0,1,2} (uint8), i.i.d. with probabilities p."""
    u = rng(seed).random((N, K), dtype=np.float32)
    c = np.zeros((N, K), dtype=np.uint8)
    c[u >= p[0]] = 1
    c[u >= p[0] + p[1]] = 2
    return c


def packed_code_bytes(nbytes: int, seed: int) -> np.ndarray:
    """Raw bytes whose four 2-bit fields are i.i.d. codes with P = (0.3, 0.4, 0.3).

    Because the codes are i.i.d., the byte distribution does not depend on which
    field holds which position, so large weight payloads are drawn directly as
    bytes: each field is a uniform draw r in [0, 10) mapped to (r >= 3) + (r >= 7).
    """
    g = rng(seed)
    out = np.empty(int(nbytes), dtype=np.uint8)
    chunk = 1 << 24
    for lo in range(0, int(nbytes), chunk):
        hi = min(int(nbytes), lo + chunk)
        r = g.integers(0, 10, size=(hi - lo, 4), dtype=np.uint8)
        c = (r >= 3).astype(np.uint8) + (r >= 7).astype(np.uint8)
        out[lo:hi] = (c[:, 0] << 6) | (c[:, 1] << 4) | (c[:, 2] << 2) | c[:, 3]
    return out


def packed_code_bytes_device(nbytes: int, seed: int, device):
    """The same law as packed_code_bytes, drawn on a CUDA device with torch's
    generator (used for the benchmark's 327 MB weight set; the draws differ from
    the numpy ones, the distribution does not)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    r = torch.randint(0, 10, (int(nbytes), 4), dtype=torch.uint8, device=device, generator=g)
    c = (r >= 3).to(torch.uint8) + (r >= 7).to(torch.uint8)
    return (c[:, 0] << 6) | (c[:, 1] << 4) | (c[:, 2] << 2) | c[:, 3]


def normal_f32_device(n: int, seed: int, device, std: float = 1.0, outlier_p: float = 0.0,
                      outlier_scale: float = 20.0):
    """N(0, std) F32 drawn on a CUDA device (same law as normal_f32)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(int(n), generator=g, device=device, dtype=torch.float32) * std
    if outlier_p > 0:
        mask = torch.rand(int(n), generator=g, device=device) < outlier_p
        x = torch.where(mask, x * outlier_scale, x)
    return x


def int8_normal_device(n: int, seed: int, device, std: float = 40.0):
    """int8 drawn as round(N(0, std)) clamped to +-127, on a CUDA device."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(int(n), generator=g, device=device, dtype=torch.float32) * std
    return torch.clamp(torch.round(x), -127, 127).to(torch.int8)


def normal_f32(shape, seed: int, std: float = 1.0, outlier_p: float = 0.0,
               outlier_scale: float = 20.0) -> np.ndarray:
    g = rng(seed)
    x = g.standard_normal(shape, dtype=np.float32) * np.float32(std)
    if outlier_p > 0:
        mask = g.random(shape, dtype=np.float32) < outlier_p
        x[mask] *= np.float32(outlier_scale)
    return x


def uniform_f32(shape, seed: int, lo: float, hi: float) -> np.ndarray:
    return rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def int8_normal(shape, seed: int, std: float = 40.0) -> np.ndarray:
    """int8 weights drawn as round(N(0, std)) clamped to +-127."""
    x = rng(seed).standard_normal(shape) * std
    return np.clip(np.rint(x), -127, 127).astype(np.int8)


# Qwen2-1.5B decoder projection shapes (out N, in K): hidden 1536, intermediate
# 8960, 12 heads of 128 over 2 KV heads (so k/v project to 256).
QWEN2_1P5B_LAYER = (
    ("q", 1536, 1536),
    ("k", 256, 1536),
    ("v", 256, 1536),
    ("o", 1536, 1536),
    ("gate", 8960, 1536),
    ("up", 8960, 1536),
    ("down", 1536, 8960),
)
QWEN2_1P5B_LAYERS = 28
QWEN2_1P5B_LM_HEAD = ("lm_head", 151936, 1536)
