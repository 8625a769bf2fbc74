"""Seeded synthetic inputs for the block-scaled FP8 linear layer.

This module only draws random numbers and stores them in the bit formats the
layer consumes (bf16 activations and weights, raw e4m3 codes, UE8M0 scale
bytes).  It contains none of the layer's arithmetic: no quantisation, no
decode, no contraction.  Both the CPU oracle (through the tests) and the GPU
library (through the tests and the benchmark) take their inputs from here.

Distributions follow the workloads on the pages:
  * activations x ~ N(0, 1) in bf16; the o_proj workload adds 1 % outlier
    channels scaled x20 (the reading: floor(K/100) columns picked by a seeded
    permutation, scaled before the bf16 rounding);
  * weights w ~ N(0, 0.02) in bf16, quantised later per 128x128 block;
  * the 32x32 UE8M0 format: codes uniform over the 254 finite e4m3 codes and
    one scale byte 127+e per 32x32 block, e uniform in [-14, 7]
    ("SM70 FP8 block-32 kernels" model card, "Exactness").

Every tensor is drawn from its own numpy PCG64 sub-stream
``default_rng([seed, stream])`` so that shapes can change without shifting
the values of other tensors.
"""
from __future__ import annotations

import numpy as np

# Sub-stream ids, one per kind of tensor.
STREAM_ACT = 1
STREAM_WEIGHT = 2
STREAM_OUTLIER = 3
STREAM_UE8M0_CODES = 4
STREAM_UE8M0_SCALES = 5
STREAM_SAMPLE = 6


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and return
    the 16-bit patterns.  This is storage conversion of the synthetic data, not
    part of the layer.  Inputs are finite."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    g = rng(seed, stream)
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


def outlier_columns(seed: int, K: int, frac: float = 0.01) -> np.ndarray:
    """Indices of the floor(frac*K) outlier channels (sorted)."""
    n = int(np.floor(K * frac))
    if n == 0:
        return np.zeros((0,), dtype=np.int64)
    perm = rng(seed, STREAM_OUTLIER).permutation(K)
    return np.sort(perm[:n])


def activations(seed: int, M: int, K: int, outliers: bool = False,
                outlier_gain: float = 20.0) -> np.ndarray:
    """bf16 bits [M, K], row-major: N(0,1), optionally with outlier channels."""
    g = rng(seed, STREAM_ACT)
    x = g.standard_normal(size=(M, K), dtype=np.float32)
    if outliers:
        cols = outlier_columns(seed, K)
        if cols.size:
            x[:, cols] *= np.float32(outlier_gain)
    return f32_to_bf16_bits(x)


def weights_bf16(seed: int, N: int, K: int, std: float = 0.02) -> np.ndarray:
    """bf16 bits [N, K], row-major: N(0, std)."""
    return normal_bf16(seed, STREAM_WEIGHT, (N, K), std)


def finite_e4m3_codes(seed: int, shape) -> np.ndarray:
    """Raw e4m3 bytes drawn uniformly from the 254 codes that are not NaN
    (0x7F and 0xFF are the two NaN codes of the finite-only e4m3 variant)."""
    r = rng(seed, STREAM_UE8M0_CODES).integers(0, 254, size=shape, dtype=np.int32)
    codes = np.where(r < 127, r, r + 1)
    return codes.astype(np.uint8)


def ue8m0_scale_bytes(seed: int, shape, emin: int = -14, emax: int = 7) -> np.ndarray:
    """One UE8M0 byte 127+e per block, e uniform in [emin, emax]."""
    e = rng(seed, STREAM_UE8M0_SCALES).integers(emin, emax + 1, size=shape, dtype=np.int32)
    return (e + 127).astype(np.uint8)


def ue8m0_weights(seed: int, N: int, K: int):
    """(codes [N, K] uint8, scale bytes [N/32, K/32] uint8)."""
    assert N % 32 == 0 and K % 32 == 0
    return finite_e4m3_codes(seed, (N, K)), ue8m0_scale_bytes(seed, (N // 32, K // 32))


def sample_rows(seed: int, M: int, count: int) -> np.ndarray:
    """A seeded sorted subset of row indices (all rows when count >= M)."""
    if count >= M:
        return np.arange(M, dtype=np.int64)
    return np.sort(rng(seed, STREAM_SAMPLE).choice(M, size=count, replace=False))
