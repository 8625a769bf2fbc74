"""Shared test utilities: uploads, the GEMM tolerance, exhaustive bf16 groups."""
import numpy as np

import oracle as O

# Tolerance of the GEMM outputs, elementwise:
#   |gpu - ref| <= REL * |ref| + RMS_FRAC * rms(ref row)
REL = 8e-3
RMS_FRAC = 2e-3


def tol_violations(gpu, ref, rel=REL, rms_frac=RMS_FRAC):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    bound = rel * np.abs(ref) + rms_frac * rms
    return np.abs(gpu - ref) > bound, bound


def assert_gemm_close(gpu, ref, what=""):
    bad, bound = tol_violations(gpu, ref)
    if bad.any():
        idx = np.argwhere(bad)
        i, j = idx[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at ({i},{j}): "
            f"gpu={gpu[i, j]!r} ref={ref[i, j]!r} bound={bound[i, j]!r}")


def to_dev_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_dev(arr, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def bf16_out_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def groups_with_amax(amax_bits, rng):
    """All finite bf16 values with |v| <= amax, shuffled into groups of 127,
    each completed with +-amax at a random position (one group per row)."""
    allb = np.arange(65536, dtype=np.uint16)
    v = O.bf16_bits_to_f64(allb)
    a = O.bf16_bits_to_f64(np.array([amax_bits], dtype=np.uint16))[0]
    pool = allb[np.isfinite(v) & (np.abs(v) <= a)]
    pool = rng.permutation(pool)
    n = (len(pool) + 126) // 127
    pool = np.resize(pool, n * 127).reshape(n, 127)
    sign = rng.integers(0, 2, size=(n, 1)).astype(np.uint16) << 15
    col = (np.uint16(amax_bits) | sign).astype(np.uint16)
    g = np.concatenate([pool, col], axis=1)
    idx = rng.permuted(np.tile(np.arange(128), (n, 1)), axis=1)
    return np.take_along_axis(g, idx, axis=1)
