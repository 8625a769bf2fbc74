"""Device-side seeded generators with the same recipes as ``synth`` (for sizes
where drawing on the host and copying would dominate a benchmark run).

Like ``synth`` this holds no arithmetic of the layer: it draws N(0, std)
bf16 tensors, picks outlier channels, and draws raw e4m3 codes / UE8M0 scale
bytes.  Values differ from the numpy generators (different RNG), the
distributions do not.
"""
from __future__ import annotations

import torch


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 8) + int(stream))
    return g


def activations(seed: int, M: int, K: int, outliers: bool = False, device="cuda", gain: float = 20.0):
    g = _gen(device, seed, 1)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outliers:
        n = K // 100
        if n:
            gc = _gen("cpu", seed, 3)
            cols = torch.randperm(K, generator=gc)[:n].to(device)
            x[:, cols] *= gain
    return x.to(torch.bfloat16)


def weights_bf16(seed: int, N: int, K: int, std: float = 0.02, device="cuda"):
    g = _gen(device, seed, 2)
    return (torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def ue8m0_weights(seed: int, N: int, K: int, device="cuda"):
    """(codes [N, K] uint8 over the 254 finite e4m3 codes, bytes [N/32, K/32] = 127 + e, e in [-14, 7])."""
    g = _gen(device, seed, 4)
    r = torch.randint(0, 254, (N, K), generator=g, device=device, dtype=torch.int32)
    codes = torch.where(r < 127, r, r + 1).to(torch.uint8)
    g2 = _gen(device, seed, 5)
    e = torch.randint(-14, 8, (N // 32, K // 32), generator=g2, device=device, dtype=torch.int32)
    return codes, (e + 127).to(torch.uint8)
