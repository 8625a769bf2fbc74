"""float32 output (FP8BLK_FLAG_OUT_F32) of every GEMM kernel: within the GEMM
tolerance of the float64 oracle, and identical, after round-to-nearest-even
to bf16, to the bf16 output of the same call (the accumulation is shared;
only the final store differs)."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _both_outputs(call, M, N, ldc_pad):
    """Runs call(c) into a bf16 and a float32 output (each with ldc_pad
    columns of padding that must stay untouched)."""
    c16 = torch.full((M, N + ldc_pad), 7.0, dtype=torch.bfloat16, device="cuda")
    c32 = torch.full((M, N + ldc_pad), 7.0, dtype=torch.float32, device="cuda")
    call(c16[:, :N])
    call(c32[:, :N])
    torch.cuda.synchronize()
    import block_scaled_fp8_bf16_gb300 as fp8blk
    assert fp8blk.fp8blk_device_error() == 0
    if ldc_pad:
        assert torch.all(c16[:, N:] == 7.0) and torch.all(c32[:, N:] == 7.0)
    return c16[:, :N], c32[:, :N]


def _check_pair(c16, c32, ref, what):
    out32 = c32.double().cpu().numpy()
    assert_gemm_close(out32, ref, what + " (float32 out)")
    # bf16(float32 result) == bf16 result, bit for bit.
    assert np.array_equal(_bf16_bits(c32.to(torch.bfloat16)), _bf16_bits(c16)), what + ": bf16 rounding differs"
    # The float32 output carries no bf16 rounding: at least a few values lie off the bf16 grid.
    assert (c32 != c32.to(torch.bfloat16).float()).any(), what + ": float32 output looks rounded"


@pytest.mark.parametrize("M,N,K", [
    (16, 256, 512),        # single-CTA kernel, split-K cluster
    (129, 384, 1024),      # single-CTA kernel, ragged second row tile
    (1, 640, 4224),        # one-token GEMV
    (1000, 2432, 1024),    # CTA-pair kernel, half-width last column tile
    (2200, 4992, 512),     # CTA-pair kernel, last-round tiles split in 256 x 128 halves
    (256, 7168, 256),      # CTA-pair kernel, every tile as two 256 x 128 halves
    (256, 4992, 12288),    # CTA-pair kernel, K split over two pairs per tile
])
def test_w8a8_f32_out(lib, M, N, K):
    x = synth.activations(M + K, M, K)
    a, As = O.quant_act_1x128(x)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(N + K, N, K))
    lds = lib.act_scales_pitch(M)
    s = np.zeros((K // 128, lds), dtype=np.float32)
    s[:, :M] = As
    ad, sd, bd, bsd = to_dev(a), to_dev(s), to_dev(b), to_dev(Bs)
    c16, c32 = _both_outputs(lambda c: lib.fp8blk_gemm_w8a8(ad, sd, bd, bsd, c), M, N, 8)
    _check_pair(c16, c32, O.gemm_w8a8(a, As, b, Bs), f"w8a8 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,fmt", [
    (1, 256, 4096, 0),     # CUDA-core GEMV
    (1, 640, 4224, 1),     # CUDA-core GEMV, a one-pass second segment
    (1, 256, 512, 0),      # decode-size kernel, 16-token tile
    (24, 384, 1024, 1),    # decode-size kernel, 32-token tile
    (5, 4096, 4096, 0),    # decode-size kernel, K split over a cluster
    (100, 256, 512, 0),    # token-tiled kernel
    (200, 384, 512, 1),
    (612, 4864, 384, 1),   # token-tiled kernel, 256-token tiles
])
def test_w8a16_f32_out(lib, M, N, K, fmt):
    x = synth.activations(M * 3 + K, M, K, outliers=True)
    if fmt == 0:
        b, sc = O.quant_weight_128x128(synth.weights_bf16(N, N, K))
        ref = O.gemm_w8a16_f32scale(x, b, sc)
    else:
        b, sc = synth.ue8m0_weights(N + K, N, K)
        ref = O.gemm_w8a16_ue8m0(x, b, sc)
    xd, bd, scd = to_dev_bf16(x), to_dev(b), to_dev(sc)
    c16, c32 = _both_outputs(lambda c: lib.fp8blk_gemm_w8a16(xd, bd, scd, fmt, c), M, N, 8)
    _check_pair(c16, c32, ref, f"w8a16 fmt{fmt} {M}x{N}x{K}")


def test_f32_out_k0_and_alignment(lib):
    M, N = 3, 256
    a = torch.zeros((M, 0), dtype=torch.uint8, device="cuda")
    s = torch.zeros((0, 4), dtype=torch.float32, device="cuda")
    b = torch.zeros((N, 0), dtype=torch.uint8, device="cuda")
    bs = torch.zeros((2, 0), dtype=torch.float32, device="cuda")
    c = torch.full((M, N), 5.0, dtype=torch.float32, device="cuda")
    L = lib._L()
    st = L.fp8blk_gemm_w8a8(lib._ptr(a), 16, lib._ptr(s), 4, lib._ptr(b), 16, lib._ptr(bs), lib._ptr(c), N,
                            M, N, 0, lib.FLAG_OUT_F32, lib._stream(None))
    torch.cuda.synchronize()
    assert st == 0 and torch.all(c == 0.0)
    # ldc * 4 must be a multiple of 16 for float32 output (ldc = 258 is not).
    a1 = torch.zeros((M, 128), dtype=torch.uint8, device="cuda")
    s1 = torch.ones((1, 4), dtype=torch.float32, device="cuda")
    b1 = torch.zeros((N, 128), dtype=torch.uint8, device="cuda")
    bs1 = torch.ones((2, 1), dtype=torch.float32, device="cuda")
    c2 = torch.empty((M, 258), dtype=torch.float32, device="cuda")
    st = L.fp8blk_gemm_w8a8(lib._ptr(a1), 128, lib._ptr(s1), 4, lib._ptr(b1), 128, lib._ptr(bs1), lib._ptr(c2), 258,
                            M, N, 128, lib.FLAG_OUT_F32, lib._stream(None))
    assert st == 3   # FP8BLK_ERR_MISALIGNED
