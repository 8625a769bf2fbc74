"""GPU parity of the W8A8 and W8A16 products against the float64 oracle,
within |gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref row), elementwise."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, bf16_out_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def w8a8_inputs(seed, M, N, K, outliers=True):
    x = synth.activations(seed, M, K, outliers=outliers)
    a, As = O.quant_act_1x128(x)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(seed, N, K))
    return a, As, b, Bs


def gpu_w8a8(a, As, b, Bs, ldc_pad=0, lds_pad=0):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, K = a.shape
    N = b.shape[0]
    lds = fp8blk.act_scales_pitch(M) + lds_pad
    s = np.zeros((K // 128, lds), dtype=np.float32)
    s[:, :M] = As
    c = torch.full((M, N + ldc_pad), 7.0, dtype=torch.bfloat16, device="cuda")
    fp8blk.fp8blk_gemm_w8a8(to_dev(a), to_dev(s), to_dev(b), to_dev(Bs), c[:, :N])
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    out = bf16_out_to_f64(c)
    if ldc_pad:
        assert np.all(out[:, N:] == 7.0)
    return out[:, :N]


@pytest.mark.parametrize("M,N,K", [
    (16, 256, 512),        # tiny workload
    (1, 128, 128),         # single block, single row
    (3, 256, 256),
    (17, 384, 1024),
    (129, 256, 2048),      # ragged second row tile
    (255, 512, 512),
    (128, 4096, 4096),     # split-K cluster path
    (1, 4096, 4096),       # one-token GEMV
    (1, 384, 4224),        # one-token GEMV: a whole segment and a one-pass segment
    (1, 2048, 14336),      # one-token GEMV: three segments and a half
    (1, 8192, 4352),       # past the GEMV's weight-set limit: split-K kernel
    (300, 1024, 1024),     # persistent path
    (2200, 4992, 512),     # CTA-pair path, ragged M, a half-width last column tile; 180 tiles: last 28 split
    (1000, 2432, 1024),    # CTA-pair path, 40 tiles (no split last round)
    (513, 8192, 384),      # CTA-pair path, one row past a tile boundary; 96 tiles: last 20 split in halves
    (2304, 2304, 256),     # CTA-pair path, 81 tiles: the last 5 run as 10 half tiles
    (256, 7168, 512),      # CTA-pair path, 28 tiles all run as 56 half tiles (too many 128 x 128 tiles to split K)
    (200, 6144, 384),      # all halves, ragged second CTA of every pair
    (130, 4992, 256),      # all halves, the last tile's second half lies wholly past N
    (200, 4992, 12416),    # CTA-pair path with K split over two pairs per tile: ragged M, a half-width
                           # last column tile, 97 K blocks split 48 / 49
])
def test_w8a8_matches_oracle(lib, M, N, K):
    a, As, b, Bs = w8a8_inputs(M + N + K, M, N, K)
    out = gpu_w8a8(a, As, b, Bs, ldc_pad=8 if M < 200 else 0, lds_pad=4)
    assert_gemm_close(out, O.gemm_w8a8(a, As, b, Bs), f"w8a8 {M}x{N}x{K}")


def test_w8a8_two_weight_scales_per_256_columns(lib):
    """Neighbouring 128-column slices carry very different weight scales."""
    M, N, K = 64, 512, 512
    a, As, b, Bs = w8a8_inputs(9, M, N, K)
    Bs = Bs * np.array([[1.0], [1000.0], [1e-3], [7.0]], dtype=np.float32)
    assert_gemm_close(gpu_w8a8(a, As, b, Bs), O.gemm_w8a8(a, As, b, Bs), "w8a8 Bs slices")


def test_w8a8_pair_path_weight_scales_per_slice(lib):
    """The CTA-pair kernel (M = 1024, N = 2560: 40 tiles of 256 x 256, each
    spanning two weight-scale slices) with weight scales that differ by up
    to 10^6 between the two 128-column halves of a tile and between K
    blocks: each half must take the scale of its own slice for every K
    block."""
    M, N, K = 1024, 2560, 512
    a, As, b, Bs = w8a8_inputs(11, M, N, K)
    f = np.array([1.0, 1000.0, 1e-3, 7.0, 0.5], dtype=np.float32)
    Bs = Bs * f[(np.arange(N // 128)[:, None] + 2 * np.arange(K // 128)[None, :]) % len(f)]
    assert_gemm_close(gpu_w8a8(a, As, b, Bs), O.gemm_w8a8(a, As, b, Bs), "w8a8 pair Bs slices")


def test_w8a8_special_rows(lib):
    """A zero row, an outlier row and a row of +-448 codes."""
    M, N, K = 8, 256, 1024
    x = synth.activations(3, M, K)
    x[0] = 0
    x[1, 5] = 0x4700          # 32768
    x[2] = np.where(np.arange(K) % 2 == 0, 0x43E0, 0xC3E0)   # +-448
    a, As = O.quant_act_1x128(x)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(3, N, K))
    out = gpu_w8a8(a, As, b, Bs)
    ref = O.gemm_w8a8(a, As, b, Bs)
    assert np.all(out[0] == 0)
    assert_gemm_close(out, ref, "w8a8 special rows")


def test_w8a8_full_size_sampled_rows(lib):
    """o_proj shape at M = 4096 in the benchmark's launch configuration,
    checked on 64 sampled rows."""
    M, N, K = 4096, 4096, 4096
    a, As, b, Bs = w8a8_inputs(0, M, N, K)
    out = gpu_w8a8(a, As, b, Bs)
    rows = synth.sample_rows(0, M, 64)
    assert_gemm_close(out[rows], O.gemm_w8a8_rows(a, As, b, Bs, rows), "w8a8 4096^3 sampled")


def test_w8a8_prefill_size_sampled_rows(lib):
    """A prefill workload at full size (M = 2048, N = 18432, K = 7168: 576
    CTA-pair tiles, 7.6 rounds), checked on 16 sampled rows."""
    M, N, K = 2048, 18432, 7168
    a, As = O.quant_act_1x128(synth.activations(2, M, K))
    # Weight codes and block scales drawn directly (quantising 132 M weights
    # in float64 would dominate the test): uniform finite codes, scales 2^-12..2^-6.
    b = synth.finite_e4m3_codes(2, (N, K))
    Bs = np.exp2(np.random.default_rng(2).uniform(-12, -6, size=(N // 128, K // 128))).astype(np.float32)
    out = gpu_w8a8(a, As, b, Bs)
    rows = synth.sample_rows(2, M, 16)
    assert_gemm_close(out[rows], O.gemm_w8a8_rows(a, As, b, Bs, rows), "w8a8 2048x18432x7168 sampled")


def test_w8a8_one_hot_rows(lib):
    """Each A row holds a single 1.0 at column k0: C row = Bs * dec(B[:, k0])."""
    N, K = 256, 512
    ks = [0, 31, 32, 127, 128, 300, 511]
    a = np.zeros((len(ks), K), dtype=np.uint8)
    for i, k0 in enumerate(ks):
        a[i, k0] = 0x38
    As = np.ones((K // 128, len(ks)), dtype=np.float32)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(4, N, K))
    out = gpu_w8a8(a, As, b, Bs)
    ref = O.gemm_w8a8(a, As, b, Bs)
    assert np.array_equal(out, O.bf16_bits_to_f64(O.f64_to_bf16_bits(ref)))


def gpu_w8a16(x, b, sc, fmt, gemv=False, ldx_pad=0):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, K = x.shape
    N = b.shape[0]
    xf = np.zeros((M, K + ldx_pad), dtype=np.uint16)
    xf[:, :K] = x
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fn = fp8blk.fp8blk_gemv_w8a16 if gemv else fp8blk.fp8blk_gemm_w8a16
    fn(to_dev_bf16(xf)[:, :K], to_dev(b), to_dev(sc), fmt, c)
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    return bf16_out_to_f64(c)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (2, 256, 512), (4, 384, 1024), (8, 512, 384),
                                   (16, 256, 14336), (5, 28672, 256)])
def test_gemv_w8a16_f32(lib, M, N, K):
    x = synth.activations(M + K, M, K)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(M + N, N, K))
    out = gpu_w8a16(x, b, Bs, 0, gemv=True, ldx_pad=8)
    assert_gemm_close(out, O.gemm_w8a16_f32scale(x, b, Bs), f"gemv f32 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 2048, 7168), (4, 7168, 2048), (16, 256, 512), (3, 128, 128)])
def test_gemv_w8a16_ue8m0(lib, M, N, K):
    x = synth.activations(M, M, K)
    b, e = synth.ue8m0_weights(N, N, K)
    out = gpu_w8a16(x, b, e, 1, gemv=True)
    assert_gemm_close(out, O.gemm_w8a16_ue8m0(x, b, e), f"gemv ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(17, 256, 512), (32, 512, 1024), (33, 256, 256), (64, 384, 2048),
                                   (100, 256, 512), (128, 512, 512), (129, 256, 1024), (512, 1024, 512),
                                   (128, 512, 1152),      # K split over 4 CTAs with 9 K blocks: ranks of 2 and 3
                                   (64, 256, 896)])       # K split over 2 CTAs with 7 K blocks
@pytest.mark.parametrize("fmt", [0, 1])
def test_gemm_w8a16(lib, M, N, K, fmt):
    x = synth.activations(M * 3 + K, M, K, outliers=True)
    if fmt == 0:
        b, sc = O.quant_weight_128x128(synth.weights_bf16(N, N, K))
        ref = O.gemm_w8a16_f32scale(x, b, sc)
    else:
        b, sc = synth.ue8m0_weights(N + K, N, K)
        ref = O.gemm_w8a16_ue8m0(x, b, sc)
    out = gpu_w8a16(x, b, sc, fmt)
    assert_gemm_close(out, ref, f"w8a16 fmt{fmt} {M}x{N}x{K}")


# 256-token tiles (UE8M0 only; on 152 SMs taken when they need fewer rounds
# than 128-token tiles, a 256-token tile counted as 1.41): whole tiles, a
# ragged last tile whose last two 64-token epilogue slices lie wholly past M,
# an odd K block count (the two MMA issuers swap parity every tile), and more
# tiles than SMs (the one accumulator reused within a CTA).
@pytest.mark.parametrize("M,N,K", [(768, 6528, 256), (612, 4864, 384), (1100, 6528, 128)])
def test_gemm_w8a16_ue8m0_tile256(lib, M, N, K):
    x = synth.activations(M + N + K, M, K, outliers=True)
    b, sc = synth.ue8m0_weights(N + K, N, K)
    out = gpu_w8a16(x, b, sc, 1)
    assert_gemm_close(out, O.gemm_w8a16_ue8m0(x, b, sc), f"w8a16 ue8m0 tile256 {M}x{N}x{K}")


def test_w8a16_tile256_one_hot_rows_exact(lib):
    """Token r holds a single 1.0 at column r mod K: C row r is then exactly
    the decoded weight column times its block scale, so every token lands in
    its own output row through the 256-token tile's streamed epilogue."""
    M, N, K = 530, 19456, 256
    x = np.zeros((M, K), dtype=np.uint16)
    x[np.arange(M), np.arange(M) % K] = 0x3F80
    b, e = synth.ue8m0_weights(3, N, K)
    out = gpu_w8a16(x, b, e, 1)
    assert np.array_equal(out, O.gemm_w8a16_ue8m0(x, b, e))


def test_w8a16_ue8m0_full_size_sampled(lib):
    M, N, K = 4096, 7168, 2048
    x = synth.activations(1, M, K)
    b, e = synth.ue8m0_weights(1, N, K)
    out = gpu_w8a16(x, b, e, 1)
    rows = synth.sample_rows(1, M, 32)
    assert_gemm_close(out[rows], O.gemm_w8a16_ue8m0_rows(x, b, e, rows), "w8a16 ue8m0 4096 sampled")


def test_w8a16_one_hot_columns_exact_decode(lib):
    """x rows with a single 1.0 read one weight column through the bf16 MMA:
    every finite code must come back exactly times its block scale."""
    N, K = 256, 256
    b = np.zeros((N, K), dtype=np.uint8)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    b[:254, 0] = finite
    b[:254, 200] = finite[::-1]
    e = synth.ue8m0_scale_bytes(5, (N // 32, K // 32))
    x = np.zeros((2, K), dtype=np.uint16)
    x[0, 0] = 0x3F80
    x[1, 200] = 0x3F80
    out = gpu_w8a16(x, b, e, 1)
    ref = O.gemm_w8a16_ue8m0(x, b, e)
    assert np.array_equal(out, ref)          # exact: a single product, no rounding
