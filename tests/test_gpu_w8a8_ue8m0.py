"""GPU parity of W8A8 in the 32x32 UE8M0 format (power-of-two 1x32 activation
scales, tensor-core block scaling) against the float64 oracle: the exponent
bytes and codes bit for bit, the product within
|gpu - ref| <= 8e-3 |ref| + 2e-3 rms(ref row), elementwise."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, bf16_out_to_f64, groups_with_amax, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def gpu_quant(x_bits, ldx_pad=0):
    """Codes [M, K] and exponent bytes [K/32, M] (the oracle's orientation),
    read back from the tiled scale layout; the padding rows of the last
    128-row block must hold 127."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, K = x_bits.shape
    xf = np.zeros((M, K + ldx_pad), dtype=np.uint16)
    xf[:, :K] = x_bits
    x = to_dev_bf16(xf)[:, :K]
    a, sf = fp8blk.quant_act_ue8m0(x)
    torch.cuda.synchronize()
    assert sf.numel() == fp8blk.fp8blk_ue8m0_sf_bytes(M, K)
    rows = fp8blk.ue8m0_sf_to_rows(sf.cpu(), (M + 127) // 128 * 128, K).numpy()
    assert np.all(rows[M:] == 127)
    return a.cpu().numpy(), np.ascontiguousarray(rows[:M].T)


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x43E0, 0x43E1, 0x40F0, 0x7F7F, 0x0080, 0x0003, 0x3C01])
def test_quant_ue8m0_exhaustive_groups(lib, amax_bits):
    """Every finite bf16 value of magnitude <= amax, in 32-value groups that
    keep amax: codes and exponent bytes equal the oracle's."""
    g = groups_with_amax(amax_bits, np.random.default_rng(amax_bits))
    x = g.reshape(-1, 128)
    a, e = gpu_quant(x)
    a_ref, e_ref = O.quant_act_1x32_ue8m0(x)
    assert np.array_equal(e, e_ref)
    assert np.array_equal(a, a_ref)


def test_quant_ue8m0_every_bf16_group_maximum(lib):
    """One group per finite non-negative bf16 maximum (every exponent the
    rule can produce), padded with a ragged row pitch."""
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    n = len(bits)
    rows = (n + 3) // 4
    x = np.zeros((rows * 4, 32), dtype=np.uint16)
    x[:n, 0] = bits
    x[:n, 1] = bits & 0x7FFF | 0x8000 * (bits % 2 == 0)          # a negative copy of the maximum
    x = x.reshape(rows, 128)
    a, e = gpu_quant(x, ldx_pad=8)
    a_ref, e_ref = O.quant_act_1x32_ue8m0(x)
    assert np.array_equal(e, e_ref)
    assert np.array_equal(a, a_ref)


def ue8m0_w8a8_inputs(seed, M, N, K):
    x = synth.activations(seed, M, K, outliers=True)
    a, ea = O.quant_act_1x32_ue8m0(x)
    b, eb = synth.ue8m0_weights(seed, N, K)
    return x, a, ea, b, eb


def gpu_gemm(a, ea, b, eb, f32=False, ldc_pad=0):
    """The product on the device; ea [K/32, M] as the oracle holds it, tiled
    on the host with the NaN byte in the padding rows (they only feed rows
    past M, which are never stored); the weight exponents tiled on the
    device."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, K = a.shape
    N = b.shape[0]
    a_sf = fp8blk.ue8m0_sf_from_rows(torch.from_numpy(np.ascontiguousarray(ea.T)), pad=0xFF).cuda()
    b_sf = fp8blk.ue8m0_weight_sf(to_dev(eb))
    c = torch.full((M, N + ldc_pad), 7.0, dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
    fp8blk.fp8blk_gemm_w8a8_ue8m0(to_dev(a), a_sf, to_dev(b), b_sf, c[:, :N])
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    out = c.float().cpu().numpy().astype(np.float64)
    if ldc_pad:
        assert np.all(out[:, N:] == 7.0)
    return out[:, :N]


@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024), (7168, 2048), (2048, 7168), (256, 384)])
def test_weight_sf_is_the_block_exponents_per_column(lib, N, K):
    """fp8blk_ue8m0_weight_sf writes block (n/32, g)'s byte for every column
    n of the block, in the tiled layout, bit for bit."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    _, eb = synth.ue8m0_weights(N + K, N, K)
    sf = fp8blk.ue8m0_weight_sf(to_dev(eb)).cpu()
    torch.cuda.synchronize()
    assert sf.numel() == fp8blk.fp8blk_ue8m0_sf_bytes(N, K)
    per_column = np.repeat(eb, 32, axis=0)                          # [N, K/32]
    assert np.array_equal(fp8blk.ue8m0_sf_to_rows(sf, N, K).numpy(), per_column)
    assert torch.equal(sf, fp8blk.ue8m0_sf_from_rows(torch.from_numpy(per_column)))


@pytest.mark.parametrize("M,N,K", [
    (1, 128, 128),        # one row, one K block, a half-width column tile
    (16, 256, 512),       # the tiny workload's shape
    (129, 384, 1024),     # ragged second row tile, a half-width last column tile
    (200, 2048, 7168),    # the UE8M0 workload's shapes, ragged M
    (300, 7168, 2048),
    (64, 512, 384),       # three K blocks
    (520, 4992, 384),     # CTA-pair kernel: ragged M (a pair tile's second CTA wholly past M), a last column
                          # tile of 128 (its second B half and scale block past N)
    (1024, 4864, 1024),   # CTA-pair kernel, whole tiles
])
def test_gemm_ue8m0_matches_oracle(lib, M, N, K):
    _, a, ea, b, eb = ue8m0_w8a8_inputs(M + N + K, M, N, K)
    out = gpu_gemm(a, ea, b, eb, ldc_pad=8 if M < 200 else 0)
    assert_gemm_close(out, O.gemm_w8a8_ue8m0(a, ea, b, eb), f"w8a8 ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(130, 512, 1024), (520, 4992, 384)])
def test_gemm_ue8m0_f32_out_is_unrounded(lib, M, N, K):
    _, a, ea, b, eb = ue8m0_w8a8_inputs(5, M, N, K)
    ref = O.gemm_w8a8_ue8m0(a, ea, b, eb)
    c32 = gpu_gemm(a, ea, b, eb, f32=True, ldc_pad=4)
    c16 = gpu_gemm(a, ea, b, eb)
    assert_gemm_close(c32, ref, "w8a8 ue8m0 float32 out")
    assert np.array_equal(O.bf16_bits_to_f64(O.f64_to_bf16_bits(c32)), c16)


@pytest.mark.parametrize("M,N,rows", [
    (12, 512, None),                                        # single-CTA kernel: rows 0..11
    (512, 4864, [0, 37, 127, 128, 200, 255, 256, 300, 383, 384, 450, 511]),   # CTA-pair kernel: rows in both CTAs
])
def test_gemm_ue8m0_one_hot_rows_exact(lib, M, N, rows):
    """Row r of A holds one 1.0 at column k_r, with its own activation
    exponent there (all other rows zero); C row r is then exactly
    dec(B[:, k_r]) 2^(ea + eb - 254): this pins which scale byte (block,
    slice, row, column) the hardware applies to every product, on both
    kernels (on CTA pairs, rows of the even and of the odd CTA)."""
    K = 512
    ks = [0, 31, 32, 63, 64, 127, 128, 200, 300, 383, 384, 511]
    rows = rows if rows is not None else list(range(M))
    a = np.zeros((M, K), dtype=np.uint8)
    ea = np.full((K // 32, M), 127, dtype=np.uint8)
    for i, (r, k0) in enumerate(zip(rows, ks)):
        a[r, k0] = 0x38
        ea[k0 // 32, r] = 127 + (i % 7) - 3
    b, eb = synth.ue8m0_weights(9, N, K)
    out = gpu_gemm(a, ea, b, eb, f32=True)
    assert np.array_equal(out, O.gemm_w8a8_ue8m0(a, ea, b, eb))


def test_linear_ue8m0_full_size_sampled(lib):
    """Quantiser + product on the device at M = 4096, N = 7168, K = 2048,
    checked on 32 sampled rows against the oracle run on the same bf16 input."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, N, K = 4096, 7168, 2048
    x = synth.activations(4, M, K)
    b, eb = synth.ue8m0_weights(4, N, K)
    a, sf = fp8blk.quant_act_ue8m0(to_dev_bf16(x))
    c = fp8blk.gemm_w8a8_ue8m0(a, sf, to_dev(b), fp8blk.ue8m0_weight_sf(to_dev(eb)))
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    rows = synth.sample_rows(4, M, 32)
    a_ref, ea_ref = O.quant_act_1x32_ue8m0(x[rows])
    assert np.array_equal(a[rows].cpu().numpy(), a_ref)
    assert np.array_equal(fp8blk.ue8m0_sf_to_rows(sf.cpu(), M, K).numpy()[rows].T, ea_ref)
    ref = O.gemm_w8a8_ue8m0(a_ref, ea_ref, b, eb)
    assert_gemm_close(bf16_out_to_f64(c)[rows], ref, "w8a8 ue8m0 4096x7168x2048 sampled")
