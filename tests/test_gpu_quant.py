"""GPU parity of the quantisers and the decode: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import groups_with_amax, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def gpu_quant_act(x_bits, lds_pad=0, ldx_pad=0):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, K = x_bits.shape
    xfull = np.zeros((M, K + ldx_pad), dtype=np.uint16)
    xfull[:, :K] = x_bits
    xt = to_dev_bf16(xfull)[:, :K]
    a = torch.full((M, K), 0xAB, dtype=torch.uint8, device="cuda")
    lds = fp8blk.act_scales_pitch(M) + lds_pad
    s = torch.full((K // 128, lds), -7.0, dtype=torch.float32, device="cuda")
    fp8blk.fp8blk_quant_act(xt, a, s)
    torch.cuda.synchronize()
    return a.cpu().numpy(), s.cpu().numpy(), lds


@pytest.mark.parametrize("M,K,outliers", [(16, 512, False), (1, 128, False), (3, 384, True), (17, 1024, True),
                                          (129, 4096, True), (300, 256, False),
                                          (257, 640, True),      # TMA-fed kernel, one row past a 64-row tile
                                          (4100, 384, True)])    # more tiles than CTAs, ragged last tile
def test_quant_act_matches_oracle(lib, M, K, outliers):
    x = synth.activations(M * 7 + K, M, K, outliers=outliers)
    a, s, lds = gpu_quant_act(x, lds_pad=4, ldx_pad=64)
    qa, qs = O.quant_act_1x128(x)
    assert np.array_equal(a, qa)
    assert np.array_equal(s[:, :M].view(np.uint32), qs.view(np.uint32))
    assert np.all(s[:, M:] == -7.0)            # padding of the scale pitch untouched


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x43E0, 0x40F0, 0x7F7F, 0x0080, 0x0003])
def test_quant_act_exhaustive_bf16_groups(lib, amax_bits):
    rng = np.random.default_rng(5)
    g = groups_with_amax(amax_bits, rng)                 # [n, 128]
    if g.shape[0] % 2:
        g = np.concatenate([g, g[-1:]], axis=0)
    x = g.reshape(g.shape[0] // 2, 256)                  # two groups per row
    a, s, _ = gpu_quant_act(x)
    qa, qs = O.quant_act_1x128(x)
    assert np.array_equal(a, qa)
    assert np.array_equal(s[:, : x.shape[0]].view(np.uint32), qs.view(np.uint32))


def test_quant_act_zero_and_signed_zero_groups(lib):
    x = np.zeros((4, 256), dtype=np.uint16)
    x[1, :128] = 0x8000
    x[2, 5] = 0x3F80
    x[3] = 0x8000
    a, s, _ = gpu_quant_act(x)
    qa, qs = O.quant_act_1x128(x)
    assert np.array_equal(a, qa)
    assert np.array_equal(s[:, :4], qs)


def test_quant_act_large_row_count_sampled(lib):
    M, K = 8192, 7168
    x = synth.activations(0, M, K)
    a, s, _ = gpu_quant_act(x)
    rows = synth.sample_rows(0, M, 64)
    qa, qs = O.quant_act_1x128(x[rows])
    assert np.array_equal(a[rows], qa)
    assert np.array_equal(s[:, rows], qs)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 512), (384, 1024)])
def test_quant_weight_matches_oracle(lib, N, K):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    w = synth.weights_bf16(N + K, N, K)
    b, bs = fp8blk.quant_weight(to_dev_bf16(w))
    torch.cuda.synchronize()
    qb, qbs = O.quant_weight_128x128(w)
    assert np.array_equal(b.cpu().numpy(), qb)
    assert np.array_equal(bs.cpu().numpy().view(np.uint32), qbs.view(np.uint32))


@pytest.mark.parametrize("e", [0, -14, -1, 3, 7])
def test_decode_all_codes_exact(lib, e):
    """The kernels' integer e4m3 -> bf16 decode gives dec(code) * 2^e exactly,
    for every finite code including subnormals and both zeros."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F] + [0, 0], dtype=np.uint8)   # 256 = 4k
    ct = to_dev(codes)
    out = torch.zeros(codes.size, dtype=torch.int16, device="cuda")
    fp8blk.fp8blk_debug_decode_e4m3(ct, e, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    ref = O.f64_to_bf16_bits(O.e4m3_decode(codes) * 2.0 ** e)
    assert np.array_equal(got, ref)


def test_validate_weights_counts(lib):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    b = synth.finite_e4m3_codes(1, (256, 512))
    b[3, 7] = 0x7F
    b[200, 511] = 0xFF
    bs = np.full((2, 4), 0.01, dtype=np.float32)
    bs[1, 2] = np.inf
    bs[0, 0] = 0.0
    assert fp8blk.validate_weights(to_dev(b), to_dev(bs), fp8blk.SCALE_F32_128x128) == (2, 2)
    e = np.full((8, 16), 127, dtype=np.uint8)
    e[0, 0] = 127 - 15
    e[7, 15] = 127 + 8
    e[3, 3] = 127 + 7
    b2 = synth.finite_e4m3_codes(2, (256, 512))
    assert fp8blk.validate_weights(to_dev(b2), to_dev(e), fp8blk.SCALE_UE8M0_32x32) == (0, 2)


def test_quant_act_many_scales_across_the_exponent_range(lib):
    """400 group maxima spread over the whole bf16 exponent range (tiny,
    denormal and huge scales included), 1023 random companions each."""
    rng = np.random.default_rng(21)
    allb = np.arange(65536, dtype=np.uint16)
    vals = O.bf16_bits_to_f64(allb)
    fin_pos = allb[np.isfinite(vals) & (vals > 0)]
    amaxes = np.concatenate([rng.choice(fin_pos, 392, replace=False),
                             np.array([0x0001, 0x0002, 0x0080, 0x0F80, 0x1000, 0x6F80, 0x7F7F, 0x43E0],
                                      dtype=np.uint16)])
    rows = []
    for ab in amaxes:
        a = O.bf16_bits_to_f64(np.array([ab], dtype=np.uint16))[0]
        pool = allb[np.isfinite(vals) & (np.abs(vals) <= a)]
        g = rng.choice(pool, 1024)
        g[rng.integers(0, 1024)] = ab | (rng.integers(0, 2) << 15)
        rows.append(g.reshape(8, 128))
    x = np.concatenate(rows, axis=0).reshape(-1, 256)        # two groups per row
    a, s, _ = gpu_quant_act(x)
    qa, qs = O.quant_act_1x128(x)
    assert np.array_equal(s[:, : x.shape[0]].view(np.uint32), qs.view(np.uint32))
    assert np.array_equal(a, qa)


def test_group_scale_arithmetic_every_bf16_amax(lib):
    """The quantisers' scale arithmetic on every finite non-negative bf16 group
    maximum: s equals the correctly rounded amax / 448 (1 for zero), the
    divisor is s times a power of two inside [2^-60, 2^64], and its reciprocal
    is the correctly rounded 1 / divisor (float64 quotient rounded to float32,
    which double rounding leaves exact)."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint16)
    amax = O.bf16_bits_to_f64(bits).astype(np.float32)
    n = amax.size
    dev = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    fp8blk.fp8blk_debug_group_scale(torch.from_numpy(amax).cuda(), *dev)
    torch.cuda.synchronize()
    s, ds, y = (t.cpu().numpy() for t in dev)
    s_ref = np.where(amax == 0, np.float32(1.0), O.fp32_div(amax, np.float32(448.0))).astype(np.float32)
    bad = np.nonzero(s.view(np.uint32) != s_ref.view(np.uint32))[0]
    assert bad.size == 0, f"scale differs for amax bits {bits[bad[:5]]}"
    ratio = ds.astype(np.float64) / s.astype(np.float64)
    assert np.all(np.log2(ratio) == np.round(np.log2(ratio)))
    assert np.all((ds >= 2.0 ** -60) & (ds <= 2.0 ** 64))
    y_ref = (1.0 / ds.astype(np.float64)).astype(np.float32)
    bad = np.nonzero(y.view(np.uint32) != y_ref.view(np.uint32))[0]
    assert bad.size == 0, f"reciprocal differs for amax bits {bits[bad[:5]]}"
