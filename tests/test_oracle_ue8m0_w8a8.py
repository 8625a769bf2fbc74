"""Pins of the oracle's W8A8 path in the 32x32 UE8M0 format: the 1x32
activation exponent rule, the power-of-two activation quantiser and the
product.  Independent routes: exact Fraction comparisons for the exponent
rule, torch's nearest-even float8_e4m3fn cast for the codes, torch's decoder
and Fraction sums for the product, and the (separately pinned) fp32-scale
product where both formats describe the same numbers."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import groups_with_amax


def _smallest_exponent_ok(v, e):
    """448 * 2^e >= v, and e is the smallest such integer unless clamped (exact)."""
    fv = Fraction(v)
    reach = Fraction(448) * Fraction(2) ** e >= fv
    smaller = Fraction(448) * Fraction(2) ** (e - 1) >= fv
    if e == O.ACT_EXP_MIN:
        return reach          # clamp: anything below is not representable as a UE8M0 byte
    return reach and not smaller


def test_act_exponent_special_values():
    # 448 * 2^0 = 448 reaches 448, 448 * 2^-1 = 224 does not; 450 needs 896;
    # 224 is reached by 448 * 2^-1; 1.0 by 448 * 2^-8 = 1.75 (0.875 is short);
    # the largest finite bf16, (2 - 2^-7) 2^127, by 448 * 2^120 = 1.75 * 2^128.
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    vals = [448.0, 450.0, 224.0, 1.0, bf16_max, 0.0, 2.0 ** -133, 2.0 ** -126]
    assert list(O.act_exponent_ue8m0(vals)) == [0, 1, -1, -8, 120, -127, -127, -127]


def test_act_exponent_minimal_on_every_finite_bf16():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint16)        # positive finite bf16
    v = O.bf16_bits_to_f64(bits)
    e = O.act_exponent_ue8m0(v)
    bad = [(float(x), int(k)) for x, k in zip(v, e) if not _smallest_exponent_ok(float(x), int(k))]
    assert not bad, bad[:5]


def _torch_codes(x_bits_rows, e):
    """q = float8_e4m3fn cast of x * 2^-e (rows of 32), through torch."""
    x = torch.from_numpy(x_bits_rows.astype(np.int32).astype(np.int16)).view(torch.bfloat16).double()
    y = x * torch.from_numpy(np.exp2(-e.astype(np.float64)))[:, None]
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x43E0, 0x43E1, 0x40F0, 0x7F7F, 0x0080, 0x0003])
def test_quant_1x32_exhaustive_bf16_against_torch(amax_bits):
    rng = np.random.default_rng(5)
    g = groups_with_amax(amax_bits, rng)                       # rows of 128 values, amax fixed
    x = g.reshape(-1, 32)                                      # every 32-group keeps its own amax
    q, eb = O.quant_act_1x32_ue8m0(x)
    e = eb[0].astype(np.int64) - O.UE8M0_BIAS
    assert np.array_equal(e, O.act_exponent_ue8m0(np.max(np.abs(O.bf16_bits_to_f64(x)), axis=1)))
    assert np.array_equal(q, _torch_codes(x, e))


def test_quant_1x32_invariants():
    x = synth.activations(3, 64, 512, outliers=True)
    q, eb = O.quant_act_1x32_ue8m0(x)
    xv = O.bf16_bits_to_f64(x).reshape(64, 16, 32)
    e = (eb.T.astype(np.int64) - O.UE8M0_BIAS)[..., None]
    dq = O.e4m3_decode(q).reshape(64, 16, 32) * np.exp2(e.astype(np.float64))
    # |x - dq| <= half an e4m3 ulp at q's binade: 2^-4 relative (normal codes), 2^-10 * 2^e absolute (subnormal)
    bound = np.maximum(np.abs(dq) * 2.0 ** -4, 2.0 ** -10 * np.exp2(e.astype(np.float64)))
    assert np.all(np.abs(xv - dq) <= bound)
    # no saturation: the group maximum divided by 2^e lies in (224, 448]
    amax = np.max(np.abs(xv), axis=-1)
    r = amax / np.exp2(e[..., 0].astype(np.float64))
    assert np.all((r > 224.0) & (r <= 448.0))


def _tiny_ue8m0(seed, M=3, N=64, K=96):
    g = np.random.default_rng(seed)
    a = synth.finite_e4m3_codes(seed, (M, K))
    b = synth.finite_e4m3_codes(seed + 1, (N, K))
    ea = g.integers(127 - 20, 127 + 20, size=(K // 32, M)).astype(np.uint8)
    eb = g.integers(127 - 14, 127 + 8, size=(N // 32, K // 32)).astype(np.uint8)
    return a, ea, b, eb


def test_gemm_ue8m0_against_fraction_brute_force():
    a, ea, b, eb = _tiny_ue8m0(7)
    M, K = a.shape
    N = b.shape[0]
    A = torch.from_numpy(a).view(torch.float8_e4m3fn).double().numpy()
    B = torch.from_numpy(b).view(torch.float8_e4m3fn).double().numpy()
    C = O.gemm_w8a8_ue8m0(a, ea, b, eb)
    for m in range(M):
        for n in range(N):
            ref = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                t = (Fraction(A[m, k]) * Fraction(2) ** (int(ea[k // 32, m]) - 127) *
                     Fraction(B[n, k]) * Fraction(2) ** (int(eb[n // 32, k // 32]) - 127))
                ref += t
                mag += abs(t)
            # every term is exact in float64; only the K - 1 additions round
            assert abs(Fraction(C[m, n]) - ref) <= mag * K * Fraction(1, 2 ** 53)


def test_gemm_ue8m0_reduces_to_blockwise_product():
    """Exponents constant over 1x128 activation groups and 128x128 weight
    blocks describe the same numbers as fp32 scales 2^(e-127) in the 128x128
    format: both products agree (up to float64 summation order)."""
    M, N, K = 5, 256, 384
    g = np.random.default_rng(2)
    a = synth.finite_e4m3_codes(2, (M, K))
    b = synth.finite_e4m3_codes(3, (N, K))
    ea128 = g.integers(110, 140, size=(K // 128, M))
    eb128 = g.integers(113, 134, size=(N // 128, K // 128))
    ea = np.repeat(ea128, 4, axis=0).astype(np.uint8)                      # [K/32, M]
    eb = np.repeat(np.repeat(eb128, 4, axis=0), 4, axis=1).astype(np.uint8)   # [N/32, K/32]
    As = np.exp2(ea128 - 127.0).astype(np.float32)
    Bs = np.exp2(eb128 - 127.0).astype(np.float32)
    C1 = O.gemm_w8a8_ue8m0(a, ea, b, eb)
    C2 = O.gemm_w8a8(a, As, b, Bs)
    assert np.allclose(C1, C2, rtol=1e-12, atol=0.0)


def test_gemm_ue8m0_one_hot_rows():
    N, K = 64, 128
    b = synth.finite_e4m3_codes(4, (N, K))
    eb = np.random.default_rng(4).integers(113, 135, size=(N // 32, K // 32)).astype(np.uint8)
    ks = [0, 31, 32, 77, 127]
    a = np.zeros((len(ks), K), dtype=np.uint8)
    ea = np.full((K // 32, len(ks)), 127, dtype=np.uint8)
    for i, k0 in enumerate(ks):
        a[i, k0] = 0x38                                     # 1.0
        ea[k0 // 32, i] = 130                               # 2^3
    C = O.gemm_w8a8_ue8m0(a, ea, b, eb)
    B = torch.from_numpy(b).view(torch.float8_e4m3fn).double().numpy()
    for i, k0 in enumerate(ks):
        want = B[:, k0] * 8.0 * np.exp2(eb[np.arange(N) // 32, k0 // 32].astype(np.float64) - 127.0)
        assert np.array_equal(C[i], want)
