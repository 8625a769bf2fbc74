"""Pins of the oracle's products by brute force on tiny inputs.

Values of e4m3 codes come from torch's float8_e4m3fn type (not from the
oracle's decoder); sums are taken exactly, in int64 or with Fractions, in
plain loops over the definitions' indices.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import synth


def torch_dec(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def as_int9(codes):
    """e4m3 values in units of 2^-9 as int64 (every finite value is one)."""
    v = torch_dec(codes) * 512.0
    assert np.all(v == np.round(v))
    return v.astype(np.int64)


def tiny_w8a8(seed, M=3, N=256, K=256):
    x = synth.activations(seed, M, K, outliers=True)
    a, As = O.quant_act_1x128(x)
    w = synth.weights_bf16(seed, N, K)
    b, Bs = O.quant_weight_128x128(w)
    # make the two N blocks' scales clearly different
    Bs = Bs * np.array([[1.0], [3.0]], dtype=np.float32)
    return a, As, b, Bs


def test_w8a8_unit_scales_equal_exact_integer_product():
    a, As, b, Bs = tiny_w8a8(0)
    ones_a = np.ones_like(As)
    ones_b = np.ones_like(Bs)
    C = O.gemm_w8a8(a, ones_a, b, ones_b)
    P = as_int9(a) @ as_int9(b).T                 # exact int64, units 2^-18
    assert np.array_equal(C, P.astype(np.float64) * 2.0 ** -18)


def test_w8a8_against_fraction_brute_force():
    a, As, b, Bs = tiny_w8a8(1)
    M, K = a.shape
    N = b.shape[0]
    C = O.gemm_w8a8(a, As, b, Bs)
    ai, bi = as_int9(a), as_int9(b)
    for m in range(M):
        for n in (0, 1, 77, 127, 128, 200, 255):
            tot = Fraction(0)
            for kb in range(K // 128):
                p = 0
                for k in range(kb * 128, (kb + 1) * 128):
                    p += int(ai[m, k]) * int(bi[n, k])
                tot += Fraction(p, 2 ** 18) * Fraction(float(As[kb, m])) * Fraction(float(Bs[n // 128, kb]))
            ref = float(tot)
            assert abs(C[m, n] - ref) <= 1e-13 * abs(ref) + 1e-300, (m, n)


def test_w8a8_one_hot_rows_select_scaled_weight_columns():
    """A row with a single 1.0 at column k0 and As = 1 gives Bs * dec(B[:, k0])."""
    N, K = 256, 384
    w = synth.weights_bf16(3, N, K)
    b, Bs = O.quant_weight_128x128(w)
    ks = [0, 5, 127, 128, 300, 383]
    a = np.zeros((len(ks), K), dtype=np.uint8)
    for i, k0 in enumerate(ks):
        a[i, k0] = 0x38                            # 1.0
    As = np.ones((K // 128, len(ks)), dtype=np.float32)
    C = O.gemm_w8a8(a, As, b, Bs)
    bd = torch_dec(b)
    for i, k0 in enumerate(ks):
        ref = bd[:, k0] * np.repeat(Bs[:, k0 // 128].astype(np.float64), 128)
        assert np.array_equal(C[i], ref)


def test_w8a8_rows_subset_matches_full():
    a, As, b, Bs = tiny_w8a8(4, M=7)
    C = O.gemm_w8a8(a, As, b, Bs)
    rows = np.array([0, 3, 6])
    assert np.array_equal(O.gemm_w8a8_rows(a, As, b, Bs, rows), C[rows])


def test_w8a16_f32scale_against_fraction_brute_force():
    M, N, K = 2, 256, 256
    x = synth.activations(5, M, K)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(5, N, K))
    C = O.gemm_w8a16_f32scale(x, b, Bs)
    xv = O.bf16_bits_to_f64(x)
    bd = torch_dec(b)
    for m in range(M):
        for n in (0, 64, 127, 128, 255):
            tot = Fraction(0)
            for kb in range(K // 128):
                p = Fraction(0)
                for k in range(kb * 128, (kb + 1) * 128):
                    p += Fraction(float(xv[m, k])) * Fraction(float(bd[n, k]))
                tot += p * Fraction(float(Bs[n // 128, kb]))
            ref = float(tot)
            assert abs(C[m, n] - ref) <= 1e-12 * max(abs(ref), 1e-6), (m, n)


def test_w8a16_ue8m0_against_fraction_brute_force():
    M, N, K = 2, 64, 96
    x = synth.activations(6, M, K)
    b, e = synth.ue8m0_weights(6, N, K)
    C = O.gemm_w8a16_ue8m0(x, b, e)
    xv = O.bf16_bits_to_f64(x)
    bd = torch_dec(b)
    for m in range(M):
        for n in (0, 31, 32, 63):
            tot = Fraction(0)
            for k in range(K):
                tot += Fraction(float(xv[m, k])) * Fraction(float(bd[n, k])) * Fraction(2) ** (int(e[n // 32, k // 32]) - 127)
            ref = float(tot)
            assert abs(C[m, n] - ref) <= 1e-12 * max(abs(ref), 1e-6), (m, n)


def test_w8a16_unit_scale_reduces_to_plain_matmul():
    M, N, K = 3, 128, 256
    x = synth.activations(7, M, K)
    b, _ = O.quant_weight_128x128(synth.weights_bf16(7, N, K))
    ones = np.ones((1, 2), dtype=np.float32)
    C = O.gemm_w8a16_f32scale(x, b, ones)
    ref = torch.from_numpy(O.bf16_bits_to_f64(x)) @ torch.from_numpy(torch_dec(b)).T
    assert np.allclose(C, ref.numpy(), rtol=1e-14, atol=1e-12)
    # UE8M0 with every byte 127 (scale 1) is the same product
    e = np.full((N // 32, K // 32), 127, dtype=np.uint8)
    assert np.allclose(O.gemm_w8a16_ue8m0(x, b, e), ref.numpy(), rtol=1e-14, atol=1e-12)


# ---------------------------------------------------------------- grouped (mixture-of-experts) form

def tiny_grouped(seed, G=3, rows_per_group=(2, 3, 1), N=256, K=256):
    M = sum(rows_per_group)
    x = synth.activations(seed, M, K, outliers=True)
    a, As = O.quant_act_1x128(x)
    bs, Bss = [], []
    for e in range(G):
        b, Bs = O.quant_weight_128x128(synth.weights_bf16(seed * 10 + e, N, K))
        bs.append(b)
        Bss.append(Bs * np.float32(1.0 + e))     # clearly different scales per expert
    g = np.repeat(np.arange(G), rows_per_group)
    return a, As, np.stack(bs), np.stack(Bss), g


def test_grouped_single_group_is_plain_w8a8():
    a, As, b, Bs = tiny_w8a8(6, M=5)
    C = O.gemm_w8a8_grouped(a, As, b[None], Bs[None], np.zeros(5, dtype=np.int64))
    assert np.array_equal(C, O.gemm_w8a8(a, As, b, Bs))


def test_grouped_rows_against_int64_brute_force():
    """Every row equals the exact product with its own expert's weights."""
    a, As, b, Bs, g = tiny_grouped(7)
    C = O.gemm_w8a8_grouped(a, As, b, Bs, g)
    ai = as_int9(a)
    for m in range(a.shape[0]):
        e = int(g[m])
        bi = as_int9(b[e])
        for n in (0, 100, 128, 255):
            tot = Fraction(0)
            for kb in range(a.shape[1] // 128):
                p = int(np.dot(ai[m, kb * 128:(kb + 1) * 128], bi[n, kb * 128:(kb + 1) * 128]))
                tot += Fraction(p, 2 ** 18) * Fraction(float(As[kb, m])) * Fraction(float(Bs[e, n // 128, kb]))
            assert abs(C[m, n] - float(tot)) <= 1e-13 * abs(float(tot)) + 1e-300, (m, n)


def test_grouped_row_permutation_and_padding():
    a, As, b, Bs, g = tiny_grouped(8)
    C = O.gemm_w8a8_grouped(a, As, b, Bs, g)
    perm = np.array([5, 0, 3, 1, 4, 2])
    Cp = O.gemm_w8a8_grouped(a[perm], As[:, perm], b, Bs, g[perm])
    assert np.array_equal(Cp, C[perm])
    g2 = g.copy()
    g2[[1, 4]] = -1                               # padding rows
    C2 = O.gemm_w8a8_grouped(a, As, b, Bs, g2, fill=-7.0)
    assert np.all(C2[[1, 4]] == -7.0)
    keep = [0, 2, 3, 5]
    assert np.array_equal(C2[keep], C[keep])
