"""Pins of the oracle's number formats against what the pages and the
mathematics fix, independent of the oracle's own formulas.

Routes used here, none of which re-types the oracle's decode formula:
  * the page facts in tests/golden/e4m3_page_facts.txt;
  * the integer identity of "SM70 FP8 block-32 kernels", How it works
    ((b & 0x7F) << 7 | (b & 0x80) << 8 read as FP16 is the value x 2^-8),
    evaluated by numpy's float16;
  * torch's float8_e4m3fn type (a library implementation of the format);
  * exhaustive searches and closed-form properties.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_page_facts.txt")


def _parse_value(tok):
    if tok.startswith("2^"):
        return 2.0 ** int(tok[2:])
    return float(tok)


def page_facts():
    facts = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, _cite = line.split("|", 1)
            name, value = head.split()
            facts[name] = _parse_value(value)
    return facts


ALL = np.arange(256, dtype=np.uint8)
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_golden_file_has_citations():
    with open(GOLDEN) as f:
        rows = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    for r in rows:
        assert "|" in r and len(r.split("|", 1)[1].strip()) > 10


def test_decode_against_page_facts():
    F = page_facts()
    v = O.e4m3_decode(FINITE)
    assert np.nanmax(np.abs(v)) == F["e4m3_max"]
    # multiples of the grid step, at most 4 significant bits
    q = v / F["e4m3_grid"]
    assert np.all(q == np.round(q))
    for x in np.abs(v[v != 0]):
        fr = Fraction(float(x))
        num = fr.numerator
        while num % 2 == 0:
            num //= 2
        assert num.bit_length() <= F["e4m3_max_significant_bits"]
    # smallest nonzero magnitude and largest binade
    assert np.min(np.abs(v[v != 0])) == F["e4m3_smallest_binade"]
    assert 2.0 ** np.floor(np.log2(np.max(np.abs(v)))) == F["e4m3_largest_binade"]
    # 3 mantissa bits: 8 values per binade above the subnormals
    b = v[(v >= 1.0) & (v < 2.0)]
    assert len(b) == 2 ** int(F["e4m3_mantissa_bits"])


def test_decode_nan_codes_and_specials():
    v = O.e4m3_decode(ALL)
    nan = np.isnan(v)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6           # smallest normal
    assert v[0x01] == 2.0 ** -9           # smallest subnormal
    assert v[0x00] == 0.0 and not np.signbit(v[0x00])
    assert v[0x80] == 0.0 and np.signbit(v[0x80])
    assert v[0x38] == 1.0
    assert np.count_nonzero(~nan) == 254


def test_decode_matches_p3_fp16_identity():
    """(b & 0x7F) << 7 | (b & 0x80) << 8, read as an IEEE fp16 bit pattern,
    equals the e4m3 value times 2^-8 for every finite code."""
    F = page_facts()
    b = FINITE.astype(np.uint16)
    bits = ((b & 0x7F) << 7) | ((b & 0x80) << 8)
    h = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(h, O.e4m3_decode(FINITE) * F["fp16_identity_factor"])
    # 2^-8 is the fp16/e4m3 exponent-bias gap stated by the 3090 page
    assert F["fp16_identity_factor"] == 1.0 / F["fp16_bias_gap"]


def test_decode_matches_torch_float8_e4m3fn():
    t = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = O.e4m3_decode(ALL)
    assert np.array_equal(np.isnan(t), np.isnan(v))
    ok = ~np.isnan(v)
    assert np.array_equal(t[ok], v[ok])
    assert np.array_equal(np.signbit(t[ok]), np.signbit(v[ok]))


def test_bf16_bias_gap_identity():
    """(b & 0x7F) << 4 | (b & 0x80) << 8, read as bf16, is the value x 2^-120:
    the bias gap the 3090 page states for bf16."""
    F = page_facts()
    b = FINITE.astype(np.uint32)
    bits = (((b & 0x7F) << 4) | ((b & 0x80) << 8)) << 16
    f = bits.astype(np.uint32).view(np.float32).astype(np.float64)
    assert np.array_equal(f * F["bf16_bias_gap"], O.e4m3_decode(FINITE))


def test_window_exact_in_fp16_and_bf16():
    """v * 2^e is exact in fp16 (and bf16) for every finite code and every e
    in the page's window; at e = 8 the largest code overflows fp16."""
    F = page_facts()
    v = O.e4m3_decode(FINITE)
    for e in range(int(F["ue8m0_window_min"]), int(F["ue8m0_window_max"]) + 1):
        x = v * 2.0 ** e
        assert np.array_equal(x.astype(np.float16).astype(np.float64), x), e
        xb = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(xb, x), e
    big = 448.0 * 2.0 ** F["fp16_overflow_exponent"]
    with np.errstate(over="ignore"):
        assert np.isinf(np.float16(big))


def test_ue8m0_value():
    assert O.ue8m0_value(127) == 1.0
    assert O.ue8m0_value(127 - 14) == 2.0 ** -14
    assert O.ue8m0_value(127 + 7) == 128.0


def test_encode_roundtrip_all_finite_codes():
    v = O.e4m3_decode(FINITE)
    assert np.array_equal(O.e4m3_encode(v), FINITE)


def _torch_encode(x64):
    """torch's float32 -> float8_e4m3fn cast (nearest-even; overflow -> NaN)."""
    t = torch.from_numpy(np.asarray(x64, dtype=np.float32).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encode_matches_torch_on_all_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.astype(np.uint32).view(np.float32)
    fin = np.isfinite(x) & (np.abs(x) < 464.0)      # torch does not saturate
    ours = O.e4m3_encode(x[fin].astype(np.float64))
    ref = _torch_encode(x[fin])
    assert np.array_equal(ours, ref)


def test_encode_midpoints_and_neighbours():
    """Exact midpoints between neighbouring codes go to the even code; one
    float32 ulp either side goes to the nearer code."""
    g = O.e4m3_finite_values()
    mids = ((g[:-1] + g[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (g[:-1] + g[1:]) / 2)
    pts = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    pts = np.concatenate([pts, -pts])
    assert np.array_equal(O.e4m3_encode(pts.astype(np.float64)), _torch_encode(pts))
    # ties go to the even code: code index i or i+1, whichever is even
    codes = O.e4m3_encode(mids.astype(np.float64))
    assert np.all(codes % 2 == 0)


def test_encode_saturates_and_keeps_sign():
    x = np.array([448.0, 449.0, 463.99, 464.0, 1e30, -1e30, -0.0, 0.0, -1e-30, np.nan])
    c = O.e4m3_encode(x)
    assert list(c) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00, 0x80, 0x7F]


def test_encode_random_fp32_against_torch():
    r = np.random.default_rng(123)
    x = (r.standard_normal(200000) * np.exp2(r.integers(-20, 9, 200000))).astype(np.float32)
    x = x[np.abs(x) < 464]
    assert np.array_equal(O.e4m3_encode(x.astype(np.float64)), _torch_encode(x))


def test_fp32_div_is_ieee():
    r = np.random.default_rng(7)
    a = (r.standard_normal(100000) * 100).astype(np.float32)
    b = (np.abs(r.standard_normal(100000)) + 1e-3).astype(np.float32)
    ref = (torch.from_numpy(a) / torch.from_numpy(b)).numpy()
    assert np.array_equal(O.fp32_div(a, b), ref)
    # denormal divisors (tiny amax) too
    bd = np.array([1e-42, 3e-41, 1.4e-45], dtype=np.float32)
    ad = np.array([1e-40, 2e-41, 1.4e-45], dtype=np.float32)
    assert np.array_equal(O.fp32_div(ad, bd), (torch.from_numpy(ad) / torch.from_numpy(bd)).numpy())


def test_bf16_helpers_roundtrip():
    r = np.random.default_rng(3)
    bits = r.integers(0, 65536, 10000).astype(np.uint16)
    x = O.bf16_bits_to_f64(bits)
    fin = np.isfinite(x) & (np.abs(x) > 2.0 ** -126)
    assert np.array_equal(O.f64_to_bf16_bits(x[fin]), bits[fin])
    y = r.standard_normal(1000)
    ref = torch.from_numpy(y).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    # torch rounds f64 -> f32 -> bf16 (double rounding); compare where f32 is exact enough
    ours = O.f64_to_bf16_bits(y.astype(np.float32).astype(np.float64))
    assert np.array_equal(ours, ref)
