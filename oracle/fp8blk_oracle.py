"""CPU oracle for the block-scaled FP8 linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the GPU product path imports, calls or
links this file.  It is used by ``tests/``, by ``__graft_entry__.smoke()`` and
by the CPU-baseline leg of ``bench.py``.

Everything is float64 numpy unless a step is fixed to another precision by the
method (the fp32 scales and the fp32 quotient that decides an e4m3 code).  No
blocking, fusion or reordering beyond what each definition states; one numpy
matmul per 128-wide K block is the only library primitive.

Sources (page title, section):
  [P1] "Blockwise FP8 on Ada GPUs, part 2: my kernel was correct and 4x too
       slow" -- "The starting point" (1x128 per-token activation groups,
       128x128 weight blocks), "The fix" (one FP32 partial per 128-wide K
       block, promoted once with As*Bs).
  [P2] "perf(ArcKernels): blockwise-FP8 GEMM on tensor cores, scale promoted
       per 128-K" -- "What this adds" ([N/128, K/128] weight scales, exact
       e4m3 -> 16-bit conversion), "Route-2 handover" finding 2 (activation
       scales [M, ceil(K/128)], M-major).
  [P3] "SM70 FP8 block-32 kernels (PLI Labs)" -- "How it works" (UE8M0 scale
       per 32x32 block, integer e4m3 -> fp16 identity), "Exactness" (e4m3
       values are multiples of 2^-9 with at most 4 significant bits, |v|<=448;
       v*2^e exact in fp16 for e in [-14, 7]; NaN codes refused).
  [P4] "FP8 / NVFP4 weight-only inference on the RTX 3090 loses nothing" --
       section 4.1 (E4M3 "fn" variant, exact conversion to fp16/bf16).

Parity pins (tests/test_oracle_pins.py, tests/test_oracle_quant.py,
tests/test_oracle_gemm.py):
  e4m3_decode            pinned: page facts (tests/golden), P3's fp16 integer
                         identity via numpy float16, torch float8_e4m3fn.
  e4m3_encode            pinned: round trip on all finite codes, torch's RNE
                         conversion on all bf16 patterns and on midpoints.
  quant_act_1x128        pinned: torch CPU route (fp32 divide + RNE cast) on
                         exhaustive bf16 groups, error-bound invariants.
  quant_weight_128x128   pinned: same rule per block; block-structure checks.
  gemm_w8a8              pinned: exact int64 / Fraction brute force on tiny
                         inputs, one-hot rows, unit-scale reduction.
  gemm_w8a16_f32scale    pinned: Fraction brute force on tiny inputs.
  gemm_w8a16_ue8m0       pinned: Fraction brute force on tiny inputs.
  gemm_w8a8_grouped      pinned: one group reduces to gemm_w8a8; every row
                         equals the single-weight product with its group's
                         weights (int64 brute force on tiny inputs); row-block
                         permutation invariance; padding rows stay untouched.
  act_exponent_ue8m0     pinned: minimality checked by exact comparisons on
                         every finite bf16 magnitude; page-independent special
                         values (448 -> 0, 450 -> 1, 224 -> -1, 1 -> -8, 0 and
                         subnormals -> -127).
  quant_act_1x32_ue8m0   pinned: torch's float8_e4m3fn cast of x * 2^-e on
                         exhaustive bf16 groups; reconstruction within half an
                         e4m3 ulp; the group maximum lands in (224, 448].
  gemm_w8a8_ue8m0        pinned: Fraction brute force on tiny inputs; reduces
                         to gemm_w8a8 when the exponents are constant over
                         1x128 / 128x128 blocks; one-hot rows.
  End-to-end output numbers are "parity unpinned" against the pages: no page
  prints a per-element worked example of the product.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "E4M3_MAX", "E4M3_NAN_CODES", "e4m3_decode", "e4m3_encode", "e4m3_finite_values",
    "bf16_bits_to_f64", "f64_to_bf16_bits", "fp32_div", "ue8m0_value",
    "quant_act_1x128", "quant_weight_128x128",
    "gemm_w8a8", "gemm_w8a16_f32scale", "gemm_w8a16_ue8m0", "gemm_w8a8_grouped",
    "gemm_w8a8_rows", "gemm_w8a16_f32scale_rows", "gemm_w8a16_ue8m0_rows",
    "UE8M0_EMIN", "UE8M0_EMAX", "UE8M0_BIAS",
    "ACT_EXP_MIN", "ACT_EXP_MAX", "act_exponent_ue8m0", "quant_act_1x32_ue8m0",
    "gemm_w8a8_ue8m0", "gemm_w8a8_ue8m0_rows",
]

# Largest finite e4m3 magnitude and the two NaN codes of the finite-only
# ("fn") e4m3 variant [P3 "Exactness"; P4 4.1].
E4M3_MAX = 448.0
E4M3_NAN_CODES = (0x7F, 0xFF)

# UE8M0 scale: one unsigned byte per block holding a power of two.  The pages
# give the window e in [-14, 7] [P3 "Exactness"] but not the byte's bias; the
# reading here is the usual E8M0 bias 127 (byte = e + 127).
UE8M0_BIAS = 127
UE8M0_EMIN = -14
UE8M0_EMAX = 7

QBLOCK = 128          # K width of one scale block [P1 "The starting point"]
UE8M0_BLOCK = 32      # side of one UE8M0 block [P3 "How it works"]

# W8A8 in the 32x32 UE8M0 format needs power-of-two activation scales too,
# one per token per 32 values of K (a 32x32 weight block meets 1x32
# activation groups).  The pages fix neither the rule nor the range; the
# reading: the smallest power of two 2^e with 448 * 2^e >= amax (no element
# saturates), e clamped to the byte range of a UE8M0 scale [-127, 127]
# (byte 255 is NaN in E8M0), and amax == 0 takes the clamp, e = -127.
ACT_EXP_MIN = -127
ACT_EXP_MAX = 127


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 byte, as float64 [P3 "Exactness"; P4 4.1].

    Byte b = s|EEEE|mmm.  E == 0 is the subnormal range: (-1)^s * m * 2^-9.
    Otherwise (-1)^s * (1 + m/8) * 2^(E-7).  0x7F and 0xFF are NaN; there is
    no infinity, so 0x7E = 448 is the largest finite value.
    """
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    E = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(E == 0,
                   m.astype(np.float64) * 2.0 ** -9,
                   (1.0 + m.astype(np.float64) / 8.0) * np.exp2((E - 7).astype(np.float64)))
    v = np.where(s == 1, -mag, mag)
    nan = (b & 0x7F) == 0x7F
    return np.where(nan, np.nan, v)


def e4m3_finite_values() -> np.ndarray:
    """The 127 non-negative finite e4m3 values, ascending (codes 0x00..0x7E)."""
    return e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))


_POS = None


def _pos_grid():
    global _POS
    if _POS is None:
        _POS = e4m3_finite_values()
    return _POS


def e4m3_encode(x) -> np.ndarray:
    """Round values to e4m3 codes: nearest, ties to even, saturating.

    The pages never state the overflow rule; the reading is "satfinite": any
    magnitude above 448 becomes +-448.  The sign is kept, so a negative value
    (or -0.0) that rounds to zero gives 0x80.  A NaN input gives 0x7F.
    Ties pick the code whose last mantissa bit is 0 (the even code).
    Comparisons are made against the exact midpoints of neighbouring grid
    values, so the rounding is exact for every float64 input.
    """
    x = np.asarray(x, dtype=np.float64)
    grid = _pos_grid()
    a = np.abs(x)
    sign = np.signbit(x)
    hi = np.searchsorted(grid, a, side="left")           # grid[hi-1] < a <= grid[hi]
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    glo = grid[lo]
    ghi = grid[hi]
    mid = (glo + ghi) * 0.5                                # exact: <= 5 significant bits
    pick_hi = (a > mid) | ((a == mid) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == grid[hi], hi, code)               # exact hits
    code = np.where(a >= E4M3_MAX, 0x7E, code)             # satfinite
    code = code.astype(np.int64) | np.where(sign, 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns to float64 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (nearest, ties to even), for
    reporting.  Rounds straight to 8 significant bits with frexp/rint (numpy
    rint is ties-to-even), so there is no double rounding.  Meant for values
    in bf16's normal range."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    r = np.rint(np.ldexp(m, 8))           # 8 significant bits
    y = np.ldexp(r, e - 8).astype(np.float32)   # exact: fits in float32
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp32_div(a, b) -> np.ndarray:
    """Correctly rounded float32 quotient of float32 operands.

    Computed as the float64 quotient rounded to float32.  Double rounding is
    harmless for division when the wide format has at least 2p+2 bits
    (53 >= 2*24+2), so this equals IEEE float32 division.
    """
    a = np.asarray(a, dtype=np.float32).astype(np.float64)
    b = np.asarray(b, dtype=np.float32).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        return (a / b).astype(np.float32)


def ue8m0_value(byte) -> np.ndarray:
    """Scale value 2^(byte - 127) of a UE8M0 byte [P3 "How it works"]."""
    return np.exp2(np.asarray(byte, dtype=np.int64).astype(np.float64) - UE8M0_BIAS)


# ---------------------------------------------------------------------------
# Quantisers
# ---------------------------------------------------------------------------

def _quant_group(x32: np.ndarray):
    """Quantise the last axis of ``x32`` (float32, one group per row) to e4m3.

    amax = max |x| (exact), s = fl32(amax / 448), q = e4m3(fl32(x / s)).
    The code is decided on the float32 quotient, the precision the scales are
    stored in.  amax == 0 (pages silent): s = 1.0, and every element still goes
    through q = e4m3(x / s), which gives 0x00 or 0x80 by the sign of zero.
    """
    amax = np.max(np.abs(x32), axis=-1)
    s = fp32_div(amax, np.float32(E4M3_MAX))
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    q = e4m3_encode(fp32_div(x32, s[..., None]))
    return q, s


def quant_act_1x128(x_bf16_bits: np.ndarray):
    """Per-token 1x128 activation quantisation [P1 "The starting point";
    P2 "Route-2 handover" finding 2].

    x: bf16 bits [M, K], K % 128 == 0.
    Returns (codes uint8 [M, K], scales float32 [K/128, M]).  The scale layout
    is the reading of "[M, ceil(K/128)], M-major": M is the contiguous axis.
    """
    x = np.asarray(x_bf16_bits, dtype=np.uint16)
    M, K = x.shape
    assert K % QBLOCK == 0
    x32 = bf16_bits_to_f64(x).astype(np.float32).reshape(M, K // QBLOCK, QBLOCK)
    q, s = _quant_group(x32)
    return q.reshape(M, K), np.ascontiguousarray(s.T)


def quant_weight_128x128(w_bf16_bits: np.ndarray):
    """128x128 weight block quantisation [P1 "The starting point";
    P2 "What this adds"].

    w: bf16 bits [N, K], N % 128 == 0, K % 128 == 0.
    Returns (codes uint8 [N, K], scales float32 [N/128, K/128]).
    """
    w = np.asarray(w_bf16_bits, dtype=np.uint16)
    N, K = w.shape
    assert N % QBLOCK == 0 and K % QBLOCK == 0
    nb, kb = N // QBLOCK, K // QBLOCK
    w32 = bf16_bits_to_f64(w).astype(np.float32)
    blocks = w32.reshape(nb, QBLOCK, kb, QBLOCK).transpose(0, 2, 1, 3).reshape(nb, kb, QBLOCK * QBLOCK)
    q, s = _quant_group(blocks)
    q = q.reshape(nb, kb, QBLOCK, QBLOCK).transpose(0, 2, 1, 3).reshape(N, K)
    return np.ascontiguousarray(q), s.astype(np.float32)


# ---------------------------------------------------------------------------
# Products
# ---------------------------------------------------------------------------

def gemm_w8a8_rows(a_codes, a_scales, b_codes, b_scales, rows=None) -> np.ndarray:
    """W8A8 block-scaled product for selected rows, float64.

    C[m, n] = sum_kb As[kb, m] * Bs[n // 128, kb] * P[m, n, kb],
    P[m, n, kb] = sum_{k in block kb} dec(A[m, k]) * dec(B[n, k])
    [P1 "The fix"; P2 "What this adds"].  P is exact in float64 (every e4m3
    value is an integer times 2^-9, |P| < 2^25, so at most 43 significant
    bits), so the matmul's summation order does not matter.

    a_codes [M, K] uint8, a_scales [K/128, M] float32 (M contiguous),
    b_codes [N, K] uint8, b_scales [N/128, K/128] float32.
    """
    A = np.asarray(a_codes)
    B = np.asarray(b_codes)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A = A[rows]
    As = np.asarray(a_scales, dtype=np.float32).astype(np.float64)
    As = As if rows is None else As[:, rows]
    Bs = np.asarray(b_scales, dtype=np.float32).astype(np.float64)
    Mr, K = A.shape
    N = B.shape[0]
    Ad = e4m3_decode(A)
    Bd = e4m3_decode(B)
    C = np.zeros((Mr, N), dtype=np.float64)
    n_block = np.arange(N) // QBLOCK
    for kb in range(K // QBLOCK):
        ks = slice(kb * QBLOCK, (kb + 1) * QBLOCK)
        P = Ad[:, ks] @ Bd[:, ks].T
        C += P * As[kb][:, None] * Bs[n_block, kb][None, :]
    return C


def gemm_w8a8(a_codes, a_scales, b_codes, b_scales) -> np.ndarray:
    return gemm_w8a8_rows(a_codes, a_scales, b_codes, b_scales, None)


def gemm_w8a8_grouped(a_codes, a_scales, b_codes, b_scales, row_group, fill=np.nan) -> np.ndarray:
    """Grouped (mixture-of-experts) form of the W8A8 product: row m of A is
    multiplied by the weights of group row_group[m] (one expert per row, the
    rows of each expert stored contiguously), with the same block scaling as
    gemm_w8a8 [P1 "The fix"].  Rows with row_group[m] < 0 are padding and
    get `fill` (the GPU leaves them untouched).

    b_codes [G, N, K] uint8, b_scales [G, N/128, K/128] float32,
    row_group [M] int; other arguments as gemm_w8a8.
    """
    A = np.asarray(a_codes)
    g = np.asarray(row_group, dtype=np.int64)
    M = A.shape[0]
    B = np.asarray(b_codes)
    C = np.full((M, B.shape[1]), fill, dtype=np.float64)
    for e in range(B.shape[0]):
        rows = np.nonzero(g == e)[0]
        if rows.size:
            C[rows] = gemm_w8a8_rows(A, a_scales, B[e], np.asarray(b_scales)[e], rows)
    return C


def gemm_w8a16_f32scale_rows(x_bf16_bits, b_codes, b_scales, rows=None) -> np.ndarray:
    """W8A16 product with 128x128 fp32 weight scales, float64.

    C[m, n] = sum_kb Bs[n // 128, kb] * sum_{k in kb} x[m, k] * dec(B[n, k])
    [P2 "What this adds": weights stay FP8, the block scale is applied once
    per 128-K block].  x is bf16, widened exactly.
    """
    X = np.asarray(x_bf16_bits, dtype=np.uint16)
    if rows is not None:
        X = X[np.asarray(rows, dtype=np.int64)]
    x = bf16_bits_to_f64(X)
    Bd = e4m3_decode(b_codes)
    Bs = np.asarray(b_scales, dtype=np.float32).astype(np.float64)
    Mr, K = x.shape
    N = Bd.shape[0]
    C = np.zeros((Mr, N), dtype=np.float64)
    n_block = np.arange(N) // QBLOCK
    for kb in range(K // QBLOCK):
        ks = slice(kb * QBLOCK, (kb + 1) * QBLOCK)
        C += (x[:, ks] @ Bd[:, ks].T) * Bs[n_block, kb][None, :]
    return C


def gemm_w8a16_f32scale(x_bf16_bits, b_codes, b_scales) -> np.ndarray:
    return gemm_w8a16_f32scale_rows(x_bf16_bits, b_codes, b_scales, None)


def gemm_w8a16_ue8m0_rows(x_bf16_bits, b_codes, b_scale_bytes, rows=None) -> np.ndarray:
    """W8A16 product with one UE8M0 scale per 32x32 weight block, float64.

    C[m, n] = sum_k x[m, k] * dec(B[n, k]) * 2^(e[n // 32, k // 32])
    [P3 "How it works", "Exactness"].
    """
    X = np.asarray(x_bf16_bits, dtype=np.uint16)
    if rows is not None:
        X = X[np.asarray(rows, dtype=np.int64)]
    x = bf16_bits_to_f64(X)
    Bd = e4m3_decode(b_codes)
    N, K = Bd.shape
    sc = ue8m0_value(b_scale_bytes)                                   # [N/32, K/32]
    W = Bd * np.repeat(np.repeat(sc, UE8M0_BLOCK, axis=0), UE8M0_BLOCK, axis=1)
    return x @ W.T


def gemm_w8a16_ue8m0(x_bf16_bits, b_codes, b_scale_bytes) -> np.ndarray:
    return gemm_w8a16_ue8m0_rows(x_bf16_bits, b_codes, b_scale_bytes, None)


# ---------------------------------------------------------------------------
# W8A8 in the 32x32 UE8M0 format
# ---------------------------------------------------------------------------

def act_exponent_ue8m0(amax) -> np.ndarray:
    """Exponent e of a 1x32 activation group's power-of-two scale: the
    smallest integer with 448 * 2^e >= amax, clamped to [-127, 127]
    (reading; see ACT_EXP_MIN).  Written out as that definition: start from
    the float estimate ceil(log2(amax / 448)) and step to the smallest
    integer that passes the exact test 448 * 2^e >= amax (both sides exact
    in float64).  amax == 0 gives the clamp, -127."""
    a = np.asarray(amax, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.int64)
    for idx, v in np.ndenumerate(a):
        if v == 0.0:
            out[idx] = ACT_EXP_MIN
            continue
        e = int(np.ceil(np.log2(v / E4M3_MAX)))
        while np.ldexp(E4M3_MAX, e) < v:            # too small: 448 * 2^e must reach amax
            e += 1
        while np.ldexp(E4M3_MAX, e - 1) >= v:       # not the smallest
            e -= 1
        out[idx] = min(max(e, ACT_EXP_MIN), ACT_EXP_MAX)
    return out


def quant_act_1x32_ue8m0(x_bf16_bits: np.ndarray):
    """Per-token 1x32 activation quantisation with UE8M0 (power-of-two)
    scales, for W8A8 in the 32x32 UE8M0 weight format ("SM70 FP8 block-32
    kernels", "How it works": one power of two per 32x32 block; "perf
    (ArcKernels)", "Cheap checks done first": the VEC32_UE8M0 scale modes).

    x: bf16 bits [M, K], K % 32 == 0.  Per group of 32: e from
    act_exponent_ue8m0(max |x|), q = e4m3(x * 2^-e) (nearest, ties to even;
    x * 2^-e is exact and never above 448, so no code saturates).
    Returns (codes uint8 [M, K], exponent bytes uint8 [K/32, M] = e + 127,
    M contiguous like the fp32 activation scales).
    """
    x = np.asarray(x_bf16_bits, dtype=np.uint16)
    M, K = x.shape
    assert K % UE8M0_BLOCK == 0
    xv = bf16_bits_to_f64(x).reshape(M, K // UE8M0_BLOCK, UE8M0_BLOCK)
    e = act_exponent_ue8m0(np.max(np.abs(xv), axis=-1))           # [M, K/32]
    q = e4m3_encode(xv * np.exp2(-e.astype(np.float64))[..., None])
    return q.reshape(M, K), np.ascontiguousarray((e + UE8M0_BIAS).astype(np.uint8).T)


def gemm_w8a8_ue8m0_rows(a_codes, a_exp_bytes, b_codes, b_exp_bytes, rows=None) -> np.ndarray:
    """W8A8 product in the 32x32 UE8M0 format, float64:

        C[m, n] = sum_k dec(A[m, k]) 2^(ea[k/32, m] - 127) dec(B[n, k]) 2^(eb[n/32, k/32] - 127)

    ("SM70 FP8 block-32 kernels", "How it works": the weight's power of two
    per 32x32 block; the activation's per 1x32 group).  a_exp_bytes
    [K/32, M] (M contiguous), b_exp_bytes [N/32, K/32].
    """
    A = np.asarray(a_codes)
    ea = np.asarray(a_exp_bytes)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        A = A[rows]
        ea = ea[:, rows]
    Ad = e4m3_decode(A) * np.repeat(ue8m0_value(ea).T, UE8M0_BLOCK, axis=1)
    Bd = e4m3_decode(b_codes)
    sb = ue8m0_value(b_exp_bytes)
    Bd = Bd * np.repeat(np.repeat(sb, UE8M0_BLOCK, axis=0), UE8M0_BLOCK, axis=1)
    return Ad @ Bd.T


def gemm_w8a8_ue8m0(a_codes, a_exp_bytes, b_codes, b_exp_bytes) -> np.ndarray:
    return gemm_w8a8_ue8m0_rows(a_codes, a_exp_bytes, b_codes, b_exp_bytes, None)
