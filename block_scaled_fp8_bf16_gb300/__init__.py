"""Python binding of libfp8blk.so, the block-scaled FP8 linear layer for GB300.

Argument marshalling only: every function hands device pointers, sizes and
strides of PyTorch tensors to the C ABI declared in include/fp8blk.h, on the
current CUDA stream unless one is given.  Every step of the computation runs
in the library's CUDA kernels; there is no Python or CPU fallback, and the
first call raises ImportError when the library has not been built.

Functions named ``fp8blk_*`` mirror the C entry points one to one and write
into caller-provided tensors.  The short names (``quant_act``, ``gemm_w8a8``,
...) allocate their outputs and call the same entry points.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8blk.so")

SCALE_F32_128x128 = 0
SCALE_UE8M0_32x32 = 1

# Launch flags of the GEMM entry points (FP8BLK_FLAG_* in the header).
FLAG_PDL = 1
FLAG_OUT_F32 = 2

# Largest token count fp8blk_linear_w8a8 takes (quantisation fused into the GEMM).
LINEAR_FUSED_MAX_M = 32

STATUS_NAMES = {
    0: "FP8BLK_OK",
    1: "FP8BLK_ERR_INVALID_ARG",
    2: "FP8BLK_ERR_UNSUPPORTED_SHAPE",
    3: "FP8BLK_ERR_MISALIGNED",
    4: "FP8BLK_ERR_ARCH",
    5: "FP8BLK_ERR_CUDA",
    6: "FP8BLK_ERR_NAN_CODE",
    7: "FP8BLK_ERR_SCALE_WINDOW",
    8: "FP8BLK_ERR_TIMEOUT",
}

# Every symbol the header declares: name -> (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U32 = ctypes.c_uint32
EXPORTS = {
    "fp8blk_quant_act": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    "fp8blk_gemm_w8a8": (_I32, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _U32, _P]),
    "fp8blk_linear_w8a8": (_I32, [_P, _I64, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _U32, _P]),
    "fp8blk_gemm_w8a8_grouped": (_I32, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I64, _I64, _I64, _U32,
                                         _P]),
    "fp8blk_ue8m0_sf_bytes": (_I64, [_I64, _I64]),
    "fp8blk_quant_act_ue8m0": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "fp8blk_ue8m0_weight_sf": (_I32, [_P, _I64, _I64, _P, _P]),
    "fp8blk_gemm_w8a8_ue8m0": (_I32, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _U32, _P]),
    "fp8blk_gemm_w8a16": (_I32, [_P, _I64, _P, _I64, _P, _I32, _P, _I64, _I64, _I64, _I64, _U32, _P]),
    "fp8blk_gemv_w8a16": (_I32, [_P, _I64, _P, _I64, _P, _I32, _P, _I64, _I64, _I64, _I64, _U32, _P]),
    "fp8blk_quant_weight": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "fp8blk_validate_weights": (_I32, [_P, _I64, _P, _I32, _I64, _I64, _P, _P]),
    "fp8blk_debug_decode_e4m3": (_I32, [_P, _I64, _I32, _P, _P]),
    "fp8blk_debug_group_scale": (_I32, [_P, _I64, _P, _P, _P, _P]),
    "fp8blk_debug_stream_read": (_I32, [_P, _I64, _P, _P]),
    "fp8blk_debug_wait_timeout": (_I32, [_I64, _P]),
    "fp8blk_query_constraints": (_I32, [_P]),
    "fp8blk_status_string": (ctypes.c_char_p, [_I32]),
    "fp8blk_device_error": (_I32, [_P, _I32]),
}


class Constraints(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "abi_version", "scale_block_k", "scale_block_n", "ue8m0_block", "w8a8_tile_m", "w8a8_tile_n",
        "w8a16_tile_n", "w8a16_max_tile_m", "gemv_max_m", "ptr_align_bytes", "row_align_bytes",
        "lds_multiple", "max_split_k")]


class Fp8BlkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = _L().fp8blk_status_string(self.status).decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)} ({msg})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m block_scaled_fp8_bf16_gb300.build` "
            "(or __graft_entry__.build()) first")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


lib = None


def _L():
    """The loaded library (loaded on first use; raises ImportError when it is
    not built, so no call can silently run anything else)."""
    global lib
    if lib is None:
        lib = _load()
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise Fp8BlkError(status, where)


# ---------------------------------------------------------------- marshalling

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ld(t):
    """Row pitch in elements of a 2-D tensor whose last dimension is contiguous."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("last dimension must be contiguous")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def _bytes_tensor(t):
    import torch
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def _out_flags(c, flags):
    """The GEMM output is bf16 or float32; a float32 tensor selects FLAG_OUT_F32."""
    import torch
    _expect(c, (torch.bfloat16, torch.float32), "c")
    return int(flags) | (FLAG_OUT_F32 if c.dtype == torch.float32 else 0)


def _expect(t, dtypes, name):
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")


# ---------------------------------------------------------------- C entry points

def fp8blk_quant_act(x, a, a_scales, stream=None):
    """x [M, K] bf16 -> a [M, K] e4m3 (uint8 view), a_scales [K/128, lds] fp32."""
    import torch
    _expect(x, (torch.bfloat16,), "x")
    a = _bytes_tensor(a)
    M, K = x.shape
    _check(_L().fp8blk_quant_act(_ptr(x), M, K, _ld(x), _ptr(a), _ld(a), _ptr(a_scales), _ld(a_scales),
                                _stream(stream)), "fp8blk_quant_act")


def fp8blk_ue8m0_sf_bytes(rows, K):
    """Bytes of a UE8M0 scale array in the tiled layout (rows padded to 128)."""
    n = _L().fp8blk_ue8m0_sf_bytes(rows, K)
    if n < 0:
        raise ValueError(f"fp8blk_ue8m0_sf_bytes: no tiled scale layout for rows={rows}, K={K}")
    return n


def _sf_buffer(t, rows, K, name):
    import torch
    _expect(t, (torch.uint8,), name)
    if not t.is_contiguous() or t.numel() < fp8blk_ue8m0_sf_bytes(rows, K):
        raise ValueError(f"{name}: a contiguous uint8 buffer of fp8blk_ue8m0_sf_bytes({rows}, {K}) bytes")


def fp8blk_quant_act_ue8m0(x, a, a_sf, stream=None):
    """x [M, K] bf16 -> a [M, K] e4m3 (uint8 view), a_sf: one power-of-two
    exponent byte per token per 32 values, tiled scale layout."""
    import torch
    _expect(x, (torch.bfloat16,), "x")
    a = _bytes_tensor(a)
    M, K = x.shape
    _sf_buffer(a_sf, M, K, "a_sf")
    _check(_L().fp8blk_quant_act_ue8m0(_ptr(x), M, K, _ld(x), _ptr(a), _ld(a), _ptr(a_sf), _stream(stream)),
           "fp8blk_quant_act_ue8m0")


def fp8blk_ue8m0_weight_sf(b_exps, b_sf, stream=None):
    """b_exps [N/32, K/32] uint8 (32x32 block exponents) -> b_sf, per-column
    exponents in the tiled scale layout."""
    import torch
    _expect(b_exps, (torch.uint8,), "b_exps")
    if not b_exps.is_contiguous():
        raise ValueError("b_exps: packed [N/32, K/32]")
    N, K = b_exps.shape[0] * 32, b_exps.shape[1] * 32
    _sf_buffer(b_sf, N, K, "b_sf")
    _check(_L().fp8blk_ue8m0_weight_sf(_ptr(b_exps), N, K, _ptr(b_sf), _stream(stream)), "fp8blk_ue8m0_weight_sf")


def fp8blk_gemm_w8a8_ue8m0(a, a_sf, b, b_sf, c, stream=None, flags=0):
    """C[M, N] (bf16, or float32 when c is float32) = a[M, K] e4m3 x b[N, K] e4m3
    with 1x32 activation and 32x32 weight UE8M0 exponents (both in the tiled
    scale layout), on the tensor cores' block scaling."""
    a, b = _bytes_tensor(a), _bytes_tensor(b)
    M, K = a.shape
    N = b.shape[0]
    _sf_buffer(a_sf, M, K, "a_sf")
    _sf_buffer(b_sf, N, K, "b_sf")
    _check(_L().fp8blk_gemm_w8a8_ue8m0(_ptr(a), _ld(a), _ptr(a_sf), _ptr(b), _ld(b), _ptr(b_sf), _ptr(c), _ld(c),
                                      M, N, K, _out_flags(c, flags), _stream(stream)), "fp8blk_gemm_w8a8_ue8m0")


def fp8blk_gemm_w8a8(a, a_scales, b, b_scales, c, stream=None, flags=0):
    """C[M, N] (bf16, or float32 when c is float32) = block-scaled a[M, K] e4m3 x b[N, K] e4m3."""
    a, b = _bytes_tensor(a), _bytes_tensor(b)
    M, K = a.shape
    N = b.shape[0]
    _check(_L().fp8blk_gemm_w8a8(_ptr(a), _ld(a), _ptr(a_scales), _ld(a_scales), _ptr(b), _ld(b), _ptr(b_scales),
                                _ptr(c), _ld(c), M, N, K, _out_flags(c, flags), _stream(stream)), "fp8blk_gemm_w8a8")


def fp8blk_linear_w8a8(x, b, b_scales, c, stream=None, flags=0):
    """Decode-size (M <= 32) W8A8 linear in one launch: x [M, K] bf16 is quantised
    per token per 128 inside the GEMM kernel; C as fp8blk_gemm_w8a8."""
    import torch
    _expect(x, (torch.bfloat16,), "x")
    b = _bytes_tensor(b)
    M, K = x.shape
    N = b.shape[0]
    _check(_L().fp8blk_linear_w8a8(_ptr(x), _ld(x), _ptr(b), _ld(b), _ptr(b_scales), _ptr(c), _ld(c), M, N, K,
                                  _out_flags(c, flags), _stream(stream)), "fp8blk_linear_w8a8")


def fp8blk_gemm_w8a8_grouped(a, a_scales, b, b_scales, row_group, c, stream=None, flags=0):
    """Grouped (mixture-of-experts) W8A8: row m uses the weights of group
    row_group[m].  b [G, N, K] e4m3 (K contiguous), b_scales [G, N/128, K/128],
    row_group int32 [M] (constant per aligned 128-row block, negative = padding)."""
    import torch
    a, b = _bytes_tensor(a), _bytes_tensor(b)
    _expect(row_group, (torch.int32,), "row_group")
    M, K = a.shape
    G, N, Kb = b.shape
    if Kb != K or b.stride(2) != 1 or b.stride(0) != N * b.stride(1):
        raise ValueError("b must be [G, N, K] with K contiguous and the groups stacked at one row pitch")
    _check(_L().fp8blk_gemm_w8a8_grouped(_ptr(a), _ld(a), _ptr(a_scales), _ld(a_scales), _ptr(b), b.stride(1),
                                        _ptr(b_scales), _ptr(row_group), G, _ptr(c), _ld(c), M, N, K,
                                        _out_flags(c, flags), _stream(stream)), "fp8blk_gemm_w8a8_grouped")


def fp8blk_gemm_w8a16(x, b, b_scales, fmt, c, stream=None, flags=0):
    """C[M, N] bf16 = x[M, K] bf16 x b[N, K] e4m3 with fp32 128x128 or UE8M0 32x32 scales."""
    b = _bytes_tensor(b)
    M, K = x.shape
    N = b.shape[0]
    _check(_L().fp8blk_gemm_w8a16(_ptr(x), _ld(x), _ptr(b), _ld(b), _ptr(b_scales), int(fmt), _ptr(c), _ld(c),
                                 M, N, K, _out_flags(c, flags), _stream(stream)), "fp8blk_gemm_w8a16")


def fp8blk_gemv_w8a16(x, b, b_scales, fmt, c, stream=None, flags=0):
    """Decode-size (M <= 16) form of fp8blk_gemm_w8a16."""
    b = _bytes_tensor(b)
    M, K = x.shape
    N = b.shape[0]
    _check(_L().fp8blk_gemv_w8a16(_ptr(x), _ld(x), _ptr(b), _ld(b), _ptr(b_scales), int(fmt), _ptr(c), _ld(c),
                                 M, N, K, _out_flags(c, flags), _stream(stream)), "fp8blk_gemv_w8a16")


def fp8blk_quant_weight(w, b, b_scales, stream=None):
    """w [N, K] bf16 -> b [N, K] e4m3, b_scales [N/128, K/128] fp32 (packed)."""
    b = _bytes_tensor(b)
    N, K = w.shape
    _check(_L().fp8blk_quant_weight(_ptr(w), N, K, _ld(w), _ptr(b), _ld(b), _ptr(b_scales), _stream(stream)),
           "fp8blk_quant_weight")


def fp8blk_validate_weights(b, b_scales, fmt, dev_counts, stream=None):
    b = _bytes_tensor(b)
    N, K = b.shape
    _check(_L().fp8blk_validate_weights(_ptr(b), _ld(b), _ptr(b_scales), int(fmt), N, K, _ptr(dev_counts),
                                       _stream(stream)), "fp8blk_validate_weights")


def fp8blk_debug_group_scale(amax, s_out, divisor_out, recip_out, stream=None):
    """Runs the quantisers' scale arithmetic on float32 group maxima (device)."""
    _check(_L().fp8blk_debug_group_scale(_ptr(amax), amax.numel(), _ptr(s_out), _ptr(divisor_out), _ptr(recip_out),
                                         _stream(stream)), "fp8blk_debug_group_scale")


def fp8blk_debug_decode_e4m3(codes, exp_shift, out, stream=None):
    _check(_L().fp8blk_debug_decode_e4m3(_ptr(codes), codes.numel(), int(exp_shift), _ptr(out), _stream(stream)),
           "fp8blk_debug_decode_e4m3")


DIAG_TIMEOUT_CODE = 0x4F01   # FP8BLK_DIAG_TIMEOUT_CODE in the header


def fp8blk_debug_stream_read(buf, sink, stream=None):
    """Reads every byte of the contiguous device tensor buf with the plain
    streaming-read kernel and XORs its 32-bit words into sink (a one-element
    int32/uint32 device tensor)."""
    assert buf.is_contiguous(), "fp8blk_debug_stream_read reads a contiguous buffer"
    _check(_L().fp8blk_debug_stream_read(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink), _stream(stream)),
           "fp8blk_debug_stream_read")


def fp8blk_debug_wait_timeout(limit_ns: int, stream=None):
    """Launches the bounded-wait failure check: one warp waits limit_ns on an
    mbarrier nobody completes, then records DIAG_TIMEOUT_CODE in the device
    error word and returns."""
    _check(_L().fp8blk_debug_wait_timeout(int(limit_ns), _stream(stream)), "fp8blk_debug_wait_timeout")


def fp8blk_query_constraints() -> dict:
    c = Constraints()
    _check(_L().fp8blk_query_constraints(ctypes.byref(c)), "fp8blk_query_constraints")
    return {n: getattr(c, n) for n, _ in Constraints._fields_}


def fp8blk_device_error(clear: bool = False) -> int:
    """Raw device error word (0 = none).  Synchronises the device."""
    code = ctypes.c_int32(0)
    st = _L().fp8blk_device_error(ctypes.byref(code), 1 if clear else 0)
    if st not in (0, 8):
        _check(st, "fp8blk_device_error")
    return int(code.value)


# ---------------------------------------------------------------- allocating helpers

def act_scales_pitch(M: int) -> int:
    return (M + 3) // 4 * 4


def quant_act(x, stream=None):
    import torch
    M, K = x.shape
    a = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, act_scales_pitch(M)), dtype=torch.float32, device=x.device)
    fp8blk_quant_act(x, a, s, stream)
    return a, s


def ue8m0_sf_from_rows(e_rows, pad=127):
    """[rows, K/32] exponent bytes -> the flat tiled scale layout (rows padded
    to 128 with `pad`).  Pure indexing; any device."""
    import torch
    rows, G = e_rows.shape
    R = (rows + 127) // 128
    full = torch.full((R * 128, G), pad, dtype=torch.uint8, device=e_rows.device)
    full[:rows] = e_rows
    # row = 128 mb + 32 q + r, slice g = 4 kb + j  ->  [mb][kb][r][q][j]
    return full.view(R, 4, 32, G // 4, 4).permute(0, 3, 2, 1, 4).contiguous().view(-1)


def ue8m0_sf_to_rows(sf, rows, K):
    """The tiled scale layout -> [rows, K/32] exponent bytes (a copy)."""
    R, KB = (rows + 127) // 128, K // 128
    t = sf[:R * KB * 512].view(R, KB, 32, 4, 4).permute(0, 3, 2, 1, 4)   # [mb][q][r][kb][j]
    return t.reshape(R * 128, KB * 4)[:rows].contiguous()


def quant_act_ue8m0(x, stream=None):
    import torch
    M, K = x.shape
    a = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sf = torch.empty(fp8blk_ue8m0_sf_bytes(M, K), dtype=torch.uint8, device=x.device)
    fp8blk_quant_act_ue8m0(x, a, sf, stream)
    return a, sf


def ue8m0_weight_sf(b_exps, stream=None):
    import torch
    N, K = b_exps.shape[0] * 32, b_exps.shape[1] * 32
    sf = torch.empty(fp8blk_ue8m0_sf_bytes(N, K), dtype=torch.uint8, device=b_exps.device)
    fp8blk_ue8m0_weight_sf(b_exps, sf, stream)
    return sf


def gemm_w8a8_ue8m0(a, a_sf, b, b_sf, out=None, stream=None, flags=0, out_dtype=None):
    import torch
    if out is None:
        out = torch.empty((a.shape[0], b.shape[0]), dtype=out_dtype or torch.bfloat16, device=a.device)
    fp8blk_gemm_w8a8_ue8m0(a, a_sf, b, b_sf, out, stream, flags)
    return out


def quant_weight(w, stream=None):
    import torch
    N, K = w.shape
    b = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8blk_quant_weight(w, b, s, stream)
    return b, s


def gemm_w8a8(a, a_scales, b, b_scales, out=None, stream=None, flags=0, out_dtype=None):
    import torch
    if out is None:
        out = torch.empty((a.shape[0], b.shape[0]), dtype=out_dtype or torch.bfloat16, device=a.device)
    fp8blk_gemm_w8a8(a, a_scales, b, b_scales, out, stream, flags)
    return out


def gemm_w8a8_grouped(a, a_scales, b, b_scales, row_group, out=None, stream=None, flags=0, out_dtype=None):
    import torch
    if out is None:
        out = torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype or torch.bfloat16, device=a.device)
    fp8blk_gemm_w8a8_grouped(a, a_scales, b, b_scales, row_group, out, stream, flags)
    return out


def gemm_w8a16(x, b, b_scales, fmt=SCALE_F32_128x128, out=None, stream=None, flags=0, out_dtype=None):
    import torch
    if out is None:
        out = torch.empty((x.shape[0], b.shape[0]), dtype=out_dtype or torch.bfloat16, device=x.device)
    fp8blk_gemm_w8a16(x, b, b_scales, fmt, out, stream, flags)
    return out


def gemv_w8a16(x, b, b_scales, fmt=SCALE_F32_128x128, out=None, stream=None, flags=0, out_dtype=None):
    import torch
    if out is None:
        out = torch.empty((x.shape[0], b.shape[0]), dtype=out_dtype or torch.bfloat16, device=x.device)
    fp8blk_gemv_w8a16(x, b, b_scales, fmt, out, stream, flags)
    return out


def linear_fused_preferred(M: int, N: int, K: int, flags: int = 0) -> bool:
    """Whether the one-launch quantising W8A8 kernel (fp8blk_linear_w8a8) beats
    fp8blk_quant_act + fp8blk_gemm_w8a8 at this shape, from the measured
    CUDA-graph rows of both forms at M = 2..32 on (N, K) = (4096, 4096),
    (7168, 2048), (2048, 7168), (256, 512), with and without programmatic
    dependent launch: one launch wins for small layers (N*K <= 2^21) at every
    M <= 32, for M <= 2, for M <= 4 unless K > 4096 without PDL, and for
    M <= 8 when K <= 4096 (K <= 2048 with PDL); elsewhere the quantiser's
    per-row work inside every weight tile's pipeline costs more than the
    saved launch and round trip."""
    if M < 1 or M > LINEAR_FUSED_MAX_M:
        return False
    pdl = bool(int(flags) & FLAG_PDL)
    if N * K <= 1 << 21 or M <= 2:
        return True
    if M <= 4:
        return pdl or K <= 4096
    return M <= 8 and K <= (2048 if pdl else 4096)


def linear_w8a8(x, b, b_scales, out=None, stream=None, flags=0, out_dtype=None):
    """bf16 x -> per-token quantisation -> W8A8 GEMM: the fused one-launch
    kernel where linear_fused_preferred says it is faster, else quant_act +
    gemm_w8a8 (two launches, an e4m3 copy of x in between)."""
    import torch
    if linear_fused_preferred(x.shape[0], b.shape[0], x.shape[1], flags):
        if out is None:
            out = torch.empty((x.shape[0], b.shape[0]), dtype=out_dtype or torch.bfloat16, device=x.device)
        fp8blk_linear_w8a8(x, b, b_scales, out, stream, flags)
        return out
    a, s = quant_act(x, stream)
    return gemm_w8a8(a, s, b, b_scales, out, stream, flags, out_dtype)


def validate_weights(b, b_scales, fmt=SCALE_F32_128x128, stream=None):
    """(nan_code_count, bad_scale_count); synchronises the stream."""
    import torch
    counts = torch.empty(2, dtype=torch.int32, device=b.device)
    fp8blk_validate_weights(b, b_scales, fmt, counts, stream)
    c = counts.cpu()
    return int(c[0]), int(c[1])
