"""GPU parity of the CUDA-core W8A16 GEMV (M = 1, K >= 4096, at most 2^25
weight codes) against the float64 oracle: whole and partial 4096-code
segments and 512-code passes, fewer rows than SMs, several rows per warp,
padded pitches, both scale formats, the exact e4m3 decode, and the
hand-over to the decode-size tensor-core kernel outside that window."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, bf16_out_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def weights(fmt, seed, N, K):
    if fmt == 0:
        return O.quant_weight_128x128(synth.weights_bf16(seed, N, K))
    return synth.ue8m0_weights(seed, N, K)


def ref_w8a16(fmt, x, b, sc):
    return O.gemm_w8a16_f32scale(x, b, sc) if fmt == 0 else O.gemm_w8a16_ue8m0(x, b, sc)


def run(x, b, sc, fmt, ldx_pad=0, ldc_pad=0, gemv=False):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, K = x.shape
    N = b.shape[0]
    xf = np.zeros((M, K + ldx_pad), dtype=np.uint16)
    xf[:, :K] = x
    c = torch.full((M, N + ldc_pad), 7.0, dtype=torch.bfloat16, device="cuda")
    fn = fp8blk.fp8blk_gemv_w8a16 if gemv else fp8blk.fp8blk_gemm_w8a16
    fn(to_dev_bf16(xf)[:, :K], to_dev(b), to_dev(sc), fmt, c[:, :N])
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    out = bf16_out_to_f64(c)
    assert np.all(out[:, N:] == 7.0)          # nothing written past N
    return out[:, :N]


@pytest.mark.parametrize("M,N,K", [
    (1, 128, 4096),      # fewer rows than SMs: one row per CTA
    (1, 384, 4224),      # a whole segment and a one-pass segment
    (1, 2048, 14336),    # three whole segments and a half segment
    (1, 3712, 4608),     # one row per warp on most CTAs; a segment and a pass
    (1, 8192, 4096),     # several rows per warp
])
@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_matches_oracle(lib, M, N, K, fmt):
    x = synth.activations(M * 11 + N + K, M, K, outliers=True)
    b, sc = weights(fmt, N + 5 * K + fmt, N, K)
    out = run(x, b, sc, fmt, ldx_pad=8, ldc_pad=8, gemv=fmt == 1)
    assert_gemm_close(out, ref_w8a16(fmt, x, b, sc), f"gemv fmt{fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_gemv_exact_decode_of_every_code(lib, fmt):
    """x = one-hot at column k0 reads one weight column: every finite code
    must come back exactly times its power-of-two scale (float32 output, no
    rounding anywhere)."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    N, K = 256, 4096
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    b = synth.finite_e4m3_codes(7, (N, K))
    k0 = 777
    b[:254, k0] = finite
    b[254:, k0] = 0
    if fmt == 0:
        sc = np.exp2(np.random.default_rng(3).integers(-14, 8, size=(N // 128, K // 128))).astype(np.float32)
    else:
        sc = synth.ue8m0_scale_bytes(5, (N // 32, K // 32))
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, k0] = 0x3F80
    c = torch.full((1, N), 7.0, dtype=torch.float32, device="cuda")
    fp8blk.fp8blk_gemm_w8a16(to_dev_bf16(x), to_dev(b), to_dev(sc), fmt, c)
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy().astype(np.float64), ref_w8a16(fmt, x, b, sc))


def test_gemv_hands_over_outside_its_window(lib):
    """K = 25216 leaves too little shared memory next to the f32 token for
    two 4 KB slots per warp, K = 2048 is below a segment and N x K = 2^25 +
    4096 x 128 is past the weight-set limit: those calls run on the
    decode-size kernel.  K = 25088 still runs on the GEMV.  All stay correct."""
    for N, K in ((256, 25088), (256, 25216), (512, 2048), (8192 + 128, 4096)):
        x = synth.activations(K + N, 1, K)
        b, sc = weights(0, K, N, K)
        out = run(x, b, sc, 0)
        assert_gemm_close(out, ref_w8a16(0, x, b, sc), f"gemv window N={N} K={K}")


def test_gemv_zero_tokens_and_zero_rows(lib):
    """Zero activations give exact zeros; rows of zero codes give zeros."""
    N, K = 512, 4096
    b, sc = weights(0, 9, N, K)
    b[100:228] = 0
    out = run(np.zeros((1, K), dtype=np.uint16), b, sc, 0)
    assert np.all(out == 0)
    x = synth.activations(2, 1, K)
    out = run(x, b, sc, 0)
    assert np.all(out[0, 100:228] == 0)
    assert_gemm_close(out, ref_w8a16(0, x, b, sc), "gemv zeros")
