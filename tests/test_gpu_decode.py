"""GPU parity of the decode-size W8A16 kernel (M <= 32) against the float64
oracle, over the work splits it chooses (split-K clusters of 1..8 CTAs,
one or several tiles per cluster, uneven K ranges, scale windows longer
than 32 K blocks), and of programmatic dependent launch (FP8BLK_FLAG_PDL):
chained calls must read their inputs only after the previous kernel wrote
them, and write their output only after the previous kernel read it."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, bf16_out_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def bits_of(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def weights(fmt, seed, N, K):
    if fmt == 0:
        return O.quant_weight_128x128(synth.weights_bf16(seed, N, K))
    return synth.ue8m0_weights(seed, N, K)


def ref_w8a16(fmt, x, b, sc):
    return O.gemm_w8a16_f32scale(x, b, sc) if fmt == 0 else O.gemm_w8a16_ue8m0(x, b, sc)


# (M, N, K): comments give the work split the kernel picks on 152 SMs.
@pytest.mark.parametrize("M,N,K", [
    (3, 28672, 4096),    # clusters of 2, three tiles per cluster (per-tile cluster reductions)
    (4, 28672, 1024),    # clusters of 2, three tiles per cluster, 4 K blocks per CTA
    (7, 16384, 2048),    # no split: one tile per CTA
    (24, 19968, 1152),   # token tile 32, clusters of 2 with 4 and 5 K blocks, several tiles each
    (32, 8192, 1024),    # token tile 32, clusters of 2
    (3, 19456, 5120),    # no split, 40 K blocks per CTA: scale windows reloaded after 32 blocks
    (13, 128, 8192),     # one tile, clusters of 8
])
@pytest.mark.parametrize("fmt", [0, 1])
def test_decode_splits(lib, M, N, K, fmt):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    x = synth.activations(M * 7 + N + K, M, K, outliers=True)
    b, sc = weights(fmt, N + 3 * K + fmt, N, K)
    c = torch.full((M, N + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    fp8blk.fp8blk_gemm_w8a16(to_dev_bf16(x), to_dev(b), to_dev(sc), fmt, c[:, :N])
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    out = bf16_out_to_f64(c)
    assert np.all(out[:, N:] == 7.0)          # nothing written past N
    assert_gemm_close(out[:, :N], ref_w8a16(fmt, x, b, sc), f"decode fmt{fmt} {M}x{N}x{K}")


def test_decode_repeatable(lib):
    """The split-K sums run in rank order: repeated calls give identical bits."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, N, K = 5, 4096, 14336
    x = to_dev_bf16(synth.activations(3, M, K))
    b, sc = weights(0, 4, N, K)
    b, sc = to_dev(b), to_dev(sc)
    outs = [fp8blk.gemm_w8a16(x, b, sc, 0) for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("M", [1, 4])      # CUDA-core GEMV for the first product, decode-size kernel
@pytest.mark.parametrize("fmt", [0, 1])
def test_pdl_chain_reads_previous_output(lib, fmt, M):
    """c1 = x W1, c2 = c1 W2, c1 = x' W1 again, all with FP8BLK_FLAG_PDL on one
    stream, repeated: every c2 must be the product of the c1 written just
    before it, and the later write of c1 must not reach the c2 that reads it."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    N1, K1, N2 = 8192, 4096, 2048
    x = [synth.activations(10 + i, M, K1) for i in range(2)]
    b1, s1 = weights(fmt, 20, N1, K1)
    b2, s2 = weights(fmt, 21, N2, N1)
    xd = [to_dev_bf16(v) for v in x]
    b1d, s1d, b2d, s2d = to_dev(b1), to_dev(s1), to_dev(b2), to_dev(s2)
    c1 = torch.full((M, N1), 7.0, dtype=torch.bfloat16, device="cuda")
    rounds = 6
    c2 = [torch.full((M, N2), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(rounds)]
    f = fp8blk.FLAG_PDL
    for r in range(rounds):
        fp8blk.fp8blk_gemm_w8a16(xd[r % 2], b1d, s1d, fmt, c1, flags=f)
        fp8blk.fp8blk_gemm_w8a16(c1, b2d, s2d, fmt, c2[r], flags=f)
    fp8blk.fp8blk_gemm_w8a16(xd[0], b1d, s1d, fmt, c1, flags=f)
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    c1_ref = [ref_w8a16(fmt, x[i], b1, s1) for i in range(2)]
    assert_gemm_close(bf16_out_to_f64(c1), c1_ref[0], "pdl c1")
    # Each c2 is checked against the c1 its round wrote (recomputed on the
    # GPU without the flag, so both sides start from the same bf16 bits).
    for i in range(2):
        c1_bits = fp8blk.gemm_w8a16(xd[i], b1d, s1d, fmt)
        torch.cuda.synchronize()
        ref = ref_w8a16(fmt, bits_of(c1_bits), b2, s2)
        for r in range(i, rounds, 2):
            assert_gemm_close(bf16_out_to_f64(c2[r]), ref, f"pdl c2 round {r}")


def test_pdl_w8a8_after_quant(lib):
    """quant_act lets the next kernel start early; a GEMM launched with
    FP8BLK_FLAG_PDL must still read the codes and scales it writes."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    M, N, K = 2048, 1024, 4096
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(5, N, K))
    bd, bsd = to_dev(b), to_dev(Bs)
    xs = [synth.activations(30 + i, M, K) for i in range(2)]
    xd = [to_dev_bf16(v) for v in xs]
    a = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    lds = fp8blk.act_scales_pitch(M)
    s = torch.empty((K // 128, lds), dtype=torch.float32, device="cuda")
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    for r in range(4):
        fp8blk.fp8blk_quant_act(xd[r % 2], a, s)
        fp8blk.fp8blk_gemm_w8a8(a, s, bd, bsd, outs[r], flags=fp8blk.FLAG_PDL)
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    rows = synth.sample_rows(7, M, 24)
    for i in range(2):
        a_ref, as_ref = O.quant_act_1x128(xs[i][rows])
        ref = O.gemm_w8a8(a_ref, as_ref, b, Bs)
        for r in range(i, 4, 2):
            assert_gemm_close(bf16_out_to_f64(outs[r])[rows], ref, f"pdl w8a8 round {r}")


@pytest.mark.parametrize("M", [1, 3])      # one-token GEMV, split-K kernel
def test_pdl_w8a8_decode_size(lib, M):
    """Decode-size W8A8 with the flag, after quant_act, alternating two token
    batches so that each product must read the codes written just before it;
    the fused linear with the flag as well."""
    import block_scaled_fp8_bf16_gb300 as fp8blk
    N, K = 4096, 4096
    xs = [synth.activations(40 + i, M, K) for i in range(2)]
    xd = [to_dev_bf16(v) for v in xs]
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(41, N, K))
    bd, bsd = to_dev(b), to_dev(Bs)
    a = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((K // 128, fp8blk.act_scales_pitch(M)), dtype=torch.float32, device="cuda")
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    lins = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    for r in range(4):
        fp8blk.fp8blk_quant_act(xd[r % 2], a, s)
        fp8blk.fp8blk_gemm_w8a8(a, s, bd, bsd, outs[r], flags=fp8blk.FLAG_PDL)
        fp8blk.fp8blk_linear_w8a8(xd[r % 2], bd, bsd, lins[r], flags=fp8blk.FLAG_PDL)
    torch.cuda.synchronize()
    assert fp8blk.fp8blk_device_error() == 0
    for i in range(2):
        a_ref, as_ref = O.quant_act_1x128(xs[i])
        ref = O.gemm_w8a8(a_ref, as_ref, b, Bs)
        for r in range(i, 4, 2):
            assert_gemm_close(bf16_out_to_f64(outs[r]), ref, f"pdl w8a8 decode round {r}")
            assert torch.equal(outs[r], lins[r]), f"pdl linear round {r}"
