"""The decode-size W8A8 linear with the activation quantisation inside the
GEMM kernel (the split-K kernel, or the one-token GEMV): bit for bit equal
to fp8blk_quant_act followed by fp8blk_gemm_w8a8 (same codes, same scales,
same accumulation), and within the GEMM tolerance of the float64 oracle of
quantisation + product."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,dtype", [
    (1, 256, 512, torch.bfloat16),
    (16, 256, 512, torch.bfloat16),       # the tiny workload
    (5, 384, 512, torch.bfloat16),        # few rows on the eight-lanes-per-row quantiser path
    (4, 256, 1024, torch.float32),        # the one-warp-per-row quantiser path at its limit
    (32, 384, 1024, torch.bfloat16),
    (7, 4096, 4096, torch.bfloat16),      # K split over a cluster
    (1, 4096, 4096, torch.float32),       # one-token GEMV quantising its token
    (1, 2048, 8320, torch.bfloat16),      # one-token GEMV, a partial third segment
    (29, 1024, 2048, torch.float32),
])
def test_fused_linear_equals_two_step_and_oracle(lib, M, N, K, dtype):
    x = synth.activations(M + N + K, M, K, outliers=True)
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(N + K, N, K))
    xd, bd, bsd = to_dev_bf16(x), to_dev(b), to_dev(Bs)
    c_fused = torch.full((M, N), 7.0, dtype=dtype, device="cuda")
    lib.fp8blk_linear_w8a8(xd, bd, bsd, c_fused)
    a, s = lib.quant_act(xd)
    c_two = torch.full((M, N), 5.0, dtype=dtype, device="cuda")
    lib.fp8blk_gemm_w8a8(a, s, bd, bsd, c_two)
    torch.cuda.synchronize()
    assert lib.fp8blk_device_error() == 0
    assert torch.equal(c_fused, c_two), "fused and two-step results differ"
    a_ref, s_ref = O.quant_act_1x128(x)
    assert_gemm_close(c_fused.double().cpu().numpy(), O.gemm_w8a8(a_ref, s_ref, b, Bs), f"fused {M}x{N}x{K}")


def test_fused_linear_special_rows(lib):
    """A zero row (scale 1, zero codes), a row of one huge value and a row with
    outliers go through the in-kernel quantiser exactly as through quant_act."""
    M, N, K = 3, 256, 256
    x = synth.activations(11, M, K)
    x = x.copy()
    x[0] = 0                                        # +0.0 in bf16
    x[1] = 0
    x[1, 77] = 0x7F00                               # 2^127
    b, Bs = O.quant_weight_128x128(synth.weights_bf16(12, N, K))
    xd, bd, bsd = to_dev_bf16(x), to_dev(b), to_dev(Bs)
    c_fused = lib.linear_w8a8(xd, bd, bsd)
    a, s = lib.quant_act(xd)
    c_two = lib.gemm_w8a8(a, s, bd, bsd)
    torch.cuda.synchronize()
    assert torch.equal(c_fused, c_two)
    assert lib.fp8blk_device_error() == 0
