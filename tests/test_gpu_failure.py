"""Failure detection without a GPU fault: a wait that nothing completes runs
out its (short) limit inside a kernel, the kernel records the timeout in the
device error word and returns, the host reads FP8BLK_ERR_TIMEOUT, and the
CUDA context stays usable for the next GEMM."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    import oracle
    import synth
    from helpers import assert_gemm_close

    fp8blk.fp8blk_device_error(clear=True)
    assert fp8blk.fp8blk_device_error() == 0

    fp8blk.fp8blk_debug_wait_timeout(2_000_000)   # 2 ms of waiting on a barrier nobody arrives on
    torch.cuda.synchronize()
    code = fp8blk.fp8blk_device_error()
    assert code == fp8blk.DIAG_TIMEOUT_CODE
    assert fp8blk.fp8blk_device_error(clear=True) == fp8blk.DIAG_TIMEOUT_CODE
    assert fp8blk.fp8blk_device_error() == 0

    # The context is intact: a W8A8 linear still matches the oracle.
    M, N, K = 16, 256, 512
    x = synth.activations(0, M, K)
    w = synth.weights_bf16(0, N, K)
    b, bs = oracle.quant_weight_128x128(w)
    dev = torch.device("cuda")
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    a, s = fp8blk.quant_act(xt)
    c = fp8blk.gemm_w8a8(a, s, torch.from_numpy(b).to(dev), torch.from_numpy(bs).to(dev))
    torch.cuda.synchronize()
    a_ref, s_ref = oracle.quant_act_1x128(x)
    ref = oracle.gemm_w8a8(a_ref, s_ref, b, bs)
    assert_gemm_close(c.float().cpu().numpy().astype(np.float64), ref, "W8A8 after a forced timeout")
    assert fp8blk.fp8blk_device_error() == 0


def test_timeout_on_a_non_blocking_stream_is_seen_without_a_sync():
    """The timeout kernel runs on a non-blocking stream (which the legacy
    default stream does not wait for); fp8blk_device_error must still see
    the code without any synchronisation by the caller."""
    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    fp8blk.fp8blk_device_error(clear=True)
    side = torch.cuda.Stream()
    fp8blk.fp8blk_debug_wait_timeout(20_000_000, side)   # 20 ms: still waiting when the read is issued
    assert fp8blk.fp8blk_device_error(clear=True) == fp8blk.DIAG_TIMEOUT_CODE
    assert fp8blk.fp8blk_device_error() == 0


def test_timeout_status_maps_to_err_timeout():
    import ctypes

    import torch

    import block_scaled_fp8_bf16_gb300 as fp8blk
    fp8blk.fp8blk_device_error(clear=True)
    fp8blk.fp8blk_debug_wait_timeout(1_000_000)
    torch.cuda.synchronize()
    raw = ctypes.c_int32(0)
    st = fp8blk._L().fp8blk_device_error(ctypes.byref(raw), 1)
    assert st == 8 and raw.value == fp8blk.DIAG_TIMEOUT_CODE   # FP8BLK_ERR_TIMEOUT, then cleared
    assert fp8blk.fp8blk_device_error() == 0
