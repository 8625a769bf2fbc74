"""Every GEMM path gives bit-identical float32 output when run again on the
same inputs.  The accumulation order is fixed by design: two MMA issuers
take turns where K blocks share an accumulator, and split-K partials are
summed in a fixed order, so a run-to-run difference in any bit would mean an
ordering race (the parity tests only bound the error)."""
import pytest
import torch

import block_scaled_fp8_bf16_gb300 as fp8blk
from synth import torch_gen as tg

pytestmark = pytest.mark.gpu

RUNS = 3


def _same_every_run(call, out):
    results = []
    for _ in range(RUNS):
        out.fill_(7.0)
        call()
        torch.cuda.synchronize()
        assert fp8blk.fp8blk_device_error() == 0
        results.append(out.clone())
    for r in results[1:]:
        assert torch.equal(r, results[0])


@pytest.mark.parametrize("M,N,K", [
    (1024, 4096, 2048),    # CTA pairs, whole tiles
    (2304, 2304, 512),     # CTA pairs, last round in halves
    (256, 7168, 1024),     # CTA pairs, every tile as two halves
    (256, 4992, 12288),    # CTA pairs, K split over two pairs
    (300, 1024, 1024),     # single CTA, persistent, two issuers
    (16, 4096, 4096),      # single CTA, K split over a cluster
])
def test_w8a8_deterministic(lib, M, N, K):
    a, s = fp8blk.quant_act(tg.activations(M + N + K, M, K))
    b, bs = fp8blk.quant_weight(tg.weights_bf16(M + N + K, N, K))
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    _same_every_run(lambda: fp8blk.fp8blk_gemm_w8a8(a, s, b, bs, c), c)


@pytest.mark.parametrize("groups,rows,N,K", [
    (4, 512, 2048, 1024),  # CTA pairs (groups of at least 256 rows)
    (8, 128, 1024, 1024),  # single CTA (128-row groups)
    (4, 384, 4096, 512),   # CTA pairs: halves in the last round, second passes for tiles holding two groups
])
def test_w8a8_grouped_deterministic(lib, groups, rows, N, K):
    M = groups * rows
    a, s = fp8blk.quant_act(tg.activations(groups + N, M, K))
    ws = [fp8blk.quant_weight(tg.weights_bf16(groups + e, N, K)) for e in range(groups)]
    b = torch.stack([w[0] for w in ws])
    bs = torch.stack([w[1] for w in ws])
    rg = torch.arange(groups, dtype=torch.int32, device="cuda").repeat_interleave(rows)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    _same_every_run(lambda: fp8blk.fp8blk_gemm_w8a8_grouped(a, s, b, bs, rg, c), c)


@pytest.mark.parametrize("M,N,K", [
    (1024, 4864, 1024),    # CTA pairs, two issuers taking turns
    (300, 2048, 2048),     # single CTA, persistent, two issuers taking turns
    (128, 2048, 7168),     # single CTA, K split over a cluster of 8
])
def test_w8a8_ue8m0_deterministic(lib, M, N, K):
    a, sf = fp8blk.quant_act_ue8m0(tg.activations(M + K, M, K))
    b, eb = tg.ue8m0_weights(N + K, N, K)
    bsf = fp8blk.ue8m0_weight_sf(eb)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    _same_every_run(lambda: fp8blk.fp8blk_gemm_w8a8_ue8m0(a, sf, b, bsf, c), c)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("M,N,K", [
    (1024, 2048, 2048),    # 128-token tiles, two issuers (taking turns for UE8M0)
    (64, 2048, 4096),      # 64-token tiles
    (128, 2048, 7168),     # K split over a cluster
    (1024, 7168, 1024),    # 256-token tiles for UE8M0, two issuers taking turns
    (4096, 7168, 2048),    # 256-token tiles over six rounds of the SMs (a release race showed in the last rounds)
])
def test_w8a16_deterministic(lib, M, N, K, fmt):
    x = tg.activations(M + N, M, K)
    if fmt == 0:
        b, bs = fp8blk.quant_weight(tg.weights_bf16(N + K, N, K))
    else:
        b, bs = tg.ue8m0_weights(N + K, N, K)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    _same_every_run(lambda: fp8blk.fp8blk_gemm_w8a16(x, b, bs, fmt, c), c)
