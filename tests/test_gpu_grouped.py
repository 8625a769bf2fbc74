"""GPU parity of the grouped (mixture-of-experts) W8A8 product against the
float64 oracle: every non-padding row within the GEMM tolerance, padding
blocks untouched, an out-of-range group skipped and reported."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import assert_gemm_close, to_dev

pytestmark = pytest.mark.gpu


def grouped_inputs(seed, tiles_per_group, N, K, pad_tiles=()):
    """Rows for each group in whole 128-row tiles; pad_tiles are tile indices
    (in the final order) marked as padding (-1)."""
    G = len(tiles_per_group)
    groups = []
    for e, t in enumerate(tiles_per_group):
        groups += [e] * t
    for p in sorted(pad_tiles):
        groups.insert(p, -1)
    row_group = np.repeat(np.array(groups, dtype=np.int32), 128)
    M = row_group.size
    x = synth.activations(seed, M, K, outliers=True)
    a, As = O.quant_act_1x128(x)
    bs, Bss = [], []
    for e in range(G):
        b, Bs = O.quant_weight_128x128(synth.weights_bf16(seed * 31 + e, N, K))
        bs.append(b)
        Bss.append(Bs)
    return a, As, np.stack(bs), np.stack(Bss), row_group


def run_grouped(lib, a, As, b, Bs, row_group, dtype=torch.bfloat16):
    M, K = a.shape
    lds = lib.act_scales_pitch(M)
    s = np.zeros((K // 128, lds), dtype=np.float32)
    s[:, :M] = As
    c = torch.full((M, b.shape[1]), 7.0, dtype=dtype, device="cuda")
    lib.fp8blk_gemm_w8a8_grouped(to_dev(a), to_dev(s), to_dev(b), to_dev(Bs), to_dev(row_group), c)
    torch.cuda.synchronize()
    return c.double().cpu().numpy()


@pytest.mark.parametrize("tiles,N,K,pads,dtype", [
    ((2, 1, 3), 256, 512, (), torch.bfloat16),
    ((1, 0, 2, 1), 384, 1024, (1, 5), torch.bfloat16),     # an empty group and two padding tiles
    ((3, 2), 512, 256, (2,), torch.float32),                # float32 output
    ((1,), 128, 128, (), torch.bfloat16),                   # one group, one tile, one K block
    ((6, 5, 7, 4, 8, 2, 3, 5), 1024, 1024, (9, 20), torch.bfloat16),   # more tiles than one wave
    # CTA-pair path (enough 256 x 256 tiles): groups not aligned to 256 rows,
    # so many pair tiles hold two groups (two passes), padding halves, and
    # one group of 256-row multiples
    ((3, 4, 1, 6, 2), 2048, 512, (0, 7), torch.float32),
    ((4, 2, 6), 4096, 384, (), torch.bfloat16),
    ((1, 3, 2, 5, 1, 4), 2048, 1024, (1, 12), torch.bfloat16),
    # 96 pair tiles on 76 pairs: the first passes' last round runs as 256 x 128
    # halves, and groups of 384 and 640 rows give pair tiles a second pass
    ((3, 4, 5), 4096, 256, (), torch.bfloat16),
])
def test_grouped_matches_oracle(lib, tiles, N, K, pads, dtype):
    a, As, b, Bs, g = grouped_inputs(sum(tiles) + N + K, tiles, N, K, pads)
    lib.fp8blk_device_error(clear=True)
    out = run_grouped(lib, a, As, b, Bs, g, dtype)
    assert lib.fp8blk_device_error() == 0
    ref = O.gemm_w8a8_grouped(a, As, b, Bs, g)
    real = g >= 0
    assert_gemm_close(out[real], ref[real], f"grouped {tiles} N={N} K={K}")
    assert np.all(out[~real] == 7.0)


@pytest.mark.parametrize("tiles,N,bad", [
    ((1, 2), 256, 1),        # single-CTA path
    ((5, 6), 2048, 3),       # CTA-pair path: the second half of a pair tile
    ((5, 6), 2048, 4),       # CTA-pair path: the first half of a pair tile
])
def test_grouped_out_of_range_group_is_skipped_and_reported(lib, tiles, N, bad):
    a, As, b, Bs, g = grouped_inputs(3, tiles, N, 256)
    g = g.copy()
    r0 = 128 * bad
    g[r0:r0 + 128] = 5                              # this tile names a group past the expert weights
    lib.fp8blk_device_error(clear=True)
    out = run_grouped(lib, a, As, b, Bs, g)
    code = lib.fp8blk_device_error(clear=True)
    assert code == 0x100 | 11
    good = np.ones(g.size, dtype=bool)
    good[r0:r0 + 128] = False
    ref = O.gemm_w8a8_grouped(a, As, b, Bs, np.where(good, g, -1))
    assert_gemm_close(out[good], ref[good], "grouped with a bad tile")
    assert np.all(out[~good] == 7.0)
    assert lib.fp8blk_device_error() == 0
