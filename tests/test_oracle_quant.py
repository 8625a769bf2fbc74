"""Pins of the oracle's quantisers.

The oracle quantises with its own grid search and a float64-emulated float32
quotient.  These tests compare it with an independent route (torch CPU float32
division, which is IEEE, and torch's nearest-even float8_e4m3fn cast) and with
error bounds that hold for any correct quantiser.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth


def _torch_quant_groups(x_bits_groups):
    """Reference route for rows of 128 bf16 values: amax, s = amax / 448 in
    float32, q = cast(x / s) to float8_e4m3fn (in range, so no saturation)."""
    x = torch.from_numpy(x_bits_groups.astype(np.int32).astype(np.int16)).view(torch.bfloat16).float()
    amax = x.abs().amax(dim=-1)
    s = amax / 448.0
    s = torch.where(amax == 0, torch.ones_like(s), s)
    q = (x / s[..., None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.numpy(), s.numpy()


def _groups_with_amax(amax_bits, rng):
    """All finite bf16 values with |v| <= amax, shuffled into groups of 127,
    each completed with +-amax (so every group's amax is amax)."""
    allb = np.arange(65536, dtype=np.uint16)
    v = O.bf16_bits_to_f64(allb)
    a = O.bf16_bits_to_f64(np.array([amax_bits], dtype=np.uint16))[0]
    pool = allb[np.isfinite(v) & (np.abs(v) <= a)]
    pool = rng.permutation(pool)
    n = (len(pool) + 126) // 127
    pool = np.resize(pool, n * 127).reshape(n, 127)
    sign = rng.integers(0, 2, size=(n, 1)).astype(np.uint16) << 15
    col = (np.uint16(amax_bits) | sign).astype(np.uint16)
    g = np.concatenate([pool, col], axis=1)
    # put the amax element at a random position of each group
    idx = rng.permuted(np.tile(np.arange(128), (n, 1)), axis=1)
    return np.take_along_axis(g, idx, axis=1)


AMAX_CASES = {
    "one": 0x3F80,            # 1.0
    "e4m3max": 0x43E0,        # 448
    "odd": 0x40F0,            # 7.5
    "bf16max": 0x7F7F,        # largest finite bf16
    "tiny_normal": 0x0080,    # 2^-126
    "denormal": 0x0003,       # 3 * 2^-133
}


@pytest.mark.parametrize("name", list(AMAX_CASES))
def test_quant_act_exhaustive_bf16_against_torch(name):
    rng = np.random.default_rng(11)
    g = _groups_with_amax(AMAX_CASES[name], rng)
    x = g.reshape(-1, 128)
    q, s = O.quant_act_1x128(x)                  # one group per row here
    qt, st = _torch_quant_groups(x)
    assert np.array_equal(s[0].view(np.uint32), st.view(np.uint32))
    assert np.array_equal(q, qt)


def test_quant_act_error_bound_and_amax_code():
    x = synth.activations(0, 64, 1024, outliers=True)
    q, s = O.quant_act_1x128(x)
    xv = O.bf16_bits_to_f64(x).reshape(64, 8, 128)
    dq = O.e4m3_decode(q).reshape(64, 8, 128) * s.T[:, :, None]
    sc = s.T[:, :, None].astype(np.float64)
    # half an e4m3 ulp: 2^-4 relative in the normal range, 2^-10 absolute
    # (times s) in the subnormal range, plus float32 quotient rounding.
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 2.0 ** -20)
    assert np.all(np.abs(dq - xv) <= bound)
    # the element that sets amax lands on +-448 (or the neighbouring code)
    amax_pos = np.argmax(np.abs(xv), axis=-1)
    qa = np.take_along_axis(q.reshape(64, 8, 128), amax_pos[..., None], axis=-1)
    assert np.all(np.isin(qa & 0x7F, [0x7E, 0x7D]))


def test_quant_act_scale_layout_is_m_contiguous():
    """Scales come out [K/128, M]: the scale of row m, group g sits at [g, m]."""
    M, K = 5, 384
    x = synth.activations(1, M, K)
    q, s = O.quant_act_1x128(x)
    assert s.shape == (K // 128, M) and s.dtype == np.float32
    for m in range(M):
        for g in range(K // 128):
            grp = O.bf16_bits_to_f64(x[m, g * 128:(g + 1) * 128])
            amax = np.max(np.abs(grp))
            assert s[g, m] == np.float32(np.float64(np.float32(amax)) / 448.0)


def test_quant_act_zero_group():
    x = np.zeros((2, 256), dtype=np.uint16)
    x[1, :128] = 0x8000                          # -0.0
    x[1, 128] = 0x3F80                            # 1.0 in the second group
    q, s = O.quant_act_1x128(x)
    assert s[0, 0] == 1.0 and s[1, 0] == 1.0 and s[0, 1] == 1.0
    assert np.all(q[0] == 0)
    assert np.all(q[1, :128] == 0x80)            # sign of zero kept
    assert q[1, 128] == 0x7E and np.all(q[1, 129:] == 0)


def test_quant_weight_blocks_against_torch():
    N, K = 256, 384
    w = synth.weights_bf16(0, N, K)
    q, s = O.quant_weight_128x128(w)
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].reshape(1, -1)
            qt, st = _torch_quant_groups(blk)
            assert s[nb, kb] == st[0]
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].reshape(-1), qt[0])


def test_quant_weight_block_independence():
    """Changing one block changes only that block's codes and scale."""
    w = synth.weights_bf16(2, 256, 256)
    q0, s0 = O.quant_weight_128x128(w)
    w2 = w.copy()
    w2[130, 5] = 0x4400                         # 512.0 in block (1, 0)
    q1, s1 = O.quant_weight_128x128(w2)
    assert s1[1, 0] != s0[1, 0]
    assert s1[0, 0] == s0[0, 0] and s1[0, 1] == s0[0, 1] and s1[1, 1] == s0[1, 1]
    mask = np.zeros_like(q0, dtype=bool)
    mask[128:, :128] = True
    assert np.array_equal(q0[~mask], q1[~mask])
