"""The streaming-read diagnostic reads every byte it is given: the XOR of all
32-bit words it reports equals the host's, on sizes with a ragged tail of the
grid-stride loop, and an initial sink value is kept (XORed into)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("words16", [1, 7, 4096 * 608 * 8 + 5, 3_000_017])
def test_stream_read_xor_of_every_word(lib, words16):
    import block_scaled_fp8_bf16_gb300 as fp8blk
    rng = np.random.default_rng(words16)
    host = rng.integers(0, 2**32, size=words16 * 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    sink = torch.tensor([0x5A5A5A5A], dtype=torch.int32, device="cuda")
    fp8blk.fp8blk_debug_stream_read(buf, sink)
    torch.cuda.synchronize()
    expect = np.bitwise_xor.reduce(host) ^ np.uint32(0x5A5A5A5A)
    assert np.uint32(sink.cpu().numpy().view(np.uint32)[0]) == expect
