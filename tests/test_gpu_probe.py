"""The read-only streaming probe (gqa_stream_read), through the C ABI: every
byte of the buffer is read once, so the XOR of its 32-bit words must equal
the host's."""
import numpy as np
import pytest
import torch

import grouped_query_decode_kv_b300 as gqa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    torch.cuda.set_device(0)
    gqa.load_library()
    yield


@pytest.mark.parametrize("mode,nbytes", [(0, 16), (0, 4096 + 48), (0, 37 << 20), (1, 32768), (1, 77 * 32768),
                                         (1, 1 << 26)])
def test_stream_read_checksum(mode, nbytes):
    g = torch.Generator().manual_seed(12000 + nbytes + mode)
    host = torch.randint(-2 ** 31, 2 ** 31 - 1, (nbytes // 4,), generator=g, dtype=torch.int64).to(torch.int32)
    buf = host.cuda()
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    gqa.gqa_stream_read(buf, mode, sink)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(host.numpy().view(np.uint32))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)
    assert gqa.gqa_get_device_error() == 0


def test_stream_read_rejects_bad_sizes():
    buf = torch.zeros(1000, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gqa.GQAError):
        gqa.gqa_stream_read(buf, 1, sink)  # not a multiple of 32 KB
    with pytest.raises(gqa.GQAError):
        gqa.gqa_stream_read(buf, 2, sink)  # no such mode
