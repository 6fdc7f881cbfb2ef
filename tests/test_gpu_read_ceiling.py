"""The benchmark's plain-read ceiling kernel (ceiling/read.cu) reads every byte:
its XOR checksum over all 32-bit words matches the host's, for every grid shape
the benchmark tries, on buffers with a ragged last chunk."""
import numpy as np
import pytest

from gpu_util import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4608 * 3 + 16, 20643840, 50135040 + 16 * 7])
def test_checksum_covers_every_word(nbytes):
    import ceiling
    t = torch()
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint32)
    buf = t.from_numpy(host.view(np.uint8)).cuda()
    want = int(np.bitwise_xor.reduce(host))
    sms = t.cuda.get_device_properties(0).multi_processor_count
    for cfg in ceiling.CONFIGS:
        sink = t.zeros(2, dtype=t.int32, device="cuda")
        ceiling.read(buf, sink, cfg, sms)
        t.cuda.synchronize()
        got = sink.cpu().numpy().view(np.uint32)
        assert got[1] == 0, f"{cfg}: a wait gave up"
        assert int(got[0]) == want, f"{cfg}: checksum {got[0]:#x} != {want:#x}"
