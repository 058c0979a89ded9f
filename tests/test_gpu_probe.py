"""The read-only streaming probe loads every word once: its sink equals the
XOR of all 8-byte words of the buffer, computed on the host.  Marked gpu."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_w4a4_decode_gb300 as nvmod
    from nvfp4_w4a4_decode_gb300 import build as nvbuild
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nvbuild.build()
    nvmod.library()
    return nvmod


# one word; a ragged count of words; more words than one pass of the grid
# (several iterations of the four-load loop plus the one-load tail)
@pytest.mark.parametrize("nbytes", [16, 4096 + 16, (1 << 20) + 48, (64 << 20) + 16 * 999])
def test_probe_sink_is_xor_of_all_words(nv, nbytes):
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2**63, size=nbytes // 8, dtype=np.int64).view(np.uint64)
    buf = torch.from_numpy(host.view(np.int64)).cuda()
    sink = nv.read_probe(buf)
    torch.cuda.synchronize()
    got = int(sink.cpu().numpy().view(np.uint64)[0])
    assert got == int(np.bitwise_xor.reduce(host))


def test_probe_empty_and_reused_sink(nv):
    sink = torch.full((1,), 12345, dtype=torch.int64, device="cuda")
    st = nv.library().nvfp4_read_probe(None, 0, sink.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(sink.item()) == 0
    buf = torch.arange(64, dtype=torch.int64, device="cuda")
    nv.read_probe(buf, sink=sink)
    nv.read_probe(buf, sink=sink)      # zeroed first each time: not XORed twice
    torch.cuda.synchronize()
    assert int(sink.item()) == int(np.bitwise_xor.reduce(np.arange(64)))
