"""The streaming-read probe reads every 16-byte vector of its buffer exactly
once, whichever loader and span layout it uses (needs a GB300).

In its xor mode each lane folds the words it reads into one word, and a
vector past the end reads as four equal words (which cancel).  So the xor of
all the lanes' results is the xor of every word of the buffer (the probe
keeps the low 30 bits of each result), a value the host computes alone: a
vector missed or read twice changes it."""
import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def D():
    import draft_tree_construction_gb300 as D
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D.build()
    return D


@pytest.mark.parametrize("mode,ctas,warps,stages", [
    (0, 5, 8, 0),      # direct loads, contiguous spans
    (1, 5, 12, 3),     # bulk ring, contiguous spans
    (5, 5, 12, 3),     # bulk ring, the warps of a CTA interleaved over one span
    (5, 3, 8, 4),
    (5, 7, 16, 2),
])
@pytest.mark.parametrize("nvec", [1, 4096 * 12 + 37, 300_001])
def test_every_vector_is_read_once(D, mode, ctas, warps, stages, nvec):
    rng = np.random.default_rng(nvec * 31 + mode)
    words = rng.integers(0, 2**32, size=4 * nvec, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32).copy()).cuda()
    out = torch.zeros(ctas * warps * 32, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = D.lib().dart_probe_stream(C.c_void_p(buf.data_ptr()), 16 * nvec, mode, ctas, warps, stages,
                                   C.c_void_p(out.data_ptr()), C.c_void_p(err.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = np.bitwise_xor.reduce(out.cpu().numpy().view(np.uint32))
    want = np.bitwise_xor.reduce(words) & np.uint32(0x3FFFFFFF)
    assert int(got) == int(want)
