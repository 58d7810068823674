"""dart_tree_build_noalloc against the oracle and dart_tree_build, through the C ABI.

The no-allocation entry point serves callers that cannot hand the library a
workspace of their own: engines whose pool allocator owns the device memory,
plugins without access to the application's allocator, or decode loops that
must not pay for cudaMalloc's device synchronisation.  It runs the same
kernels on a fixed buffer inside the library, so its outputs must equal those
of dart_tree_build bit for bit (scores included) and match the oracle.
Several calls in a row check that no call depends on what the previous one
left in the shared buffer.  This file is collected last, so the buffer has
already served the other tests' process when it runs in the full suite.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def D():
    import draft_tree_construction_gb300 as D
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D.build()
    return D


def _noalloc(D, case, z, tab, ctx):
    """Call dart_tree_build_noalloc directly; outputs are caller-owned tensors."""
    N = D.num_nodes(case.d, case.k, case.W)
    MW = D.mask_words(N)
    out = {key: torch.empty((case.B, N), dtype=torch.int32, device="cuda")
           for key in ("tokens", "parents", "pos")}
    out["mask"] = torch.empty((case.B, N, MW), dtype=torch.int32, device="cuda")
    out["scores"] = torch.empty((case.B, N), dtype=torch.float32, device="cuda")
    p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
    rc = D.lib().dart_tree_build_noalloc(
        p(z), case.B, case.d, case.V, D.DTYPE_CODES()[z.dtype], case.T, case.k, case.W,
        case.lam, case.beta, C.byref(tab.desc) if tab is not None else None,
        p(ctx) if tab is not None else None, p(out["tokens"]), p(out["parents"]), p(out["pos"]),
        p(out["mask"]), p(out["scores"]), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, D.lib().dart_status_string(rc).decode()
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_oracle_and_tree_build_on_consecutive_calls(D):
    assert D.noalloc_device_error() == 0
    cases = [synth.make_config(2, seed=1, B=6, M=1 << 15),
             synth.make_config(0, seed=0),
             synth.make_config(4, seed=2, B=2, V=20011, M=1 << 15, dtype="f16"),
             synth.make_config(3, seed=4, B=12, M=1 << 14, T=0.0)]
    for case in cases + cases[:1]:          # the last call repeats the first on a used buffer
        z = parity.to_device(case)
        tab, ctx = parity.gpu_table(case)
        ref = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx)
        assert D.device_error(ref["workspace"]) == 0
        got = _noalloc(D, case, z, tab, ctx)
        assert D.noalloc_device_error() == 0
        for key in ("tokens", "parents", "pos", "mask", "scores"):
            assert torch.equal(got[key], ref[key]), key
        want = oracle.tree_build(case)
        host = {key: v.cpu().numpy() for key, v in got.items()}
        stats = parity.compare_all(case, host, want, want["ngram"])
        assert stats["exact"] == case.B


def test_noalloc_binding_and_error_readout(D):
    """A wait limit of 64 SM cycles makes the row pass give up (no fault: the
    warps let their copies land and return); the bit shows up in the internal
    buffer's error word, is cleared by the read, and the next call is exact."""
    case = synth.make_config(2, seed=3, B=8, M=1 << 12)
    z = parity.to_device(case)
    tab, ctx = parity.gpu_table(case)
    # the logits come from HBM, not from L2, so no bulk copy can land within
    # the first waits' 64 cycles
    flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    D.set_wait_limit(64)
    try:
        flush.mul_(1.0)
        D.tree_build_noalloc(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx)
        flags = D.noalloc_device_error()
    finally:
        D.set_wait_limit(0)
    assert flags & 1, flags                      # DART_DEVERR_WAIT_TIMEOUT
    assert D.noalloc_device_error() == 0         # reported once
    got = D.tree_build_noalloc(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx,
                               check_errors=True)
    want = oracle.tree_build(case)
    host = {key: v.cpu().numpy() for key, v in got.items() if v is not None}
    assert parity.compare_all(case, host, want, want["ngram"])["exact"] == case.B
