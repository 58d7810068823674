"""The row pass's bounded waits, made to run out on purpose (needs a GB300).

No fault is involved: with every wait limited to 64 SM cycles a warp's wait
for its first bulk-copy stage (which cannot land that fast) gives up, the warp
lets its copies in flight land and returns with DART_DEVERR_WAIT_TIMEOUT in
the workspace.  The
context stays usable: dart_device_error reports the bit and clears the
workspace, and the next call with the default limit is exact again.
"""
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


def test_a_wait_that_runs_out_is_reported_and_the_workspace_recovers(D):
    rows, V, k = 48, 151936, 8
    case = synth.make_case(B=rows, d=1, V=V, dtype="bf16", T=1.0, k=k, W=1, n=0, M=0, lam=0, beta=0,
                           recipe=("normal_spike", 3.0, 12.0), seed=77)
    z = parity.to_device(case).reshape(rows, V)
    ws = torch.zeros(D.workspace_bytes(rows, 1, V, 2, k), dtype=torch.uint8, device="cuda")
    D.set_wait_limit(64)
    try:
        D.row_topk(z, 1.0, k, workspace=ws)
        flags = D.device_error(ws)
    finally:
        D.set_wait_limit(0)
    assert flags & 1, flags                      # DART_DEVERR_WAIT_TIMEOUT
    # the bit is reported once: the read cleared the workspace
    assert D.device_error(ws) == 0
    ids, logp, lse, _ = D.row_topk(z, 1.0, k, workspace=ws)
    assert D.device_error(ws) == 0
    rid, rlogp, rlse = oracle.rows(case.logits, "bf16", V, 1.0, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - rlse).max() <= 1e-5
