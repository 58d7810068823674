"""Caller-supplied pair scores as the continuity term, against the oracle (needs a GB300).

DARTree, Method / Tree Construction scores every child of a depth with a head
in one batch.  An order-2 head restricted to the candidate sets is a table of
pair scores [B][d][k][k]; here it is a random low-rank head (synth), scored on
the host from the oracle's own candidate lists and handed to both sides.
Tree stage from lists: tokens, parents, depths, masks and float scores
bit-exact.  Tree stage on the row pass's workspace: the row ids must equal the
oracle's first, then the same bar as the whole path (structure bit-exact,
scores within 1e-5).
"""
import numpy as np
import pytest

import oracle
import synth
from tests import oracle_refs as R
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


def _np(t):
    return t.cpu().numpy()


PAIR_CASES = [
    # B, d, k, W, lam
    (4, 8, 8, 10, 0.3),
    (3, 16, 16, 32, 0.25),
    (2, 16, 32, 64, 0.5),        # 64-key runs
    (5, 6, 5, 50, 1.0),
    (3, 1, 7, 3, 0.7),           # one depth
    (4, 5, 1, 1, 0.5),           # a chain
    (3, 3, 3, 27, 0.4),          # nothing pruned
    (2, 5, 6, 8, 0.0),           # lambda = 0
]


@pytest.mark.parametrize("B,d,k,W,lam", PAIR_CASES)
def test_tree_from_topk_pairs_bit_exact(D, B, d, k, W, lam):
    V = 5000
    case = synth.make_case(B=B, d=d, V=V, dtype="bf16", T=1.0, k=k, W=W, n=0, M=0, lam=lam, beta=0.0,
                           recipe=("normal_spike", 3.0, 8.0), seed=B * 100 + d + k)
    rid, rlp, _ = oracle.rows(case.logits, "bf16", V, 1.0, k)
    rid = rid.reshape(B, d, k)
    rlp = rlp.reshape(B, d, k)
    roots = np.arange(B) + 17
    pair = synth.head_pair_scores(rid, roots, rank=8, seed=B + d)
    ref = oracle.tree_from_pairs(rid, rlp, pair, B=B, d=d, k=k, W=W, lam=case.lam)
    out = D.tree_from_topk(torch.from_numpy(rid).cuda(), torch.from_numpy(rlp).cuda(), W, case.lam,
                           pairs=torch.from_numpy(pair).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(out["tokens"]), ref["tokens"])
    np.testing.assert_array_equal(_np(out["parents"]), ref["parents"])
    np.testing.assert_array_equal(_np(out["pos"]), ref["pos"])
    np.testing.assert_array_equal(_np(out["mask"]).view(np.uint32), ref["mask"])
    np.testing.assert_array_equal(_np(out["scores"]), ref["scores"].astype(np.float32))


@pytest.mark.parametrize("cfg,over", [
    (1, dict(V=20000)),
    (2, dict(B=6)),
    (3, dict(B=24)),
    (4, dict(B=3)),
    (2, dict(B=4, T=0.0)),                       # greedy
    (4, dict(B=2, V=7777, dtype="f32", T=1.7)),  # ragged rows
])
def test_tree_from_rows_pairs_matches_oracle(D, cfg, over):
    """row_topk, then the caller's head on the candidates, then the tree stage
    on the workspace the row pass left."""
    case = synth.make_config(cfg, seed=3, M=0, n=0, **over)
    B, d, V, k, W = case.B, case.d, case.V, case.k, case.W
    z = parity.to_device(case)
    ids, logp, lse, ws = D.row_topk(z.reshape(B * d, V), case.T, k)
    assert D.device_error(ws) == 0
    rid, rlp, rlse = oracle.rows(case.logits, case.dtype, V, case.T, k)
    np.testing.assert_array_equal(_np(ids), rid)
    rid = rid.reshape(B, d, k)
    pair = synth.head_pair_scores(rid, np.arange(B) + 3, rank=16, seed=cfg)
    out = D.tree_from_rows(ws, torch.from_numpy(pair).cuda(), B=B, d=d, V=V, dtype=z.dtype, T=case.T,
                           k=k, W=W, lam=case.lam)
    assert D.device_error(ws) == 0
    # the oracle's ranking key: candidate logits * (1 / T) + lam * pair sum, scores minus the lse sums
    zf = R.decode_np(case.logits, case.dtype).reshape(B, d, V).astype(np.float64)
    base = np.take_along_axis(zf, rid.astype(np.int64), axis=2)
    T = 1.0 if case.T == 0 else float(case.T)
    ref = oracle.tree_from_pairs(rid, base, pair, B=B, d=d, k=k, W=W, lam=case.lam, invT=1.0 / T,
                                 off=rlse.reshape(B, d))
    got = {key: _np(v) for key, v in out.items() if v is not None}
    for key in ("tokens", "parents", "pos"):
        np.testing.assert_array_equal(got[key], ref[key])
    np.testing.assert_array_equal(got["mask"].view(np.uint32), ref["mask"])
    assert np.abs(got["scores"].astype(np.float64) - ref["scores"]).max() <= parity.SCORE_TOL


def test_pair_arguments(D):
    ids = torch.zeros((2, 3, 4), dtype=torch.int32, device="cuda")
    logp = torch.zeros((2, 3, 4), dtype=torch.float64, device="cuda")
    with pytest.raises(D.DartError):
        D.tree_from_topk(ids, logp, 4, 0.5, pairs=torch.zeros((2, 3, 4, 3), device="cuda"))
    with pytest.raises(D.DartError):
        D.tree_from_topk(ids, logp, 4, 0.5, pairs=torch.zeros((2, 3, 4, 4), dtype=torch.float64, device="cuda"))
    empty = D.tree_from_topk(ids[:0], logp[:0], 4, 0.5, pairs=torch.zeros((0, 3, 4, 4), device="cuda"))
    assert empty["tokens"].shape == (0, D.num_nodes(3, 4, 4))
