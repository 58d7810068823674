"""Verification-tree selection on the GPU against the oracle (needs a GB300).

Both sides get the same seeded candidate trees (float32 scores, the oracle
reading them as doubles), so index, tokens, renumbered parents, depths and
masks must be bit-exact, for every budget from 0 to past N and for trees up to
the 1024-node limit.  The whole path (tree build then selection) is compared
with the oracle's own path on every tree whose candidate tree matched exactly
and whose oracle scores leave a gap of at least 1e-4 at the budget's cut.
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


def _dev(tree):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in tree.items()}


def _compare(D, tree, M, err=None):
    t = _dev(tree)
    got = D.tree_select(t["tokens"], t["parents"], t["pos"], t["scores"], M, device_err=err)
    want = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"],
                              tree["scores"].astype(np.float64), M)
    for key in ("index", "tokens", "parents", "pos"):
        assert np.array_equal(got[key].cpu().numpy(), want[key]), (M, key)
    assert np.array_equal(got["mask"].cpu().numpy().view(np.uint32), want["mask"]), M
    gathered = np.take_along_axis(tree["scores"], want["index"].astype(np.int64), axis=1)
    assert np.array_equal(got["scores"].cpu().numpy(), gathered)


SHAPES = [(4, 4, 4), (3, 3, 5), (8, 8, 10), (8, 10, 16), (5, 2, 7), (16, 16, 32), (32, 32, 32)]


@pytest.mark.parametrize("d,k,W", SHAPES)
def test_select_matches_oracle(D, d, k, W):
    tree = synth.make_candidate_trees(B=6, d=d, k=k, W=W, seed=d * 100 + k + W)
    N = tree["parents"].shape[1]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    budgets = sorted({1, 2, N // 3, N // 2, N - 1, N, N + 3, 60 % N + 1})
    for M in budgets:
        _compare(D, tree, M, err)
    assert int(err.item()) == 0


def test_every_budget_small_trees(D):
    tree = synth.make_candidate_trees(B=8, d=4, k=3, W=6, seed=11, tie_frac=0.3, zero_frac=0.2)
    N = tree["parents"].shape[1]
    for M in range(0, N + 2):
        _compare(D, tree, M)


def test_32_trees_of_496_nodes(D):
    # the largest benchmarked tree shape (d = 16, k = 16, W = 32): 32 trees of 496 nodes, budget 256
    tree = synth.make_candidate_trees(B=32, d=16, k=16, W=32, seed=4)
    _compare(D, tree, 256)


def test_a_node_above_its_parent_is_flagged(D):
    tree = dict(tokens=np.array([[7, 8, 9]], dtype=np.int32), parents=np.array([[-1, -1, 1]], dtype=np.int32),
                pos=np.array([[1, 1, 2]], dtype=np.int32), scores=np.array([[-5.0, -6.0, -1.0]], dtype=np.float32))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = _dev(tree)
    got = D.tree_select(t["tokens"], t["parents"], t["pos"], t["scores"], 2, device_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 16          # DART_DEVERR_SCORE_RISES
    # the two best scores: node 2 (whose parent is not kept) and node 0
    assert got["index"].cpu().tolist() == [[0, 2]] and got["parents"].cpu().tolist() == [[-1, -2]]


@pytest.mark.parametrize("cfg,over,M", [
    (0, {}, 6),
    (2, dict(B=8, M=1 << 16), 40),
    (3, dict(B=32, M=1 << 16), 60),
    (4, dict(B=4, M=1 << 18), 200),
])
def test_whole_path_then_select(D, cfg, over, M):
    case = synth.make_config(cfg, seed=21, **over)
    z = parity.to_device(case)
    tab, ctx = parity.gpu_table(case)
    out = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx)
    assert D.device_error(out["workspace"]) == 0
    sel = D.tree_select(out["tokens"], out["parents"], out["pos"], out["scores"], M)
    want = oracle.tree_build(case)
    ref = oracle.select_tree(want["tokens"], want["parents"], want["pos"], want["scores"], M)
    B, N = want["parents"].shape
    checked = 0
    for b in range(B):
        same = all(np.array_equal(out[key][b].cpu().numpy(), want[key][b]) for key in ("tokens", "parents", "pos"))
        s = np.sort(want["scores"][b])[::-1]
        if not same or (M < N and s[M - 1] - s[M] < 1e-4):
            continue   # a different candidate tree, or a near tie at the cut: either side may take it
        checked += 1
        for key in ("index", "tokens", "parents", "pos"):
            assert sel[key][b].cpu().tolist() == ref[key][b].tolist(), (b, key)
        assert np.array_equal(sel["mask"][b].cpu().numpy().view(np.uint32), ref["mask"][b])
    assert checked >= max(1, B // 2)


@pytest.mark.parametrize("cfg,over", [
    (0, {}),
    (2, dict(B=8, M=1 << 16)),
    (3, dict(B=32, M=1 << 16)),
    (4, dict(B=4, M=1 << 18)),
    (2, dict(B=4, M=1 << 14, T=0.0)),
])
def test_tree_build_emits_the_verification_tree(D, cfg, over):
    """dart_tree_build_verify: the tree kernel chooses each tree's verification
    tree right after building it.  Its result must be the oracle's selection
    on the candidate trees the same call returned (bit-exact), for budgets
    from 1 to past N; the candidate trees must equal those of tree_build."""
    case = synth.make_config(cfg, seed=31, **over)
    z = parity.to_device(case)
    tab, ctx = parity.gpu_table(case)
    plain = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx)
    N = plain["parents"].shape[1]
    for M in sorted({1, 7, 16, N // 2, N, N + 5}):
        out = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx, verify_budget=M)
        assert D.device_error(out["workspace"]) == 0
        for key in ("tokens", "parents", "pos", "mask", "scores"):
            assert torch.equal(out[key], plain[key]), key
        tree = {key: out[key].cpu().numpy() for key in ("tokens", "parents", "pos", "scores")}
        want = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"].astype(np.float64), M)
        v = out["verify"]
        for key in ("index", "tokens", "parents", "pos"):
            assert np.array_equal(v[key].cpu().numpy(), want[key]), (M, key)
        assert np.array_equal(v["mask"].cpu().numpy().view(np.uint32), want["mask"]), M
        gathered = np.take_along_axis(tree["scores"], want["index"].astype(np.int64), axis=1)
        assert np.array_equal(v["scores"].cpu().numpy(), gathered)
