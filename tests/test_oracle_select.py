"""Pins of the oracle's verification-tree selection (best-first with a budget).

DARTree (abstract; Verification): the candidate tree is built first, then
best-first pruning picks the tree sent to verification; PCTree (abstract): a
fixed verification budget goes to the most probable paths.  The pins: the
worked example (hand-derived budgets 1..5), brute force over every size-M
subset on small trees (for path scores that never rise, best-first picks the
M-subset of largest score sum), the availability rule on a tree whose child
outscores its parent, equal scores, and the budget edge cases.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from tests import oracle_refs as R


def _check_consistent(tree, out, M):
    """Gathered tokens / depths, renumbered parents and masks agree with the
    chosen original indices (Python sets, no oracle code)."""
    B, N = tree["parents"].shape
    for b in range(B):
        idx = out["index"][b].tolist()
        assert idx == sorted(idx) and len(set(idx)) == len(idx) == min(M, N)
        where = {x: m for m, x in enumerate(idx)}
        for m, x in enumerate(idx):
            assert out["tokens"][b, m] == tree["tokens"][b, x]
            assert out["pos"][b, m] == tree["pos"][b, x]
            p = tree["parents"][b, x]
            assert out["parents"][b, m] == (-1 if p < 0 else where[p])
        sets = R.masks_from_sets(out["parents"][b].tolist())
        for m in range(len(idx)):
            assert R.mask_row_to_set(out["mask"][b, m]) == sets[m]


def test_worked_example_budgets():
    with open(os.path.join(R.GOLDEN, "we1_select.json")) as f:
        ex = json.load(f)
    t = ex["tree"]
    tree = dict(tokens=np.array([t["tokens"]]), parents=np.array([t["parents"]]), pos=np.array([t["pos"]]),
                scores=np.array([[R.eval_closed_form(s) for s in t["scores"]]]))
    for M, want in ex["expect"].items():
        out = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"], int(M))
        for key in ("index", "tokens", "parents", "pos"):
            assert out[key][0].tolist() == want[key], (M, key)
        assert out["mask"][0, :, 0].tolist() == want["mask"]
        _check_consistent(tree, out, int(M))


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_best_sum(seed):
    d, k, W = (3, 2, 4) if seed % 2 else (2, 3, 6)
    tree = synth.make_candidate_trees(B=2, d=d, k=k, W=W, seed=100 + seed, tie_frac=0.0, zero_frac=0.0)
    N = tree["parents"].shape[1]
    for M in range(0, N + 2):
        out = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"], M)
        _check_consistent(tree, out, M)
        for b in range(2):
            s = tree["scores"][b].astype(np.float64).tolist()
            want = R.best_sum_subset(s, min(M, N))
            assert out["index"][b].tolist() == sorted(want), (seed, M, b)
            chosen = set(want)
            for x in chosen:            # ancestor-closed
                p = tree["parents"][b, x]
                assert p < 0 or p in chosen


def test_parents_are_renumbered():
    # node 0 is not taken, so node 2's parent (node 1) becomes position 0
    out = oracle.select_tree(np.array([[4, 5, 6]]), np.array([[-1, -1, 1]]), np.array([[1, 1, 2]]),
                             np.array([[-9.0, -1.0, -2.0]]), 2)
    assert out["index"][0].tolist() == [1, 2]
    assert out["tokens"][0].tolist() == [5, 6] and out["parents"][0].tolist() == [-1, 0]
    assert out["mask"][0, :, 0].tolist() == [1, 3]


def test_equal_scores_take_the_lower_index():
    par = np.array([[-1, -1, -1, 1, 2]])
    s = np.array([[-2.0, -1.0, -1.0, -1.0, -1.0]])
    tok = np.arange(5)[None]
    dep = np.array([[1, 1, 1, 2, 2]])
    assert oracle.select_tree(tok, par, dep, s, 1)["index"][0].tolist() == [1]
    # node 3 ties its parent 1 and node 2; lower index first among the available
    assert oracle.select_tree(tok, par, dep, s, 2)["index"][0].tolist() == [1, 2]
    assert oracle.select_tree(tok, par, dep, s, 3)["index"][0].tolist() == [1, 2, 3]


def test_a_child_is_available_only_after_its_parent():
    # node 2 outscores everything but hangs under node 1, which is taken after node 0
    par = np.array([[-1, -1, 1]])
    s = np.array([[-5.0, -6.0, -1.0]])
    tok = np.array([[7, 8, 9]])
    dep = np.array([[1, 1, 2]])
    assert oracle.select_tree(tok, par, dep, s, 1)["index"][0].tolist() == [0]
    assert oracle.select_tree(tok, par, dep, s, 2)["index"][0].tolist() == [0, 1]
    assert oracle.select_tree(tok, par, dep, s, 3)["index"][0].tolist() == [0, 1, 2]


def test_budget_edges():
    tree = synth.make_candidate_trees(B=3, d=3, k=3, W=5, seed=7)
    N = tree["parents"].shape[1]
    out0 = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"], 0)
    assert out0["index"].shape == (3, 0) and out0["mask"].shape == (3, 0, 0)
    for M in (N, N + 5):
        out = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"], M)
        assert (out["index"] == np.arange(N)[None]).all()
        assert (out["parents"] == tree["parents"]).all() and (out["tokens"] == tree["tokens"]).all()
    one = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"], 1)
    for b in range(3):
        d1 = np.where(tree["pos"][b] == 1)[0]
        best = d1[np.lexsort((d1, -tree["scores"][b, d1].astype(np.float64)))[0]]
        assert one["index"][b].tolist() == [best]


def test_bad_parent_array_is_rejected():
    with pytest.raises(ValueError):
        oracle.select_tree(np.zeros((1, 3)), np.array([[-1, 2, 0]]), np.ones((1, 3)), np.zeros((1, 3)), 2)


@pytest.mark.parametrize("d,k,W", [(3, 3, 5), (8, 8, 10), (16, 16, 32), (32, 32, 32)])
def test_seeded_candidate_trees_have_the_stated_shape(d, k, W):
    """The generator feeding the GPU selection tests: depth-major nodes with
    min(W, k^j) per depth, parents one depth up with at most k children each,
    scores that never rise along a path, and some exact ties."""
    tree = synth.make_candidate_trees(B=3, d=d, k=k, W=W, seed=d + k + W)
    sizes = [min(W, k ** j) for j in range(1, d + 1)]
    N = sum(sizes)
    assert tree["parents"].shape == (3, N) and tree["scores"].dtype == np.float32
    ties = 0
    for b in range(3):
        par, pos, sc = tree["parents"][b], tree["pos"][b], tree["scores"][b]
        assert pos.tolist() == [j for j, n in enumerate(sizes, start=1) for _ in range(n)]
        for i in range(N):
            p = par[i]
            if pos[i] == 1:
                assert p == -1
            else:
                assert 0 <= p < i and pos[p] == pos[i] - 1 and sc[i] <= sc[p]
        counts = np.bincount(par[par >= 0], minlength=N)
        assert counts.max(initial=0) <= k
        ties += N - len(np.unique(sc))
    assert ties > 0
