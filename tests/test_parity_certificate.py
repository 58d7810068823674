"""The near-tie exemption of tests/parity.py, driven on the CPU.

compare_tree accepts a tree that differs from the oracle's only where the
oracle's sorted candidate list has two neighbours closer than NEAR_TIE, and
then checks the tree by a certificate.  A planted near tie swapped at the cut
must pass as "certified"; the same swap without a near tie, or a certified
tree that drops a clearly better child further down, must fail.
"""
import types

import numpy as np
import pytest

import oracle
from tests import parity


def _case(d, k, W):
    return types.SimpleNamespace(B=1, d=d, k=k, W=W, n=0, lam=0.0, beta=0.0, ctx=np.zeros((1, 0), np.int32))


def _tree(ids, logp, W):
    B, d, k = ids.shape
    return oracle.tree_from_lists(ids, logp, B=B, d=d, k=k, W=W, lam=0.0, beta=0.0, ngram=None, ctx=None)


def _ref(ids, logp, W):
    ref = _tree(ids, logp, W)
    ref["row_ids"] = ids
    ref["row_logp"] = logp
    return ref


def _as_gpu(out):
    """A tree in the GPU's output form: float32 scores, int32 mask storage."""
    return {"tokens": out["tokens"][0], "parents": out["parents"][0], "pos": out["pos"][0],
            "mask": out["mask"][0].view(np.int32), "scores": out["scores"][0].astype(np.float32)}


IDS = np.array([[[10, 11, 12], [20, 21, 22]]], dtype=np.int32)


def _lists(third):
    """Row 0 keeps 2 of 3 children (W = 2); `third` is the logp of its third candidate."""
    return np.array([[[-0.1, -1.0, third], [-0.2, -0.7, -2.0]]])


def test_identical_tree_is_exact():
    logp = _lists(-1.5)
    ref = _ref(IDS, logp, 2)
    assert parity.compare_tree(_case(2, 3, 2), 0, _as_gpu(_tree(IDS, logp, 2)), ref, None) == "exact"


def test_swap_at_a_planted_near_tie_is_certified():
    logp = _lists(-1.0 - 5e-6)                 # candidates 1 and 2 of row 0 are 5e-6 apart
    ref = _ref(IDS, logp, 2)
    assert ref["min_pos_gap"][0, 0] < parity.NEAR_TIE
    swapped = logp.copy()
    swapped[0, 0, [1, 2]] = swapped[0, 0, [2, 1]]  # the other side of the tie wins the cut
    g = _as_gpu(_tree(IDS, swapped, 2))
    assert not np.array_equal(g["tokens"], ref["tokens"][0])
    assert parity.compare_tree(_case(2, 3, 2), 0, g, ref, None) == "certified"


def test_swap_without_a_near_tie_fails():
    logp = _lists(-1.5)
    ref = _ref(IDS, logp, 2)
    swapped = logp.copy()
    swapped[0, 0, [1, 2]] = swapped[0, 0, [2, 1]]
    g = _as_gpu(_tree(IDS, swapped, 2))
    with pytest.raises(AssertionError, match="no near-tie"):
        parity.compare_tree(_case(2, 3, 2), 0, g, ref, None)


def test_certificate_catches_a_bad_cut_below_the_tie():
    logp = _lists(-1.0 - 5e-6)
    ref = _ref(IDS, logp, 2)
    swapped = logp.copy()
    swapped[0, 0, [1, 2]] = swapped[0, 0, [2, 1]]
    g = _as_gpu(_tree(IDS, swapped, 2))
    # at depth 2 replace the best kept child by a dropped, clearly worse one
    depth2 = np.flatnonzero(g["pos"] == 2)
    x = depth2[0]
    g["tokens"] = g["tokens"].copy()
    g["scores"] = g["scores"].copy()
    g["tokens"][x] = 22                        # logp -2.0 instead of -0.2
    g["scores"][x] = g["scores"][g["parents"][x]] - 2.0
    with pytest.raises(AssertionError):
        parity.compare_tree(_case(2, 3, 2), 0, g, ref, None)


def test_certificate_catches_a_wrong_score():
    logp = _lists(-1.0 - 5e-6)
    ref = _ref(IDS, logp, 2)
    swapped = logp.copy()
    swapped[0, 0, [1, 2]] = swapped[0, 0, [2, 1]]
    g = _as_gpu(_tree(IDS, swapped, 2))
    g["scores"] = g["scores"].copy()
    g["scores"][1] += 1e-3
    with pytest.raises(AssertionError, match="score"):
        parity.compare_tree(_case(2, 3, 2), 0, g, ref, None)
