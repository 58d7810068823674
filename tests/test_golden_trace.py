"""The small bigram workload's step-by-step trace (tests/golden/config0_trace.*).

The committed trace was written by tests/golden/make_config0_trace.py, which
calls only the oracle.  This test (1) regenerates it and demands the same
content, so the oracle cannot drift from the printed numbers, and (2) checks
every number of the committed trace by independent arithmetic: the rows
against numpy's sort and scipy's log-softmax of the regenerated logits, the
52 probes against a Python dict of the n-gram model, each depth's table by
recomputing Z, G and the key from the parent's row and re-sorting with the
tie rule (DART, Figure 3 caption; DARTree, Method / Tree Construction).
"""
import json
import os

import numpy as np
import scipy.special

import synth
from tests import oracle_refs as R

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load():
    with open(os.path.join(HERE, "config0_trace.json")) as f:
        return json.load(f)


def _script():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_config0_trace", os.path.join(HERE, "make_config0_trace.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _same(a, b, path="trace"):
    if isinstance(a, dict):
        assert set(a) == set(b), path
        for key in a:
            _same(a[key], b[key], f"{path}.{key}")
    elif isinstance(a, list):
        assert len(a) == len(b), path
        for i, (x, y) in enumerate(zip(a, b)):
            _same(x, y, f"{path}[{i}]")
    elif isinstance(a, float):
        assert abs(a - b) <= 1e-12 * max(1.0, abs(b)), (path, a, b)
    else:
        assert a == b, (path, a, b)


def test_trace_regenerates_from_the_oracle():
    mod = _script()
    _same(mod.build_trace(), _load())
    with open(os.path.join(HERE, "config0_trace.txt")) as f:
        assert f.read() == mod.as_text(_load())


def test_rows_are_the_top4_of_the_logits():
    t = _load()
    case = synth.make_config(0, seed=0)
    z = case.logits.reshape(case.d, case.V).astype(np.float64)
    for j, row in enumerate(t["rows"]):
        want = R.topk_lexsort(z[j], 4)
        assert row["ids"] == want.tolist()
        assert row["logits"] == z[j][want].tolist()
        lsm = scipy.special.log_softmax(z[j] / t["workload"]["T"])
        np.testing.assert_allclose(row["logp"], lsm[want], rtol=0, atol=1e-12)
        np.testing.assert_allclose(row["lse"], scipy.special.logsumexp(z[j]), rtol=0, atol=1e-12)


def test_probes_against_a_dict():
    t = _load()
    case = synth.make_config(0, seed=0)
    table = R.dict_ngram(case.ng_keys, case.ng_vals)
    assert len(t["probes"]) == 4 + 16 + 16 + 16 == 52
    for p in t["probes"]:
        g = table.get((p["context"], p["token"]))
        assert p["found"] == (g is not None)
        assert p["g"] == (g if g is not None else t["workload"]["beta"])


def test_tables_recomputed_by_hand():
    t = _load()
    w = t["workload"]
    lam, T = w["lam"], w["T"]
    case = synth.make_config(0, seed=0)
    table = R.dict_ngram(case.ng_keys, case.ng_vals)
    nodes = {-1: dict(Z=0.0, G=0.0, token=t["ctx"][-1])}    # the root: its token is the context's last
    tree_tokens, tree_parents = [], []
    next_node = 0
    for j, rows in enumerate(t["tables"]):
        r = t["rows"][j]
        frontier = sorted(nodes) if j == 0 else [x for x in sorted(nodes) if x >= 0 and nodes[x]["depth"] == j]
        if j == 0:
            frontier = [-1]
        # every child of the frontier, scored from its parent and its row
        expect = []
        for par in frontier:
            for c, tok in enumerate(r["ids"]):
                g = table.get((nodes[par]["token"], tok))
                g = g if g is not None else w["beta"]
                Z = nodes[par]["Z"] + r["logits"][c]
                G = nodes[par]["G"] + g
                expect.append(dict(parent=par, token=tok, Z=Z, G=G, key=Z * (1.0 / T) + lam * G))
        expect.sort(key=lambda e: (-e["key"], e["parent"], e["token"]))
        assert [(e["parent"], e["token"]) for e in rows] == [(e["parent"], e["token"]) for e in expect]
        for got, want in zip(rows, expect):
            for key in ("Z", "G", "key"):
                assert got[key] == want[key], (j, key)
        keep = min(w["W"], len(rows))
        assert [e["node"] for e in rows] == list(range(next_node, next_node + keep)) + [-1] * (len(rows) - keep)
        for e in rows[:keep]:
            nodes[e["node"]] = dict(Z=e["Z"], G=e["G"], token=e["token"], depth=j + 1)
            tree_tokens.append(e["token"])
            tree_parents.append(e["parent"])
        next_node += keep
    tree = t["tree"]
    assert tree["tokens"] == tree_tokens
    assert tree["parents"] == tree_parents
    lse = np.cumsum([r["lse"] for r in t["rows"]])
    for x, (key, depth) in enumerate(zip([e["key"] for rows in t["tables"] for e in rows if e["node"] >= 0],
                                         tree["pos"])):
        np.testing.assert_allclose(tree["scores"][x], key - lse[depth - 1], rtol=0, atol=1e-12)
    for x, m in enumerate(tree["mask"]):
        assert R.mask_row_to_set([m]) == R.masks_from_sets(tree["parents"])[x]
