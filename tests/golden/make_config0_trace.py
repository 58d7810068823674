"""Writes config0_trace.json and config0_trace.txt: the small bigram workload
(B=1, d=4, V=1024, f32 N(0,2) logits, T=1, k=4, W=4, 4096 bigrams, lambda=0.5,
beta=-10, seed 0) traced step by step by the oracle, for reading by hand.

Contents: each row's top-4 (ids, stored logits, log-probabilities, log-sum-
exp); the 52 n-gram probes (4 children of the root, then 16 per depth); each
depth's whole sorted candidate table (Z = sum of the path's logits, G = sum
of its n-gram terms, key = Z / T + lambda * G, the node it became); and the
resulting tree.  Only the oracle and the seeded input generator are called.

    python tests/golden/make_config0_trace.py
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402

JSON_PATH = os.path.join(HERE, "config0_trace.json")
TEXT_PATH = os.path.join(HERE, "config0_trace.txt")


def build_trace(lib=None) -> dict:
    case = synth.make_config(0, seed=0)
    d, k, W, V = case.d, case.k, case.W, case.V
    ids, logp, lse = oracle.rows(case.logits, case.dtype, V, case.T, k, lib=lib)
    z = case.logits.reshape(d, V).astype(np.float64)
    base = np.take_along_axis(z, ids.astype(np.int64), 1)
    ng = oracle.NGram(case.n, case.ng_keys, case.ng_vals, lib=lib)
    tr = oracle.tree_trace(ids, base, d=d, k=k, W=W, lam=case.lam, beta=case.beta, ngram=ng,
                           ctx=case.ctx[0], invT=1.0 / case.T, off=lse, lib=lib)
    tree = oracle.tree_build(case, ngram=ng, lib=lib)
    tokens = tree["tokens"][0]
    root_ctx = int(case.ctx[0][-1])
    probes, tables = [], []
    for j in range(1, d + 1):
        rows = tr[tr["depth"] == j]
        tables.append([dict(parent=int(e["parent"]), token=int(e["token"]), Z=float(e["Z"]), G=float(e["G"]),
                            key=float(e["key"]), node=int(e["node"])) for e in rows])
        for e in sorted(rows, key=lambda e: (int(e["parent_rank"]), int(e["column"]))):
            context = root_ctx if e["parent"] < 0 else int(tokens[e["parent"]])
            probes.append(dict(depth=j, parent=int(e["parent"]), context=context, token=int(e["token"]),
                               found=bool(e["found"]), g=float(e["g"])))
    return {
        "workload": dict(B=1, d=d, V=V, dtype=case.dtype, T=float(case.T), k=k, W=W, n=case.n,
                         M=int(len(case.ng_keys)), lam=float(case.lam), beta=float(case.beta), seed=0),
        "ctx": [int(t) for t in case.ctx[0]],
        "rows": [dict(ids=[int(x) for x in ids[j]], logits=[float(x) for x in base[j]],
                      logp=[float(x) for x in logp[j]], lse=float(lse[j])) for j in range(d)],
        "probes": probes,
        "tables": tables,
        "tree": dict(tokens=[int(x) for x in tokens], parents=[int(x) for x in tree["parents"][0]],
                     pos=[int(x) for x in tree["pos"][0]], scores=[float(x) for x in tree["scores"][0]],
                     mask=[int(x) for x in tree["mask"][0, :, 0]]),
    }


def as_text(t: dict) -> str:
    w = t["workload"]
    out = [f"Small bigram workload, traced by the oracle: B=1 d={w['d']} V={w['V']} {w['dtype']} T={w['T']} "
           f"k={w['k']} W={w['W']} n={w['n']} ({w['M']} n-grams) lambda={w['lam']} beta={w['beta']} seed={w['seed']}",
           f"committed context (root last): {t['ctx']}", "", "Rows: top-4 by logit (id, logit, log-probability)"]
    for j, r in enumerate(t["rows"]):
        cells = "  ".join(f"{i}:{z:+.6f}/{p:+.6f}" for i, z, p in zip(r["ids"], r["logits"], r["logp"]))
        out.append(f"  row {j} (depth {j + 1}) lse {r['lse']:.9f}:  {cells}")
    out += ["", f"N-gram probes ({len(t['probes'])}): depth, parent node, (context, token) -> value "
            "(beta when absent)"]
    for p in t["probes"]:
        val = f"{p['g']:+.6f}" if p["found"] else f"absent -> {p['g']:+.1f}"
        out.append(f"  d{p['depth']} parent {p['parent']:>2}  ({p['context']:>4}, {p['token']:>4})  {val}")
    for j, rows in enumerate(t["tables"]):
        out += ["", f"Depth {j + 1}: sorted by key = Z/T + lambda*G, then parent, then token "
                f"({len(rows)} children, {sum(r['node'] >= 0 for r in rows)} kept)"]
        for r in rows:
            kept = f"node {r['node']}" if r["node"] >= 0 else "cut"
            out.append(f"  parent {r['parent']:>2} token {r['token']:>4}  Z {r['Z']:+.6f}  G {r['G']:+.6f}  "
                       f"key {r['key']:+.6f}  {kept}")
    tr = t["tree"]
    out += ["", "Tree: node, token, parent, depth, score, ancestor mask (bits)"]
    for x, (a, b, c, s, m) in enumerate(zip(tr["tokens"], tr["parents"], tr["pos"], tr["scores"], tr["mask"])):
        out.append(f"  {x:>2} {a:>4} {b:>3} {c} {s:+.6f} {m:016b}")
    return "\n".join(out) + "\n"


def main():
    t = build_trace()
    with open(JSON_PATH, "w") as f:
        json.dump(t, f, indent=1)
        f.write("\n")
    with open(TEXT_PATH, "w") as f:
        f.write(as_text(t))


if __name__ == "__main__":
    main()
