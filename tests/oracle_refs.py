"""Independent references used to pin the oracle (not the oracle itself).

Each helper here is written from a definition that does not go through
oracle.c: exhaustive enumeration of all k^d paths, Python dictionaries for the
n-gram model, numpy / scipy library routines for sorting and log-softmax,
Python sets for ancestor masks, and closed forms from the worked examples.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def decode_np(logits: np.ndarray, dtype: str) -> np.ndarray:
    """Stored logits -> float64 through numpy's own conversions."""
    if dtype == "f32":
        return logits.astype(np.float64)
    if dtype == "f16":
        return logits.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (logits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def topk_lexsort(z: np.ndarray, k: int) -> np.ndarray:
    """k best ids of a 1-D row: value descending, lower id first (numpy lexsort)."""
    ids = np.arange(z.shape[0])
    order = np.lexsort((ids, -z))
    return order[:k]


def load_worked_example(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        ex = json.load(f)
    V, d = ex["V"], ex["d"]
    probs = np.zeros((d, V), dtype=np.float64)
    for j, row in enumerate(ex["probs"]):
        probs[j, :] = ex_default(row)
        for tok, p in row["set"].items():
            probs[j, int(tok)] = p
    logits = np.log(probs).astype(np.float32)[None]   # [1, d, V] f32
    keys = np.array([t for t, _ in ex["table"]], dtype=np.int32).reshape(-1, ex["n"])
    vals = np.array([v for _, v in ex["table"]], dtype=np.float32)
    return ex, logits, keys, vals


def ex_default(row) -> float:
    num, den = row["default_num"].split("/")
    return float(num) / float(den)


def eval_closed_form(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"log": math.log}))


def dict_ngram(keys: np.ndarray, vals: np.ndarray) -> dict:
    """First value wins for a repeated key."""
    out = {}
    for key, v in zip(map(tuple, keys.tolist()), vals.tolist()):
        if key not in out:
            out[key] = float(np.float32(v))
    return out


def brute_force_paths(ids, logp, *, lam, beta, table: dict | None, n: int, ctx):
    """Every root-to-depth-j path for one tree, scored from its own token sequence.

    ids/logp: [d][k].  Returns {path tuple (of candidate ranks): score} over all
    depths 1..d (paths of every length), computed by direct enumeration.
    """
    d, k = len(ids), len(ids[0])
    out = {}
    for depth in range(1, d + 1):
        for ranks in itertools.product(range(k), repeat=depth):
            toks = [ids[j][ranks[j]] for j in range(depth)]
            seq = list(ctx) + toks
            s = 0.0
            for j in range(depth):
                s = s + logp[j][ranks[j]]
                if table is not None:
                    pos_in_seq = len(ctx) + j                  # index of token j in seq
                    context = tuple(seq[pos_in_seq - (n - 1):pos_in_seq])
                    g = table.get(context + (toks[j],))
                    s = s + lam * (g if g is not None else beta)
            out[ranks] = s
    return out


def node_paths(tokens, parents, ids):
    """For one tree: node -> tuple of candidate ranks from the root (via parents)."""
    N = len(tokens)
    paths = []
    for x in range(N):
        seq = []
        a = x
        while a >= 0:
            seq.append(tokens[a])
            a = parents[a]
        seq.reverse()
        ranks = tuple(list(ids[j]).index(t) for j, t in enumerate(seq))
        paths.append(ranks)
    return paths


def masks_from_sets(parents_row) -> list[set]:
    out = []
    for x in range(len(parents_row)):
        s = set()
        a = x
        while a >= 0:
            s.add(a)
            a = parents_row[a]
        out.append(s)
    return out


def mask_row_to_set(words) -> set:
    s = set()
    for w, word in enumerate(words):
        for b in range(32):
            if (int(word) >> b) & 1:
                s.add(w * 32 + b)
    return s


def whole_path_brute_force_ok(lib=None, seed=3, T=0.7) -> bool:
    """Rows + tree through oracle.tree_build with nothing pruned, against scipy's
    log_softmax and an exhaustive enumeration of the paths.  T = 0 (greedy)
    is scored with the draft's own log-probabilities, log_softmax(z)."""
    import scipy.special
    import oracle
    import synth
    case = synth.make_case(B=2, d=3, V=40, dtype="bf16", T=T, k=3, W=27, n=2, M=600, lam=0.5,
                           beta=-9.0, recipe=("normal", 3.0), seed=seed)
    T_score = 1.0 if case.T == 0 else case.T    # the temperature as the case stores it
    try:
        out = oracle.tree_build(case, lib=lib)
    except ValueError:
        return False
    z = decode_np(case.logits, "bf16")
    table = dict_ngram(case.ng_keys, case.ng_vals)
    for b in range(case.B):
        lsm = [scipy.special.log_softmax(z[b, j] / T_score) for j in range(case.d)]
        ids = [topk_lexsort(z[b, j], case.k).tolist() for j in range(case.d)]
        logp = [[lsm[j][t] for t in ids[j]] for j in range(case.d)]
        ref = brute_force_paths(ids, logp, lam=case.lam, beta=case.beta, table=table, n=case.n,
                                ctx=case.ctx[b].tolist())
        try:
            paths = node_paths(out["tokens"][b].tolist(), out["parents"][b].tolist(), ids)
        except (ValueError, IndexError):
            return False
        if sorted(paths) != sorted(ref.keys()):
            return False
        for x, p in enumerate(paths):
            if abs(out["scores"][b, x] - ref[p]) > 1e-10:
                return False
    return True


def pair_brute_force_paths(logp, pair, *, lam):
    """Every root-to-depth-j path of one tree scored with pair scores by direct
    enumeration: sum_j logp[j][c_j] + lam * sum_j pair[j][c_{j-1}][c_j], with
    c_{-1} = 0 (the root).  logp [d][k], pair [d][k][k]; keys are column tuples."""
    d, k = len(logp), len(logp[0])
    out = {}
    for depth in range(1, d + 1):
        for cols in itertools.product(range(k), repeat=depth):
            s = 0.0
            for j in range(depth):
                prev = cols[j - 1] if j > 0 else 0
                s = s + logp[j][cols[j]] + lam * float(pair[j][prev][cols[j]])
            out[cols] = s
    return out


def pair_trees_ok(lib=None, seeds=(31, 32)) -> bool:
    """Pins of oracle.tree_from_pairs.

    1. Nothing pruned (W = k^d): every path and its score against an
       enumeration.
    2. Pruned trees: pair scores that restate a bigram model on the candidate
       sets (pair[j][c'][c] = table(token of c' in row j-1, or the context's
       last token at j = 0; token of c in row j), beta when absent) give the
       n-gram tree exactly -- which needs the parent's column carried through
       every cut.
    3. lambda = 0 gives the tree with no continuity term."""
    import oracle
    import synth
    rng = np.random.default_rng(seeds[0])
    for seed in seeds:
        B, d, k = 2, 3, 3
        ids = np.stack([np.stack([rng.permutation(50)[:k] for _ in range(d)]) for _ in range(B)]).astype(np.int32)
        logp = -rng.exponential(2.0, size=(B, d, k))
        pair = (-rng.exponential(1.5, size=(B, d, k, k))).astype(np.float32)
        out = oracle.tree_from_pairs(ids, logp, pair, B=B, d=d, k=k, W=k ** d, lam=0.7, lib=lib)
        for b in range(B):
            ref = pair_brute_force_paths(logp[b], pair[b], lam=0.7)
            try:
                paths = node_paths(out["tokens"][b].tolist(), out["parents"][b].tolist(), ids[b].tolist())
            except (ValueError, IndexError):
                return False
            if sorted(paths) != sorted(ref.keys()):
                return False
            for x, q in enumerate(paths):
                if abs(out["scores"][b, x] - ref[q]) > 1e-12:
                    return False
        # 2: a bigram model restated as pair scores, with pruning
        case = synth.make_case(B=3, d=5, V=60, dtype="f32", T=1.0, k=4, W=5, n=2, M=900, lam=0.4,
                               beta=-7.0, recipe=("normal", 3.0), seed=seed)
        ng = oracle.NGram(2, case.ng_keys, case.ng_vals, lib=lib)
        rid, rlp, _ = oracle.rows(case.logits, "f32", case.V, 1.0, case.k, lib=lib)
        rid = rid.reshape(case.B, case.d, case.k)
        rlp = rlp.reshape(case.B, case.d, case.k)
        table = dict_ngram(case.ng_keys, case.ng_vals)
        pr = np.zeros((case.B, case.d, case.k, case.k), dtype=np.float32)
        for b in range(case.B):
            for j in range(case.d):
                for cp in range(case.k):
                    prev = int(case.ctx[b][-1]) if j == 0 else int(rid[b, j - 1, cp])
                    for c in range(case.k):
                        g = table.get((prev, int(rid[b, j, c])))
                        pr[b, j, cp, c] = case.beta if g is None else g
        want = oracle.tree_from_lists(rid, rlp, B=case.B, d=case.d, k=case.k, W=case.W, lam=case.lam,
                                      beta=case.beta, ngram=ng, ctx=case.ctx, lib=lib)
        got = oracle.tree_from_pairs(rid, rlp, pr, B=case.B, d=case.d, k=case.k, W=case.W,
                                     lam=case.lam, lib=lib)
        for key in ("tokens", "parents", "pos", "mask"):
            if not np.array_equal(got[key], want[key]):
                return False
        if np.abs(got["scores"] - want["scores"]).max() > 1e-12:
            return False
        # 3: lambda = 0
        plain = oracle.tree_from_lists(rid, rlp, B=case.B, d=case.d, k=case.k, W=case.W, lam=0.0,
                                       beta=0.0, ngram=None, ctx=None, lib=lib)
        zero = oracle.tree_from_pairs(rid, rlp, pr, B=case.B, d=case.d, k=case.k, W=case.W, lam=0.0,
                                      lib=lib)
        for key in ("tokens", "parents", "pos", "mask", "scores"):
            if not np.array_equal(zero[key], plain[key]):
                return False
    return True


def greedy_ok(lib=None) -> bool:
    """T = 0 rows against the closed form of logits ln 4, ln 2, 0, 0 and the
    whole path at T = 0 against the enumeration."""
    import math
    import oracle
    ln2 = math.log(2.0)
    z = np.array([[0.0, 2 * ln2, 0.0, ln2]], dtype=np.float32)
    ids, logp, lse = oracle.rows(z, "f32", 4, 0.0, 4, lib=lib)
    if ids[0].tolist() != [1, 3, 0, 2]:
        return False
    if np.abs(logp[0] - np.array([-ln2, -2 * ln2, -3 * ln2, -3 * ln2])).max() > 1e-7:
        return False
    if abs(lse[0] - 3 * ln2) > 1e-7:
        return False
    return whole_path_brute_force_ok(lib=lib, seed=6, T=0.0)


def best_sum_subset(scores, M: int):
    """Brute force: the size-M set of nodes with the largest score sum (sets
    compared by their sorted score lists when sums are equal).  For scores that
    never rise along a path this is the best-first verification tree: the M
    largest scores form a set that holds every ancestor of its members."""
    n = len(scores)
    best, best_key = None, None
    for comb in itertools.combinations(range(n), M):
        vals = sorted((scores[i] for i in comb), reverse=True)
        key = (math.fsum(vals), vals)
        if best_key is None or key > best_key:
            best, best_key = comb, key
    return list(best)
