"""Plant plausible mistakes in copies of oracle.c and check that the pins catch each one.

Every mutant is a one-line edit of the oracle source (a dropped term, a wrong
sign, a reversed tie-break, an off-by-one context window, a wrong index ...),
compiled into a temporary library on the CPU.  (Dropping T from the running
maximum alone is not listed: the maximum is only a stabilising shift, so that
edit leaves every result unchanged in exact arithmetic.)  The pin suite below reuses the
independent references of test_oracle_pins; a mutant that passes every pin
would mean the pins cannot see that kind of mistake.
"""
import itertools
import os
import shutil
import tempfile

import numpy as np
import pytest
import scipy.special

import oracle
import synth
from tests import oracle_refs as R

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "no_temperature_in_sum": ("S += exp(work[v].z / T - m);", "S += exp(work[v].z - m);"),
    "logp_sign": ("logp[r * k + c] = work[c].z / T - l;", "logp[r * k + c] = work[c].z / T + l;"),
    "lse_drops_max": ("double l = m + log(S);", "double l = log(S);"),
    "row_ties_high_id_first": ("    return (a->id > b->id) - (a->id < b->id);\n}\n\nstatic void one_row",
                               "    return (a->id < b->id) - (a->id > b->id);\n}\n\nstatic void one_row"),
    "rows_ascending": ("    if (a->z > b->z) return -1;\n    if (a->z < b->z) return 1;",
                       "    if (a->z < b->z) return -1;\n    if (a->z > b->z) return 1;"),
    "lambda_dropped": ("cand[m].key = Z * invT + lam * G;", "cand[m].key = Z * invT + G;"),
    "temperature_dropped_in_key": ("cand[m].key = Z * invT + lam * G;", "cand[m].key = Z + lam * G;"),
    "ngram_not_accumulated": ("double G = fG[i];", "double G = 0.0;"),
    "row_offsets_dropped": ("if (off) Lsum = Lsum + off[(size_t)b * d + j];", "if (off) Lsum = off[(size_t)b * d + j];"),
    "beta_unscaled": ("(double)g : beta;", "(double)g : beta / lam;"),
    "context_off_by_one": ("key[q] = seq[len - (n - 1) + q];", "key[q] = seq[len - n + q];"),
    "parent_ties_reversed": ("return a->i < b->i ? -1 : 1;", "return a->i < b->i ? 1 : -1;"),
    "token_ties_reversed": ("return (a->tok > b->tok) - (a->tok < b->tok);",
                            "return (a->tok < b->tok) - (a->tok > b->tok);"),
    "parent_is_rank": ("parents[(size_t)b * N + node] = fnode[e->i];",
                       "parents[(size_t)b * N + node] = e->i;"),
    "depth_off_by_one": ("pos[(size_t)b * N + node] = j + 1;", "pos[(size_t)b * N + node] = j;"),
    "keeps_the_worst": ("const cand_t* e = &cand[r];", "const cand_t* e = &cand[m - 1 - r];"),
    "mask_without_self": ("int a = x, steps = 0;", "int a = parents[(size_t)b * N + x], steps = 0;"),
    "ngram_last_value_wins": ("    return (a->order > b->order) - (a->order < b->order);",
                              "    return (a->order < b->order) - (a->order > b->order);"),
    "bf16_decode_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "f16_exponent_bias": ("v = ldexp((double)(m + 1024), e - 25);", "v = ldexp((double)(m + 1024), e - 24);"),
    "path_not_extended": ("nseq[(size_t)r * L + len] = e->tok;", "nseq[(size_t)r * L + len] = 0;"),
    "parent_score_dropped": ("double Z = fZ[i] + P[c];", "double Z = P[c];"),
    "cut_at_w_minus_one": ("int keep = m < W ? m : W;", "int keep = m < W - 1 ? m : W - 1;"),
    "select_worst_first": ("if (s[a] != s[b]) return s[a] > s[b];", "if (s[a] != s[b]) return s[a] < s[b];"),
    "select_ties_high_index": ("    return a < b;\n}", "    return a > b;\n}"),
    "select_all_available": ("if (par[i] < 0) avail[na++] = i;", "avail[na++] = i;"),
    "greedy_as_small_temperature": ("return T == 0.0 ? 1.0 : T;", "return T == 0.0 ? 1e-3 : T;"),
    "pair_uses_child_column": ("pair[(((size_t)b * d + j) * k + fcol[i]) * k + c]",
                               "pair[(((size_t)b * d + j) * k + c) * k + c]"),
    "pair_column_not_carried": ("ncol[r] = e->col;", "ncol[r] = 0;"),
    "pair_depth_ignored": ("pair[(((size_t)b * d + j) * k + fcol[i]) * k + c]",
                           "pair[(((size_t)b * d + 0) * k + fcol[i]) * k + c]"),
    "select_parent_not_renumbered": ("new_parents[(size_t)b * Mp + j] = par[i] < 0 ? -1 : newpos[par[i]];",
                                     "new_parents[(size_t)b * Mp + j] = par[i];"),
}


# ----------------------------------------------------------- the pin suite

def _pin_worked_examples(lib):
    for name in ("we1_ngram_hits.json", "we2_tie_breaks.json"):
        ex, logits, keys, vals = R.load_worked_example(name)
        ids, logp, _ = oracle.rows(logits, "f32", ex["V"], ex["T"], ex["k"], lib=lib)
        if ids.tolist() != ex["expect"]["row_ids"]:
            return False
        ng = oracle.NGram(ex["n"], keys, vals, lib=lib) if len(keys) else None
        out = oracle.tree_from_lists(ids.reshape(1, ex["d"], ex["k"]), logp.reshape(1, ex["d"], ex["k"]),
                                     B=1, d=ex["d"], k=ex["k"], W=ex["W"], lam=ex["lam"],
                                     beta=ex["beta"], ngram=ng,
                                     ctx=np.array([ex["ctx"]], dtype=np.int32), lib=lib)
        e = ex["expect"]
        want = np.array([R.eval_closed_form(s) for s in e["scores"]])
        if (out["tokens"][0].tolist() != e["tokens"] or out["parents"][0].tolist() != e["parents"]
                or out["pos"][0].tolist() != e["pos"] or out["mask"][0, :, 0].tolist() != e["mask"]
                or np.abs(out["scores"][0] - want).max() > 1e-6):
            return False
    return True


def _pin_rows(lib):
    for dtype, T in (("f32", 0.7), ("f16", 1.0), ("bf16", 2.5)):
        case = synth.make_case(B=2, d=2, V=129, dtype=dtype, T=T, k=5, W=4, n=0, M=0, lam=0,
                               beta=0, recipe=("ties", 6), seed=4)
        z = R.decode_np(case.logits, dtype).reshape(-1, 129)
        ids, logp, lse = oracle.rows(case.logits, dtype, 129, T, 5, lib=lib)
        for r in range(z.shape[0]):
            ref = scipy.special.log_softmax(z[r] / T)
            want = R.topk_lexsort(z[r], 5)
            if ids[r].tolist() != want.tolist() or np.abs(logp[r] - ref[want]).max() > 1e-12:
                return False
            if abs(lse[r] - scipy.special.logsumexp(z[r] / T)) > 1e-12:
                return False
    # decoding of every finite 16-bit pattern against numpy
    pat = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    np.seterr(invalid="ignore")
    for dtype, ref in (("f16", pat.view(np.float16).astype(np.float64)),
                       ("bf16", (pat.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64))):
        sel = np.nonzero(np.isfinite(ref))[0][::97]
        got = np.array([lib.oracle_decode(pat.ctypes.data, oracle.DTYPES[dtype], int(i)) for i in sel])
        if not np.array_equal(got, ref[sel]):
            return False
    return True


def _pin_brute_force(lib):
    rng = np.random.default_rng(7)
    d, k, V = 3, 3, 10
    for n, lam in ((2, 0.5), (3, 0.3)):
        ids = np.stack([rng.choice(V, size=k, replace=False) for _ in range(d)]).astype(np.int32)
        logp = np.sort(rng.uniform(-6, -0.1, size=(d, k)), axis=1)[:, ::-1].copy()
        ctx = rng.integers(0, V, size=(n - 1,)).astype(np.int32)
        allk = np.array(list(itertools.product(range(V), repeat=n)), dtype=np.int32)
        keys = allk[rng.random(allk.shape[0]) < 0.5]
        vals = rng.uniform(-8, -0.5, size=keys.shape[0]).astype(np.float32)
        # repeated keys: the first value must win
        keys = np.concatenate([keys, keys[:50]])
        vals = np.concatenate([vals, vals[:50] - 1.0]).astype(np.float32)
        ng = oracle.NGram(n, keys, vals, lib=lib)
        try:
            out = oracle.tree_from_lists(ids[None], logp[None], B=1, d=d, k=k, W=k ** d, lam=lam,
                                         beta=-11.0, ngram=ng, ctx=ctx[None], lib=lib)
        except ValueError:
            return False
        ref = R.brute_force_paths(ids.tolist(), logp.tolist(), lam=lam, beta=-11.0,
                                  table=R.dict_ngram(keys, vals), n=n, ctx=ctx.tolist())
        try:
            paths = R.node_paths(out["tokens"][0].tolist(), out["parents"][0].tolist(), ids.tolist())
        except (ValueError, IndexError):
            return False
        if sorted(paths) != sorted(ref.keys()):
            return False
        for x, p in enumerate(paths):
            if abs(out["scores"][0, x] - ref[p]) > 1e-12 or out["pos"][0, x] != len(p):
                return False
        sc, par, tok, pos = (out["scores"][0], out["parents"][0], out["tokens"][0], out["pos"][0])
        for j in range(1, d + 1):
            idx = np.where(pos == j)[0]
            keyed = [(-sc[x], par[x], tok[x]) for x in idx]
            if keyed != sorted(keyed):
                return False
        sets = R.masks_from_sets(par.tolist())
        for x in range(len(tok)):
            if R.mask_row_to_set(out["mask"][0, x]) != sets[x]:
                return False
    return True


def _pin_k_best(lib):
    rng = np.random.default_rng(9)
    d, k, W = 4, 4, 6
    ids = np.stack([rng.choice(50, size=k, replace=False) for _ in range(d)]).astype(np.int32)
    logp = np.sort(rng.uniform(-6, -0.1, size=(d, k)), axis=1)[:, ::-1].copy()
    try:
        out = oracle.tree_from_lists(ids[None], logp[None], B=1, d=d, k=k, W=W, lam=0.0, beta=-1.0,
                                     ngram=None, ctx=None, lib=lib)
    except ValueError:
        return False
    for j in range(1, d + 1):
        sums = np.zeros(1)
        for jj in range(j):
            sums = (sums[:, None] + logp[jj][None, :]).reshape(-1)
        want = np.sort(sums)[::-1][:min(W, k ** j)]
        got = out["scores"][0][out["pos"][0] == j]
        if got.shape != want.shape or np.abs(got - want).max() > 1e-12:
            return False
    return True


def _pin_whole_path_temperature(lib):
    return R.whole_path_brute_force_ok(lib)


def _pin_select(lib):
    import json
    with open(os.path.join(R.GOLDEN, "we1_select.json")) as f:
        ex = json.load(f)
    t = ex["tree"]
    sc = np.array([[R.eval_closed_form(x) for x in t["scores"]]])
    for M, want in ex["expect"].items():
        out = oracle.select_tree(np.array([t["tokens"]]), np.array([t["parents"]]), np.array([t["pos"]]), sc,
                                 int(M), lib=lib)
        if out["index"][0].tolist() != want["index"] or out["parents"][0].tolist() != want["parents"]:
            return False
    # availability: a child that outscores everything waits for its parent
    out = oracle.select_tree(np.array([[7, 8, 9]]), np.array([[-1, -1, 1]]), np.array([[1, 1, 2]]),
                             np.array([[-5.0, -6.0, -1.0]]), 2, lib=lib)
    if out["index"][0].tolist() != [0, 1]:
        return False
    # renumbering: node 0 is not taken, so node 2's parent (node 1) becomes position 0
    out = oracle.select_tree(np.array([[4, 5, 6]]), np.array([[-1, -1, 1]]), np.array([[1, 1, 2]]),
                             np.array([[-9.0, -1.0, -2.0]]), 2, lib=lib)
    if out["index"][0].tolist() != [1, 2] or out["parents"][0].tolist() != [-1, 0] or \
            out["mask"][0, :, 0].tolist() != [1, 3]:
        return False
    # equal scores: lower index first
    out = oracle.select_tree(np.arange(3)[None], np.array([[-1, -1, -1]]), np.ones((1, 3), dtype=np.int32),
                             np.array([[-1.0, -1.0, -2.0]]), 1, lib=lib)
    if out["index"][0].tolist() != [0]:
        return False
    for seed in (1, 2):
        tree = synth.make_candidate_trees(B=1, d=3, k=2, W=4, seed=200 + seed, tie_frac=0.0, zero_frac=0.0)
        N = tree["parents"].shape[1]
        for M in range(1, N + 1):
            out = oracle.select_tree(tree["tokens"], tree["parents"], tree["pos"], tree["scores"], M, lib=lib)
            if out["index"][0].tolist() != sorted(R.best_sum_subset(tree["scores"][0].astype(np.float64).tolist(), M)):
                return False
    return True


def _pin_pairs(lib):
    return R.pair_trees_ok(lib=lib)


def _pin_greedy(lib):
    return R.greedy_ok(lib=lib)


PINS = [_pin_worked_examples, _pin_rows, _pin_brute_force, _pin_k_best, _pin_whole_path_temperature, _pin_select,
        _pin_pairs, _pin_greedy]


def _all_pins_pass(lib) -> bool:
    for pin in PINS:
        try:
            if not pin(lib):
                return False
        except ValueError:
            return False
    return True


def test_unmutated_oracle_passes_the_suite():
    assert _all_pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in oracle.c"
    tmp = tempfile.mkdtemp(prefix="oracle_mut_")
    try:
        path = os.path.join(tmp, "oracle.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.build(force=True, src=path, out=os.path.join(tmp, "lib.so")))
        assert not _all_pins_pass(lib), f"mutant {name} passes every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
