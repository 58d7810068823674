"""Pins of the CPU oracle against things other than itself (no GPU needed).

- worked examples derived by hand (tests/golden/*.json, closed forms);
- exhaustive enumeration of all k^d paths when nothing is pruned (W >= k^d);
- with lambda = 0 the scores separate, so per-depth beam pruning must return
  exactly the best min(W, k^j) sums of the per-depth lists (k-best sums);
- log-softmax against scipy, top-k against numpy lexsort, dtype decoding
  against numpy's conversions, the n-gram model against a Python dict,
  ancestor masks against Python sets, and the invariants of the output
  (parent depth = depth - 1, mask row = ancestors plus self, popcount = depth).
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special

import oracle
import synth
from tests import oracle_refs as R


# ---------------------------------------------------------- worked examples

@pytest.mark.parametrize("name", ["we1_ngram_hits.json", "we2_tie_breaks.json"])
def test_worked_examples(name):
    ex, logits, keys, vals = R.load_worked_example(name)
    ids, logp, lse = oracle.rows(logits, "f32", ex["V"], ex["T"], ex["k"])
    assert ids.tolist() == ex["expect"]["row_ids"]
    ng = oracle.NGram(ex["n"], keys, vals) if len(keys) else None
    out = oracle.tree_from_lists(ids.reshape(1, ex["d"], ex["k"]), logp.reshape(1, ex["d"], ex["k"]),
                                 B=1, d=ex["d"], k=ex["k"], W=ex["W"], lam=ex["lam"],
                                 beta=ex["beta"], ngram=ng,
                                 ctx=np.array([ex["ctx"]], dtype=np.int32))
    e = ex["expect"]
    assert out["tokens"][0].tolist() == e["tokens"]
    assert out["parents"][0].tolist() == e["parents"]
    assert out["pos"][0].tolist() == e["pos"]
    assert out["mask"][0, :, 0].tolist() == e["mask"]
    want = np.array([R.eval_closed_form(s) for s in e["scores"]])
    # logits are float32(ln p): each stored logit is within 2^-24 relative of ln p
    np.testing.assert_allclose(out["scores"][0], want, rtol=0, atol=1e-6)


def test_worked_example_through_full_pipeline():
    ex, logits, keys, vals = R.load_worked_example("we1_ngram_hits.json")
    case = synth.Case(name="we1", B=1, d=ex["d"], V=ex["V"], dtype="f32", T=ex["T"], k=ex["k"],
                      W=ex["W"], n=ex["n"], lam=ex["lam"], beta=ex["beta"], logits=logits,
                      ctx=np.array([ex["ctx"]], dtype=np.int32), ng_keys=keys, ng_vals=vals)
    out = oracle.tree_build(case)
    assert out["tokens"][0].tolist() == ex["expect"]["tokens"]
    assert out["parents"][0].tolist() == ex["expect"]["parents"]
    assert out["mask"][0, :, 0].tolist() == ex["expect"]["mask"]


# ------------------------------------------------------------ row stage

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_rows_against_scipy_and_lexsort(dtype, T):
    case = synth.make_case(B=3, d=2, V=257, dtype=dtype, T=T, k=7, W=4, n=0, M=0, lam=0, beta=0,
                           recipe=("normal", 3.0), seed=11)
    z = R.decode_np(case.logits, dtype).reshape(-1, 257)
    ids, logp, lse = oracle.rows(case.logits, dtype, 257, T, 7)
    for r in range(z.shape[0]):
        ref = scipy.special.log_softmax(z[r] / T)
        want_ids = R.topk_lexsort(z[r], 7)
        assert ids[r].tolist() == want_ids.tolist()
        np.testing.assert_allclose(logp[r], ref[want_ids], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r], scipy.special.logsumexp(z[r] / T), rtol=0, atol=1e-12)
        # each softmax sums to one
        assert abs(np.exp(z[r] / T - lse[r]).sum() - 1.0) < 1e-12


def test_rows_ties_constant_and_special_values():
    V, k = 40, 9
    z = np.zeros((3, V), dtype=np.float32)
    z[0] = 1.5                                   # constant row: p = -ln V, ids 0..k-1
    z[1] = np.repeat(np.arange(8, dtype=np.float32), 5)  # blocks of 5 equal values
    z[2, :] = -3.0
    z[2, 17] = 0.0
    z[2, 3] = -0.0                               # -0.0 == +0.0: lower id (3) first
    ids, logp, lse = oracle.rows(z, "f32", V, 1.0, k)
    assert ids[0].tolist() == list(range(k))
    np.testing.assert_allclose(logp[0], -math.log(V), atol=1e-13)
    assert ids[1].tolist() == [35, 36, 37, 38, 39, 30, 31, 32, 33]
    assert ids[2].tolist()[:2] == [3, 17]
    np.testing.assert_allclose(logp[2][0], logp[2][1], atol=0)


def test_greedy_rows_closed_form():
    """T = 0 (greedy decoding, DART Figure 2 caption): candidates come from the
    raw logits and the scores are log_softmax(z).  Logits ln 4, ln 2, 0, 0
    give probabilities 1/2, 1/4, 1/8, 1/8, so the log-probabilities are -ln 2,
    -2 ln 2, -3 ln 2, -3 ln 2 and the log-sum-exp is ln 8."""
    ln2 = math.log(2.0)
    z = np.array([[0.0, 2 * ln2, 0.0, ln2], [3.0, 3.0, 3.0, 3.0]], dtype=np.float64)
    ids, logp, lse = oracle.rows(z.astype(np.float32), "f32", 4, 0.0, 4)
    assert ids[0].tolist() == [1, 3, 0, 2]
    zf = z.astype(np.float32).astype(np.float64)   # the stored logits, rounded to float32
    want = zf[0] - math.log(np.exp(zf[0]).sum())
    np.testing.assert_allclose(logp[0], want[[1, 3, 0, 2]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(logp[0], [-ln2, -2 * ln2, -3 * ln2, -3 * ln2], rtol=0, atol=1e-7)
    np.testing.assert_allclose(lse[0], 3 * ln2, rtol=0, atol=1e-7)
    assert ids[1].tolist() == [0, 1, 2, 3]           # a constant row: uniform, ids in order
    np.testing.assert_allclose(logp[1], -math.log(4.0), rtol=0, atol=1e-15)
    with pytest.raises(ValueError):
        oracle.rows(z.astype(np.float32), "f32", 4, -1.0, 2)


def test_greedy_tree_against_brute_force():
    """The whole path at T = 0 against scipy and an enumeration of every path."""
    for seed in (6, 7):
        assert R.whole_path_brute_force_ok(seed=seed, T=0.0)


def test_greedy_first_nodes_form_the_argmax_chain():
    """With lambda = 0 the best child of a depth extends the best node of the
    previous one by that depth's argmax, so node 0 of every depth lies on the
    argmax chain (ties excluded by continuous logits)."""
    case = synth.make_case(B=3, d=5, V=300, dtype="f32", T=0.0, k=4, W=6, n=0, M=0, lam=0.0,
                           beta=0.0, recipe=("normal", 3.0), seed=21)
    out = oracle.tree_build(case)
    z = case.logits.reshape(case.B, case.d, case.V).astype(np.float64)
    for b in range(case.B):
        pos, par, tok = out["pos"][b], out["parents"][b], out["tokens"][b]
        first = [int(np.flatnonzero(pos == j + 1)[0]) for j in range(case.d)]
        assert [int(tok[x]) for x in first] == [int(np.argmax(z[b, j])) for j in range(case.d)]
        assert [int(par[x]) for x in first] == [-1] + first[:-1]


def test_pair_scored_trees():
    """Caller-supplied pair scores in place of the n-gram model (DARTree,
    Method / Tree Construction: children scored by a head in one batch)."""
    assert R.pair_trees_ok()


def test_decode_all_16bit_patterns():
    pat = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    np.seterr(invalid="ignore")
    lib = oracle.load()
    for dtype, ref in (("f16", pat.view(np.float16).astype(np.float64)),
                       ("bf16", (pat.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64))):
        code = oracle.DTYPES[dtype]
        got = np.array([lib.oracle_decode(pat.ctypes.data, code, i) for i in range(1 << 16)])
        finite = np.isfinite(ref)
        np.testing.assert_array_equal(got[finite], ref[finite])
        assert np.array_equal(np.isnan(got), np.isnan(ref))
        assert np.array_equal(np.isinf(got), np.isinf(ref))


# ----------------------------------------------------------- n-gram model

def test_ngram_model_against_dict():
    rng = np.random.default_rng(5)
    for n in (2, 3, 4):
        keys = rng.integers(0, 50, size=(3000, n)).astype(np.int32)  # many repeats
        vals = rng.uniform(-9, -1, size=3000).astype(np.float32)
        ref = R.dict_ngram(keys, vals)
        ng = oracle.NGram(n, keys, vals)
        q = np.concatenate([keys[::7], rng.integers(0, 60, size=(2000, n)).astype(np.int32)])
        got, found = ng.lookup(q)
        for row, v, f in zip(map(tuple, q.tolist()), got, found):
            assert f == (row in ref)
            if f:
                assert float(v) == ref[row]


# ---------------------------------------------------- exhaustive enumeration

def _random_lists(rng, d, k, V, distinct=True):
    ids = np.stack([rng.choice(V, size=k, replace=False) for _ in range(d)]).astype(np.int32)
    logp = np.sort(rng.uniform(-6, -0.1, size=(d, k)), axis=1)[:, ::-1].copy()
    return ids, logp


@pytest.mark.parametrize("n,lam", [(2, 0.5), (3, 0.3), (4, 0.25), (3, 0.0)])
def test_no_pruning_keeps_every_path(n, lam):
    """W >= k^d: the tree is every path, each scored from its own sequence."""
    rng = np.random.default_rng(100 + n)
    d, k, V = 3, 3, 12
    W = k ** d
    for trial in range(4):
        ids, logp = _random_lists(rng, d, k, V)
        ctx = rng.integers(0, V, size=(n - 1,)).astype(np.int32)
        # a table holding about half of all n-grams over this small vocabulary
        allk = np.array(list(itertools.product(range(V), repeat=n)), dtype=np.int32)
        keep = rng.random(allk.shape[0]) < 0.5
        keys = allk[keep]
        vals = rng.uniform(-8, -0.5, size=keys.shape[0]).astype(np.float32)
        ng = oracle.NGram(n, keys, vals)
        out = oracle.tree_from_lists(ids[None], logp[None], B=1, d=d, k=k, W=W, lam=lam,
                                     beta=-11.0, ngram=ng, ctx=ctx[None])
        ref = R.brute_force_paths(ids.tolist(), logp.tolist(), lam=lam, beta=-11.0,
                                  table=R.dict_ngram(keys, vals), n=n, ctx=ctx.tolist())
        paths = R.node_paths(out["tokens"][0].tolist(), out["parents"][0].tolist(), ids.tolist())
        assert sorted(paths) == sorted(ref.keys())          # every path exactly once
        for x, p in enumerate(paths):
            assert abs(out["scores"][0, x] - ref[p]) < 1e-12
            assert out["pos"][0, x] == len(p)
        # nodes of a depth are ordered by (score desc, parent asc, token asc)
        sc, par, tok, pos = (out["scores"][0], out["parents"][0], out["tokens"][0], out["pos"][0])
        for j in range(1, d + 1):
            idx = np.where(pos == j)[0]
            keyed = [(-sc[x], par[x], tok[x]) for x in idx]
            assert keyed == sorted(keyed)


@pytest.mark.parametrize("d,k,W", [(4, 3, 5), (5, 4, 7), (6, 8, 10), (3, 16, 32), (4, 5, 1)])
def test_lambda_zero_is_exact_k_best_sums(d, k, W):
    """Separable scores: per-depth pruning returns the exact best sums at every depth."""
    rng = np.random.default_rng(d * 100 + k)
    for trial in range(3):
        ids, logp = _random_lists(rng, d, k, 64)
        out = oracle.tree_from_lists(ids[None], logp[None], B=1, d=d, k=k, W=W, lam=0.0,
                                     beta=-1.0, ngram=None, ctx=None)
        for j in range(1, d + 1):
            sums = np.zeros(1)
            for jj in range(j):
                sums = (sums[:, None] + logp[jj][None, :]).reshape(-1)
            want = np.sort(sums)[::-1][:min(W, k ** j)]
            got = out["scores"][0][out["pos"][0] == j]
            np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_whole_path_at_temperature_against_brute_force():
    """oracle.tree_build at T = 0.7, W = k^d: scores from scipy log_softmax + enumeration."""
    for seed in (3, 4, 5):
        assert R.whole_path_brute_force_ok(seed=seed)


# --------------------------------------------------------- output invariants

@pytest.mark.parametrize("cfg", [0])
def test_invariants_on_config0(cfg):
    case = synth.make_config(cfg, seed=3)
    out = oracle.tree_build(case)
    _check_invariants(case, out)


def test_invariants_on_reduced_configs():
    for i, over in [(1, dict(V=4096, M=1 << 12)), (2, dict(B=3, V=3001, M=1 << 14)),
                    (3, dict(B=5, V=2000, M=1 << 13)), (4, dict(B=2, V=5003, M=1 << 15))]:
        case = synth.make_config(i, seed=1, **over)
        out = oracle.tree_build(case)
        _check_invariants(case, out)


def _check_invariants(case, out):
    B, d, k, W = case.B, case.d, case.k, case.W
    N = oracle.num_nodes(d, k, W)
    widths = [min(W, k ** j) for j in range(1, d + 1)]
    assert N == sum(widths)
    ng = out["ngram"]
    table = None
    for b in range(B):
        tok, par, pos, sc = (out["tokens"][b], out["parents"][b], out["pos"][b], out["scores"][b])
        sets = R.masks_from_sets(par.tolist())
        start = 0
        for j, wj in enumerate(widths):
            idx = np.arange(start, start + wj)
            assert (pos[idx] == j + 1).all()
            assert set(tok[idx].tolist()) <= set(out["row_ids"][b, j].tolist())
            if j == 0:
                assert (par[idx] == -1).all()
            else:
                assert (pos[par[idx]] == j).all()
            assert (np.diff(sc[idx]) <= 0).all()
            start += wj
        for x in range(N):
            assert R.mask_row_to_set(out["mask"][b, x]) == sets[x]
            assert len(sets[x]) == pos[x]
            # score = parent score + increment drawn from the row's candidate list
            p = par[x]
            ps = 0.0 if p < 0 else sc[p]
            j = pos[x] - 1
            c = list(out["row_ids"][b, j]).index(tok[x])
            inc = out["row_logp"][b, j, c]
            if ng is not None:
                seq = list(case.ctx[b]) + _path_tokens(tok, par, x)
                context = seq[len(seq) - case.n:len(seq) - 1]
                v, f = ng.lookup(np.array(context + [tok[x]], dtype=np.int32)[None])
                inc = inc + case.lam * (float(v[0]) if f[0] else case.beta)
            assert abs(sc[x] - (ps + inc)) < 1e-12


def _path_tokens(tok, par, x):
    seq = []
    while x >= 0:
        seq.append(int(tok[x]))
        x = par[x]
    return seq[::-1]
