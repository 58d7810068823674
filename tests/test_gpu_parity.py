"""CUDA path against the oracle, through the C ABI (needs a GB300).

Row stage: candidate ids bit-exact, log-probabilities and log-sum-exp within
1e-5.  Tree stage fed the oracle's own candidate lists: everything bit-exact,
scores included (both sides accumulate the same double-precision key in the
same order).  Whole path: bit-exact tokens / parents / depths / masks and
scores within 1e-5 (the exemption for oracle near-ties is in parity.py; the
full-size test requires every tree to match exactly).
"""
import ctypes
import dataclasses

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


def _np(t):
    return t.cpu().numpy()


# ------------------------------------------------------------------ rows

ROW_CASES = [
    # dtype, V, T, k, rows, recipe
    ("f32", 1024, 1.0, 4, 4, ("normal", 2.0)),
    ("bf16", 151936, 1.0, 8, 8, ("normal_spike", 3.0, 12.0)),
    ("bf16", 151936, 0.7, 8, 24, ("normal_zipf", 3.0, 1.1)),
    ("f16", 32000, 1.0, 10, 64, ("normal_spike", 2.5, 10.0)),
    ("bf16", 151936, 1.0, 16, 40, ("gumbel_zipf", 4.0, 1.2)),
    ("bf16", 1001, 1.3, 7, 37, ("normal", 3.0)),         # rows not 16-byte aligned
    ("f16", 777, 0.5, 32, 19, ("normal", 2.0)),
    ("f32", 33, 1.0, 5, 50, ("normal", 1.0)),
    ("f32", 7777, 1.7, 16, 64, ("gumbel_zipf", 4.0, 1.2)),  # unaligned rows over several warps
    ("f32", 2, 1.0, 1, 3, ("normal", 1.0)),
    ("bf16", 4099, 1.0, 32, 11, ("ties", 3)),            # many exact ties
    ("f16", 3000, 2.0, 9, 6, ("const", 0.25)),           # constant rows
    ("bf16", 1 << 20, 1.0, 12, 3, ("normal", 3.0)),      # one row over many warps
]


@pytest.mark.parametrize("dtype,V,T,k,rows,recipe", ROW_CASES)
def test_row_topk_matches_oracle(D, dtype, V, T, k, rows, recipe):
    case = synth.make_case(B=rows, d=1, V=V, dtype=dtype, T=T, k=k, W=1, n=0, M=0, lam=0, beta=0,
                           recipe=recipe, seed=V + rows)
    z = parity.to_device(case).reshape(rows, V)
    ids, logp, lse, ws = D.row_topk(z, case.T, k)
    assert D.device_error(ws) == 0
    rid, rlp, rlse = oracle.rows(case.logits, dtype, V, case.T, k)
    np.testing.assert_array_equal(_np(ids), rid)
    np.testing.assert_allclose(_np(logp), rlp, rtol=0, atol=1e-5)
    np.testing.assert_allclose(_np(lse), rlse, rtol=0, atol=1e-5)


def test_row_topk_softmax_sums_to_one(D):
    case = synth.make_config(2, seed=4, B=2, M=0, n=0)
    R, V = case.B * case.d, case.V
    z = parity.to_device(case).reshape(R, V)
    _, _, lse, _ = D.row_topk(z, case.T, case.k)
    x = z.double() / case.T
    total = torch.exp(x - lse.double()[:, None]).sum(dim=1)
    assert (total - 1).abs().max().item() < 1e-5


def test_row_topk_negative_zero_and_inf(D):
    V = 64
    z = torch.full((2, V), -3.0, dtype=torch.float32)
    z[0, 9] = 0.0
    z[0, 4] = -0.0            # equal to +0.0: lower id first
    z[1, :] = float("-inf")   # masked vocabulary ...
    z[1, 40] = 1.0            # ... with one finite logit
    ids, logp, lse, ws = D.row_topk(z.cuda(), 1.0, 3)
    assert _np(ids)[0].tolist() == [4, 9, 0]
    assert _np(ids)[1].tolist()[0] == 40
    assert _np(ids)[1].tolist()[1:] == [0, 1]
    assert abs(float(_np(logp)[1, 0])) < 1e-6


# ------------------------------------------------------- tree stage alone

TREE_CASES = [
    # B, d, k, W, n, lam
    (3, 4, 4, 4, 2, 0.5),
    (5, 8, 8, 10, 3, 0.3),
    (4, 8, 10, 16, 2, 0.5),
    (2, 16, 16, 32, 4, 0.25),
    (2, 16, 32, 64, 3, 0.1),      # N = 992, 64-key runs
    (3, 6, 5, 50, 2, 0.0),        # W = 50
    (4, 1, 7, 3, 2, 0.7),         # one depth
    (4, 5, 1, 1, 2, 0.5),         # a chain
    (3, 3, 3, 27, 3, 0.4),        # W = k^d: nothing pruned
    (2, 5, 6, 8, 0, 0.0),         # no n-gram table
]


@pytest.mark.parametrize("B,d,k,W,n,lam", TREE_CASES)
def test_tree_from_topk_bit_exact(D, B, d, k, W, n, lam):
    V = 5000
    case = synth.make_case(B=B, d=d, V=V, dtype="bf16", T=1.0, k=k, W=W, n=n,
                           M=(1 << 14) if n else 0, lam=lam, beta=-12.0, recipe=("normal_spike", 3.0, 8.0),
                           seed=B * 100 + d)
    rid, rlp, _ = oracle.rows(case.logits, "bf16", V, 1.0, k)
    rid = rid.reshape(B, d, k)
    rlp = rlp.reshape(B, d, k)
    ng = oracle.NGram(n, case.ng_keys, case.ng_vals) if n else None
    ref = oracle.tree_from_lists(rid, rlp, B=B, d=d, k=k, W=W, lam=case.lam, beta=case.beta, ngram=ng,
                                 ctx=case.ctx if n else None)
    tab, ctx = parity.gpu_table(case)
    out = D.tree_from_topk(torch.from_numpy(rid).cuda(), torch.from_numpy(rlp).cuda(), W, case.lam,
                           case.beta, table=tab, ctx=ctx)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(out["tokens"]), ref["tokens"])
    np.testing.assert_array_equal(_np(out["parents"]), ref["parents"])
    np.testing.assert_array_equal(_np(out["pos"]), ref["pos"])
    np.testing.assert_array_equal(_np(out["mask"]).view(np.uint32), ref["mask"])
    np.testing.assert_array_equal(_np(out["scores"]), ref["scores"].astype(np.float32))


# -------------------------------------------------------------- whole path

def _run_full(D, case, scores=True):
    z = parity.to_device(case)
    tab, ctx = parity.gpu_table(case)
    out = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx,
                       scores=scores)
    assert D.device_error(out["workspace"]) == 0
    return {key: _np(v) for key, v in out.items() if key != "workspace" and v is not None}


@pytest.mark.parametrize("cfg,over", [
    (0, {}),
    (1, dict(V=20000, M=1 << 14)),
    (2, dict(B=6, M=1 << 16)),
    (3, dict(B=24, M=1 << 16)),
    (4, dict(B=3, M=1 << 18)),
    (4, dict(B=3, M=1 << 18, lam=0.0)),                 # bf16 sums: many exact ties
    (2, dict(B=5, V=30011, M=1 << 14, dtype="f16")),   # ragged rows
    (4, dict(B=4, V=7777, M=1 << 14, dtype="f32", T=1.7)),
])
@pytest.mark.parametrize("seed", [0, 1])
def test_tree_build_matches_oracle(D, cfg, over, seed):
    case = synth.make_config(cfg, seed=seed, **over)
    got = _run_full(D, case)
    ref = oracle.tree_build(case)
    stats = parity.compare_all(case, got, ref, ref["ngram"])
    assert stats["exact"] == case.B


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_tree_build_full_size(D, cfg):
    """Full workload sizes, same call the benchmark times; every tree compared."""
    case = synth.make_config(cfg, seed=0)
    got = _run_full(D, case)
    ref = oracle.tree_build(case)
    stats = parity.compare_all(case, got, ref, ref["ngram"])
    assert stats["exact"] == case.B


def test_worked_example_on_gpu(D):
    from tests import oracle_refs as R
    ex, logits, keys, vals = R.load_worked_example("we1_ngram_hits.json")
    case = synth.Case(name="we1", B=1, d=ex["d"], V=ex["V"], dtype="f32", T=ex["T"], k=ex["k"],
                      W=ex["W"], n=ex["n"], lam=ex["lam"], beta=ex["beta"], logits=logits,
                      ctx=np.array([ex["ctx"]], dtype=np.int32), ng_keys=keys, ng_vals=vals)
    got = _run_full(D, case)
    e = ex["expect"]
    assert got["tokens"][0].tolist() == e["tokens"]
    assert got["parents"][0].tolist() == e["parents"]
    assert got["pos"][0].tolist() == e["pos"]
    assert got["mask"][0, :, 0].tolist() == e["mask"]


def test_no_table_and_no_scores(D):
    case = synth.make_config(2, seed=3, B=3, V=9000, M=0, n=0)
    got = _run_full(D, case, scores=True)
    ref = oracle.tree_build(case, use_table=False)
    stats = parity.compare_all(case, got, ref, None)
    assert stats["exact"] == case.B
    z = parity.to_device(case)
    bare = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, scores=False)
    assert bare["scores"] is None
    assert np.array_equal(_np(bare["tokens"]), got["tokens"])


def test_repeated_calls_are_identical(D):
    case = synth.make_config(3, seed=5, B=16, M=1 << 15)
    z = parity.to_device(case)
    tab, ctx = parity.gpu_table(case)
    b = D.TreeBuilder(case.B, case.d, case.V, z.dtype, case.T, case.k, case.W, case.lam, case.beta,
                      table=tab, ctx=ctx)
    first = {key: v.clone() for key, v in b(z).items() if v is not None}
    for _ in range(3):
        again = b(z)
        for key, v in first.items():
            assert torch.equal(again[key], v)


def _control_clean(ws):
    """The control block (first 256 bytes): no error bits and nothing else written."""
    return not _np(ws[:256]).any()


def test_workspace_serves_repeated_calls(D):
    # the row pass keeps no state between calls beyond the error word: every
    # piece rewrites its slot, so one zero-filled workspace serves every later
    # call (of any row count that fits) without a clearing launch
    big = synth.make_case(B=6, d=1, V=1 << 20, dtype="bf16", T=1.0, k=12, W=1, n=0, M=0, lam=0,
                          beta=0, recipe=("normal", 3.0), seed=11)
    zb = parity.to_device(big).reshape(6, 1 << 20)
    ids, logp, lse, ws = D.row_topk(zb, big.T, 12)
    assert D.device_error(ws) == 0 and _control_clean(ws)
    for _ in range(2):
        ids2, logp2, lse2, _ = D.row_topk(zb, big.T, 12, workspace=ws)
        assert torch.equal(ids2, ids) and torch.equal(logp2, logp) and torch.equal(lse2, lse)
        assert _control_clean(ws)
    small = zb[:2].contiguous()
    ids3, logp3, lse3, _ = D.row_topk(small, big.T, 12, workspace=ws)
    assert torch.equal(ids3, ids[:2]) and torch.equal(lse3, lse[:2])
    assert D.device_error(ws) == 0 and _control_clean(ws)


def test_one_workspace_serves_calls_of_different_shapes(D):
    """One buffer, passed with the same size to calls of different batch,
    vocabulary and element type: the arrival counters sit where no call's
    other data goes, so every call starts from clean counters."""
    cases = [synth.make_config(2, seed=7, B=6, M=1 << 14),
             synth.make_config(0, seed=7),
             synth.make_config(2, seed=8, B=2, M=1 << 14),
             synth.make_config(3, seed=7, B=12, M=1 << 14),
             synth.make_config(4, seed=7, B=2, V=20011, M=1 << 14, dtype="f16"),
             synth.make_config(2, seed=7, B=6, M=1 << 14)]
    need = max(D.workspace_bytes(c.B, c.d, c.V, D.DTYPE_CODES()[parity.to_device(c).dtype], c.k) for c in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for case in cases:
        z = parity.to_device(case)
        tab, ctx = parity.gpu_table(case)
        out = D.tree_build(z, case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx, workspace=ws)
        assert D.device_error(ws) == 0
        got = {key: _np(v) for key, v in out.items() if key != "workspace" and v is not None}
        ref = oracle.tree_build(case)
        assert parity.compare_all(case, got, ref, ref["ngram"])["exact"] == case.B


# ------------------------------------------------------- greedy decoding, T = 0

@pytest.mark.parametrize("cfg,over", [
    (1, dict(V=20000, M=1 << 14)),
    (2, dict(B=6, M=1 << 16)),
    (3, dict(B=24, M=1 << 16)),
    (4, dict(B=3, M=1 << 18)),
])
def test_greedy_tree_build_matches_oracle(D, cfg, over):
    """T = 0 scores with log_softmax(z): the oracle at T = 0 decides, and the
    GPU result equals its own T = 1 result bit for bit."""
    case = synth.make_config(cfg, seed=2, T=0.0, **over)
    got = _run_full(D, case)
    ref = oracle.tree_build(case)
    stats = parity.compare_all(case, got, ref, ref["ngram"])
    assert stats["exact"] == case.B
    one = _run_full(D, dataclasses.replace(case, T=np.float32(1.0)))
    for key in ("tokens", "parents", "pos", "mask", "scores"):
        assert np.array_equal(got[key], one[key]), key


def test_greedy_row_topk(D):
    case = synth.make_case(B=16, d=1, V=151936, dtype="bf16", T=0.0, k=8, W=1, n=0, M=0, lam=0,
                           beta=0, recipe=("normal_spike", 3.0, 12.0), seed=5)
    z = parity.to_device(case).reshape(16, 151936)
    ids, logp, lse, ws = D.row_topk(z, 0.0, 8)
    assert D.device_error(ws) == 0
    rid, rlp, rlse = oracle.rows(case.logits, "bf16", 151936, 0.0, 8)
    np.testing.assert_array_equal(_np(ids), rid)
    np.testing.assert_allclose(_np(logp), rlp, rtol=0, atol=1e-5)
    np.testing.assert_allclose(_np(lse), rlse, rtol=0, atol=1e-5)


def test_batch_of_zero_and_errors(D):
    z = torch.zeros((0, 4, 100), dtype=torch.float32, device="cuda")
    out = D.tree_build(z, 1.0, 4, 4, 0.5, -10.0)
    assert out["tokens"].shape == (0, 16)
    good = torch.randn((2, 3, 100), device="cuda")
    with pytest.raises(D.DartError):
        D.tree_build(good, -1.0, 4, 4, 0.5, -10.0)         # T < 0 (T = 0 is greedy, accepted)
    with pytest.raises(D.DartError):
        D.tree_build(good, 1.0, 101, 4, 0.5, -10.0)        # k > V
    big = torch.randn((2, 3, 101), device="cuda")
    with pytest.raises(D.DartError):
        D.tree_build(big.view(-1)[1:1 + 2 * 3 * 100].view(2, 3, 100), 1.0, 4, 4, 0.5, -10.0)  # misaligned


# ---------------------------------------------------------- masks, lookups

def test_mask_pack_matches_oracle(D):
    rng = np.random.default_rng(0)
    B, N = 3, 1000
    par = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        for x in range(N):
            par[b, x] = -1 if x < 5 else rng.integers(max(-1, x - 40), x)
    got = D.mask_pack(torch.from_numpy(par).cuda())
    ref = oracle.mask_from_parents(par)
    np.testing.assert_array_equal(_np(got).view(np.uint32), ref)


def test_mask_pack_flags_bad_parent(D):
    par = torch.tensor([[-1, 0, 2, 1]], dtype=torch.int32, device="cuda")   # node 2 names itself
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    D.mask_pack(par, device_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 8


def test_ngram_lookup_matches_oracle(D):
    case = synth.make_config(4, seed=2, B=2, V=3000, M=1 << 16)
    tab, _ = parity.gpu_table(case)
    ng = oracle.NGram(case.n, case.ng_keys, case.ng_vals)
    rng = np.random.default_rng(1)
    q = np.concatenate([case.ng_keys[::3], rng.integers(0, case.V, size=(50000, case.n)).astype(np.int32)])
    vals, found = tab.lookup(torch.from_numpy(q).cuda())
    rv, rf = ng.lookup(q)
    np.testing.assert_array_equal(_np(found), rf)
    np.testing.assert_array_equal(_np(vals)[rf], rv[rf])


def test_tree_builder_replays_in_a_cuda_graph(D):
    """The whole path launches no allocation, copy or host synchronisation,
    so a fixed-shape builder call can be captured in a CUDA graph (as a
    decode loop does) and replayed on new logits with results identical to
    eager calls."""
    cases = [synth.make_config(2, seed=s, B=8, M=1 << 14) for s in (40, 41)]
    za, zb = parity.to_device(cases[0]), parity.to_device(cases[1])
    tab, ctx = parity.gpu_table(cases[0])
    c = cases[0]
    b = D.TreeBuilder(c.B, c.d, c.V, za.dtype, c.T, c.k, c.W, c.lam, c.beta, table=tab, ctx=ctx)
    z = za.clone()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        b(z, stream=stream)                      # warm-up outside the capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        b(z, stream=torch.cuda.current_stream())
    for src in (za, zb, za):
        z.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        got = {key: v.clone() for key, v in b.out.items() if v is not None}
        eager = D.tree_build(src, c.T, c.k, c.W, c.lam, c.beta, table=tab, ctx=ctx)
        for key in ("tokens", "parents", "pos", "mask", "scores"):
            assert torch.equal(got[key], eager[key]), key
    assert D.device_error(b.ws) == 0


@pytest.mark.parametrize("cfg,over", [(2, dict(B=8, M=1 << 14)), (4, dict(B=3, M=1 << 16)), (1, dict(V=20000))])
def test_tree_plan_replays_the_whole_path(D, cfg, over):
    """A plan records the path's launches once (dart_tree_plan_create); every
    launch on new logits in the same buffer matches the oracle and, bit for
    bit, a direct dart_tree_build call."""
    cases = [synth.make_config(cfg, seed=s, **over) for s in (50, 51)]
    c = cases[0]
    za, zb = parity.to_device(cases[0]), parity.to_device(cases[1])
    tab, ctx = parity.gpu_table(c)      # one table and context for both batches
    b = D.TreeBuilder(c.B, c.d, c.V, za.dtype, c.T, c.k, c.W, c.lam, c.beta, table=tab, ctx=ctx, graph=True)
    z = za.clone()
    for i, src in enumerate((za, zb, za)):
        z.copy_(src)
        out = b(z)
        torch.cuda.synchronize()
        assert b._plan is not None and b._plan[0] == z.data_ptr()
        eager = D.tree_build(src, c.T, c.k, c.W, c.lam, c.beta, table=tab, ctx=ctx)
        for key in ("tokens", "parents", "pos", "mask", "scores"):
            assert torch.equal(out[key], eager[key]), (i, key)
        if i == 0:
            got = {key: _np(v) for key, v in out.items() if v is not None}
            ref = oracle.tree_build(c)
            assert parity.compare_all(c, got, ref, ref["ngram"])["exact"] == c.B
    assert D.device_error(b.ws) == 0


def test_tree_plan_inside_a_callers_graph(D):
    """Launched into a stream that the caller is capturing, a plan's kernels go
    into the caller's graph, whose replays then give the same trees."""
    c = synth.make_config(2, seed=60, B=4, M=1 << 14)
    z = parity.to_device(c)
    tab, ctx = parity.gpu_table(c)
    b = D.TreeBuilder(c.B, c.d, c.V, z.dtype, c.T, c.k, c.W, c.lam, c.beta, table=tab, ctx=ctx, graph=True)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        b(z, stream=stream)                      # records the plan, outside any capture
    stream.synchronize()
    first = {key: v.clone() for key, v in b.out.items() if v is not None}
    for v in b.out.values():
        if v is not None:
            v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        rc = D.lib().dart_tree_plan_launch(b._plan[1], ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    graph.replay()
    torch.cuda.synchronize()
    for key, v in first.items():
        assert torch.equal(b.out[key], v), key
    assert D.device_error(b.ws) == 0


@pytest.mark.parametrize("shape", [
    dict(B=2, d=32, V=300, k=32, W=32, n=4, M=2000),   # N = 1024 nodes (the limit), 32 mask words per row
    dict(B=3, d=32, V=97, k=2, W=32, n=2, M=2000),     # 32 depths of two candidates, W reached at depth 5
    dict(B=4, d=1, V=2, k=2, W=1, n=2, M=2),           # the smallest vocabulary, one depth, one survivor
    dict(B=2, d=3, V=5, k=5, W=64, n=3, M=40),         # k = V: every token is a candidate, nothing pruned
])
def test_whole_path_at_the_size_limits(D, shape):
    case = synth.make_case(dtype="bf16", T=0.9, lam=0.4, beta=-9.0, recipe=("normal", 3.0), seed=77, **shape)
    assert D.num_nodes(case.d, case.k, case.W) <= 1024
    got = _run_full(D, case)
    ref = oracle.tree_build(case)
    stats = parity.compare_all(case, got, ref, ref["ngram"])
    assert stats["exact"] == case.B
