"""Seeded synthetic inputs for continuity-aware draft-tree construction.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no softmax, no scoring, no pruning).  Both the CPU oracle
and the CUDA path are fed from here, and nothing else is shared between them.

Workloads follow five configurations, numbered 0-4 (DART,
"Figure 3" pipeline: d parallel logit vectors per sequence, an n-gram model for
continuity; DARTree "Tree Construction": fixed width W per depth):

  0: B=1,   d=4,  V=1024,   f32  N(0,2),                        T=1,   k=4,  W=4,  bigram  4096 keys U(-8,-0.5),   lam=0.5,  beta=-10
  1: B=1,   d=8,  V=151936, bf16 N(0,3) + one +12 spike per row, T=1,   k=8,  W=8,  trigram 2^20 keys U(-10,-0.5), lam=0.3,  beta=-12
  2: B=64,  d=8,  V=151936, bf16 N(0,3) + Zipf(1.1) boost,       T=0.7, k=8,  W=10, trigram 2^22 keys U(-10,-0.5), lam=0.3,  beta=-12
  3: B=256, d=8,  V=32000,  f16  N(0,2.5) + one +10 spike,       T=1,   k=10, W=16, bigram  2^21 keys U(-10,-0.5), lam=0.5,  beta=-10
  4: B=32,  d=16, V=151936, bf16 4*Gumbel(0,1) + Zipf(1.2) boost, T=1,   k=16, W=32, 4-gram  2^24 keys U(-10,-0.5), lam=0.25, beta=-14

Readings taken where the workload text is silent (each is listed in the design
notes): the second N(.,.) parameter is the standard deviation; a Zipf(s) boost
gives the token at rank r of a fresh random permutation the additive logit
-s*ln(r); Gumbel draws are -ln(-ln U); values are drawn in fp32 and rounded once
(round-to-nearest-even) to the stored dtype; "1M/2M/4M/16M entries" are 2^20,
2^21, 2^22 and 2^24 keys; the committed context (the last n-1 tokens before the
root, the root last) is drawn U[0,V).

N-gram keys: uniformly random n-grams over a 152k vocabulary essentially never
occur along a draft path, which would leave the continuity term untested.  So
half of each table is drawn from n-grams that lie along candidate paths: the
context tokens and the predicted token are taken from each row's k largest
logits (found here with numpy's argpartition, only to choose which keys exist),
each such n-gram kept with probability 1/2 (or sampled, when that set is too
large to list).  The rest are uniform random n-grams.  Duplicate keys are
dropped, the first occurrence kept, so every table holds M distinct keys.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field

import numpy as np

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass
class Case:
    """One synthetic workload: logits, committed context and n-gram table."""
    name: str
    B: int
    d: int
    V: int
    dtype: str          # "f32" | "f16" | "bf16"
    T: float
    k: int
    W: int
    n: int              # n-gram order (0 = no table)
    lam: float
    beta: float
    logits: np.ndarray  # [B, d, V]; float32 / float16 / uint16 (bf16 bit patterns)
    ctx: np.ndarray     # int32 [B, n-1] (oldest first, root last); [B, 0] when n == 0
    ng_keys: np.ndarray  # int32 [M, n] (oldest context token first, predicted token last)
    ng_vals: np.ndarray  # float32 [M]
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def logit_bytes(self) -> int:
        return self.B * self.d * self.V * ELEM_BYTES[self.dtype]


CONFIGS = {
    0: dict(B=1, d=4, V=1024, dtype="f32", T=1.0, k=4, W=4, n=2, M=4096,
            vlo=-8.0, vhi=-0.5, lam=0.5, beta=-10.0, recipe=("normal", 2.0)),
    1: dict(B=1, d=8, V=151936, dtype="bf16", T=1.0, k=8, W=8, n=3, M=1 << 20,
            vlo=-10.0, vhi=-0.5, lam=0.3, beta=-12.0, recipe=("normal_spike", 3.0, 12.0)),
    2: dict(B=64, d=8, V=151936, dtype="bf16", T=0.7, k=8, W=10, n=3, M=1 << 22,
            vlo=-10.0, vhi=-0.5, lam=0.3, beta=-12.0, recipe=("normal_zipf", 3.0, 1.1)),
    3: dict(B=256, d=8, V=32000, dtype="f16", T=1.0, k=10, W=16, n=2, M=1 << 21,
            vlo=-10.0, vhi=-0.5, lam=0.5, beta=-10.0, recipe=("normal_spike", 2.5, 10.0)),
    4: dict(B=32, d=16, V=151936, dtype="bf16", T=1.0, k=16, W=32, n=4, M=1 << 24,
            vlo=-10.0, vhi=-0.5, lam=0.25, beta=-14.0, recipe=("gumbel_zipf", 4.0, 1.2)),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even), returned as uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _draw_logits(rng: np.random.Generator, B: int, d: int, V: int, recipe) -> np.ndarray:
    kind = recipe[0]
    R = B * d
    if kind == "normal":
        z = rng.standard_normal((R, V), dtype=np.float32) * np.float32(recipe[1])
    elif kind == "normal_spike":
        z = rng.standard_normal((R, V), dtype=np.float32) * np.float32(recipe[1])
        tok = rng.integers(0, V, size=R)
        z[np.arange(R), tok] += np.float32(recipe[2])
    elif kind in ("normal_zipf", "gumbel_zipf"):
        if kind == "normal_zipf":
            z = rng.standard_normal((R, V), dtype=np.float32) * np.float32(recipe[1])
        else:
            u = rng.random((R, V), dtype=np.float32)
            u = np.clip(u, np.float32(1e-30), np.float32(1.0 - 2.0 ** -24))
            z = (-np.log(-np.log(u))) * np.float32(recipe[1])
        s = recipe[2]
        boost = (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
        perm = rng.permuted(np.tile(np.arange(V, dtype=np.int64), (R, 1)), axis=1)
        rows = np.arange(R)[:, None]
        z[rows, perm] += boost[None, :]
    elif kind == "ties":
        # integer-valued logits with many exact ties (edge-case tests)
        z = rng.integers(-recipe[1], recipe[1] + 1, size=(R, V)).astype(np.float32)
    elif kind == "const":
        z = np.full((R, V), np.float32(recipe[1]), dtype=np.float32)
    else:
        raise ValueError(f"unknown logit recipe {kind!r}")
    return z.reshape(B, d, V)


def _store(z: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(z, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(z.astype(np.float16))
    if dtype == "bf16":
        return f32_to_bf16_bits(z)
    raise ValueError(dtype)


def _as_f32(logits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (logits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return logits.astype(np.float32)


def _dedupe_first(keys: np.ndarray) -> np.ndarray:
    """Boolean mask keeping the first occurrence of each row of an int32 [M, n] array."""
    M, n = keys.shape
    if M == 0:
        return np.zeros(0, dtype=bool)
    k64 = keys.astype(np.int64)
    pad = np.zeros((M, 4), dtype=np.int64)
    pad[:, :n] = k64
    hi = (pad[:, 0] << 24) | pad[:, 1]
    lo = (pad[:, 2] << 24) | pad[:, 3]
    order = np.lexsort((lo, hi))  # stable: equal keys keep their original order
    hs, ls = hi[order], lo[order]
    dup_sorted = np.zeros(M, dtype=bool)
    dup_sorted[1:] = (hs[1:] == hs[:-1]) & (ls[1:] == ls[:-1])
    keep = np.ones(M, dtype=bool)
    keep[order[dup_sorted]] = False
    return keep


def _path_keys(rng, zf32, ctx, k, n, budget):
    """n-grams lying along candidate paths (see module docstring)."""
    B, d, V = zf32.shape
    kk = min(k, V)
    top = np.argpartition(-zf32.reshape(B * d, V), kk - 1, axis=1)[:, :kk].reshape(B, d, kk)
    # sequence of token sets per tree: n-1 fixed context tokens, then the d candidate sets
    per_depth_space = []
    for j in range(d):
        size = 1
        for pos in range(j, j + n):
            size *= 1 if pos < n - 1 else kk
        per_depth_space.append(size)
    space = B * sum(per_depth_space)
    out = []
    if space <= 4_000_000:
        for b in range(B):
            seq = [np.array([ctx[b, i]], dtype=np.int64) for i in range(n - 1)]
            seq += [top[b, j].astype(np.int64) for j in range(d)]
            for j in range(d):
                sets = seq[j:j + n]
                grid = np.array(list(itertools.product(*sets)), dtype=np.int64).reshape(-1, n)
                out.append(grid)
        allk = np.concatenate(out, axis=0)
        allk = allk[rng.random(allk.shape[0]) < 0.5]
    else:
        S = budget
        b = rng.integers(0, B, size=S)
        j = rng.integers(0, d, size=S)
        cols = []
        for p in range(n):
            pos = j + p  # position in the (n-1 context ++ d sets) sequence
            is_ctx = pos < n - 1
            ci = np.clip(pos, 0, n - 2) if n > 1 else np.zeros_like(pos)
            from_ctx = ctx[b, ci] if n > 1 else np.zeros(S, dtype=np.int64)
            row = np.clip(pos - (n - 1), 0, d - 1)
            from_top = top[b, row, rng.integers(0, kk, size=S)]
            cols.append(np.where(is_ctx, from_ctx, from_top))
        allk = np.stack(cols, axis=1).astype(np.int64)
    if allk.shape[0] > budget:
        allk = allk[:budget]
    return allk.astype(np.int32)


def make_ngram_table(rng, zf32, ctx, k, n, M, vlo, vhi, V):
    """Distinct n-gram keys [M, n] (half along candidate paths) and values U(vlo, vhi)."""
    if n == 0 or M == 0:
        return np.zeros((0, max(n, 1)), dtype=np.int32), np.zeros(0, dtype=np.float32)
    path = _path_keys(rng, zf32, ctx, k, n, M // 2)
    keys = path
    while True:
        need = M - keys.shape[0]
        extra = rng.integers(0, V, size=(need + need // 8 + 16, n)).astype(np.int32)
        keys = np.concatenate([keys, extra], axis=0)
        keys = keys[_dedupe_first(keys)]
        if keys.shape[0] >= M:
            keys = np.ascontiguousarray(keys[:M])
            break
    vals = rng.uniform(vlo, vhi, size=M).astype(np.float32)
    return keys, vals


def make_case(*, B, d, V, dtype, T, k, W, n, M, lam, beta, recipe, seed=0,
              vlo=-10.0, vhi=-0.5, name="custom") -> Case:
    rng = np.random.default_rng(seed)
    zf = _draw_logits(rng, B, d, V, recipe)
    logits = _store(zf, dtype)
    zs = _as_f32(logits, dtype)  # the values actually stored
    ctx = rng.integers(0, V, size=(B, max(n - 1, 0))).astype(np.int32)
    keys, vals = make_ngram_table(rng, zs, ctx, k, n, M, vlo, vhi, V)
    # T, lambda and beta cross the C ABI as fp32: keep the fp32 value on both sides
    f32 = lambda x: float(np.float32(x))
    return Case(name=name, B=B, d=d, V=V, dtype=dtype, T=f32(T), k=k, W=W, n=n,
                lam=f32(lam), beta=f32(beta), logits=logits, ctx=ctx,
                ng_keys=keys, ng_vals=vals, seed=seed, meta=dict(recipe=recipe, M=M))


def make_config(i: int, seed: int = 0, **over) -> Case:
    """Config i (0..4) at its full size; keyword overrides shrink it for quick tests."""
    c = dict(CONFIGS[i])
    c.update(over)
    return make_case(name=f"config{i}", seed=seed, **c)


def stored_as_f32(case: Case) -> np.ndarray:
    """The stored logits widened exactly to float32 (for generators and plots only)."""
    return _as_f32(case.logits, case.dtype)


def make_candidate_trees(*, B: int, d: int, k: int, W: int, seed: int = 0, tie_frac: float = 0.1,
                         zero_frac: float = 0.05):
    """Random candidate trees shaped like the built ones, as input for choosing
    verification trees: per depth j = 1..d there are min(W, k^j) nodes (depth
    by depth, parents before children), each node below depth 1 hangs under a
    random node of the depth above (at most k children each), and scores are
    float32 values that never rise along a path: depth-1 scores are drawn
    U(-8, -0.5), a child's score is its parent's minus a drop U(0, 6).  A share
    `tie_frac` of nodes copies the score of an earlier node where that keeps
    the path non-increasing, and a share `zero_frac` of drops is exactly 0, so
    equal scores occur.  Tokens are U[0, 1000).  Returns dict(tokens, parents,
    pos, scores) of shapes [B, N]."""
    rng = np.random.default_rng(seed)
    sizes = [min(W, k ** j) for j in range(1, d + 1)]
    N = int(sum(sizes))
    tokens = rng.integers(0, 1000, size=(B, N)).astype(np.int32)
    parents = np.full((B, N), -1, dtype=np.int32)
    pos = np.zeros((B, N), dtype=np.int32)
    scores = np.zeros((B, N), dtype=np.float32)
    for b in range(B):
        start, prev = 0, None
        for j, n_j in enumerate(sizes, start=1):
            idx = np.arange(start, start + n_j)
            pos[b, idx] = j
            if prev is None:
                scores[b, idx] = rng.uniform(-8.0, -0.5, size=n_j).astype(np.float32)
            else:
                slots = np.repeat(prev, k)                   # each parent has k child slots
                par = np.sort(rng.choice(slots, size=n_j, replace=False))
                parents[b, idx] = par
                drop = rng.uniform(0.0, 6.0, size=n_j)
                drop[rng.random(n_j) < zero_frac] = 0.0
                scores[b, idx] = (scores[b, par].astype(np.float64) - drop).astype(np.float32)
            # exact ties: copy an earlier node's score when the path stays non-increasing
            for x in idx:
                if rng.random() < tie_frac and x > 0:
                    y = int(rng.integers(0, x))
                    p = parents[b, x]
                    if p < 0 or scores[b, y] <= scores[b, p]:
                        scores[b, x] = scores[b, y]
            start += n_j
            prev = idx
    return dict(tokens=tokens, parents=parents, pos=pos, scores=scores)


def head_pair_scores(ids: np.ndarray, roots: np.ndarray, *, rank: int = 8, seed: int = 0) -> np.ndarray:
    """Pair scores [B, d, k, k] of a random low-rank order-2 head, restricted to
    the candidate lists ids [B, d, k]: token t has seeded embeddings u(t) and
    v(t) in R^rank, and the score of child position c after parent position c'
    is the log-softmax over the k children of u(parent token) . v(child
    token) / sqrt(rank).  The parent of row 0 is the tree's root token
    roots[b]; rows j > 0 take row j-1's candidates as parents.  float32."""
    ids = np.asarray(ids, dtype=np.int64)
    B, d, k = ids.shape
    toks = np.unique(np.concatenate([ids.reshape(-1), np.asarray(roots, dtype=np.int64).reshape(-1)]))
    rng = np.random.default_rng(seed)
    U = rng.standard_normal((toks.size, rank))
    Vv = rng.standard_normal((toks.size, rank))
    row = {int(t): i for i, t in enumerate(toks.tolist())}
    out = np.zeros((B, d, k, k), dtype=np.float32)
    for b in range(B):
        for j in range(d):
            parents = [int(roots[b])] * k if j == 0 else ids[b, j - 1].tolist()
            child = np.array([row[int(t)] for t in ids[b, j].tolist()])
            for cp, pt in enumerate(parents):
                logits = Vv[child] @ U[row[pt]] / np.sqrt(rank)
                m = logits.max()
                out[b, j, cp] = (logits - m - np.log(np.exp(logits - m).sum())).astype(np.float32)
    return out
