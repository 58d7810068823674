"""Python face of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  It never touches the CUDA
library and the CUDA library never touches it.

``build()`` compiles oracle.c with gcc (C11, OpenMP, no floating-point
contraction, so every product and sum is rounded exactly as written).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle (or a copy of it, for mutation tests) to a shared library."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < max(
        os.path.getmtime(src), os.path.getmtime(_HDR))
    if force or stale:
        inc = os.path.dirname(os.path.abspath(src))
        cmd = ["gcc", *CFLAGS, "-I", _HERE, "-I", inc, src, "-o", out + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)
    return out


def _declare(lib):
    P = C.c_void_p
    i32, i64, dbl = C.c_int, C.c_int64, C.c_double
    lib.oracle_rows.argtypes = [P, i32, i64, i32, dbl, i32, P, P, P, i32]
    lib.oracle_rows.restype = i32
    lib.oracle_decode.argtypes = [P, i32, i64]
    lib.oracle_decode.restype = dbl
    lib.oracle_ngram_new.argtypes = [i32, P, P, i64]
    lib.oracle_ngram_new.restype = P
    lib.oracle_ngram_free.argtypes = [P]
    lib.oracle_ngram_free.restype = None
    lib.oracle_ngram_lookup.argtypes = [P, P, i64, P, P]
    lib.oracle_ngram_lookup.restype = None
    lib.oracle_tree_from_lists.argtypes = [i32, i32, i32, i32, P, P, dbl, P, dbl, dbl, P, i32, P,
                                           P, P, P, P, P, P, i32]
    lib.oracle_tree_from_lists.restype = i32
    lib.oracle_tree_from_pairs.argtypes = [i32, i32, i32, i32, P, P, dbl, P, dbl, P,
                                           P, P, P, P, P, P, i32]
    lib.oracle_tree_from_pairs.restype = i32
    lib.oracle_tree_trace.argtypes = [i32, i32, i32, P, P, dbl, P, dbl, dbl, P, i32, P, P, i64, P]
    lib.oracle_tree_trace.restype = i32
    lib.oracle_tree_build.argtypes = [P, i32, i32, i32, i32, dbl, i32, i32, dbl, dbl, P, i32, P,
                                      P, P, P, P, P, P, P, P, P, i32]
    lib.oracle_tree_build.restype = i32
    lib.oracle_num_nodes.argtypes = [i32, i32, i32]
    lib.oracle_num_nodes.restype = i32
    lib.oracle_mask_from_parents.argtypes = [i32, i32, P, P]
    lib.oracle_mask_from_parents.restype = i32
    lib.oracle_select_tree.argtypes = [i32, i32, i32, P, P, P, P]
    lib.oracle_select_tree.restype = i32
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; a path loads a specific build."""
    global _lib
    if path is not None:
        return _declare(C.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(C.CDLL(build()))
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


DTYPES = {"f32": 0, "f16": 1, "bf16": 2}


class NGram:
    """The oracle's own n-gram model: a sorted array of (key, first value)."""

    def __init__(self, n: int, keys: np.ndarray, vals: np.ndarray, lib=None):
        self.lib = lib or load()
        self.n = int(n)
        self._keys = np.ascontiguousarray(keys, dtype=np.int32).reshape(-1, self.n)
        self._vals = np.ascontiguousarray(vals, dtype=np.float32).reshape(-1)
        self.h = self.lib.oracle_ngram_new(self.n, _p(self._keys), _p(self._vals),
                                           self._keys.shape[0])
        if not self.h:
            raise MemoryError("oracle_ngram_new failed")

    def lookup(self, keys: np.ndarray):
        q = np.ascontiguousarray(keys, dtype=np.int32).reshape(-1, self.n)
        vals = np.zeros(q.shape[0], dtype=np.float32)
        found = np.zeros(q.shape[0], dtype=np.int32)
        self.lib.oracle_ngram_lookup(self.h, _p(q), q.shape[0], _p(vals), _p(found))
        return vals, found.astype(bool)

    def __del__(self):
        if getattr(self, "h", None):
            self.lib.oracle_ngram_free(self.h)
            self.h = None


def num_nodes(d: int, k: int, W: int, lib=None) -> int:
    return (lib or load()).oracle_num_nodes(d, k, W)


def rows(logits: np.ndarray, dtype: str, V: int, T: float, k: int, threads: int = 0, lib=None):
    """(ids [R,k] int32, logp [R,k] f64, lse [R] f64) for logits viewed as [R, V]."""
    lib = lib or load()
    z = np.ascontiguousarray(logits)
    R = z.size // V
    ids = np.zeros((R, k), dtype=np.int32)
    logp = np.zeros((R, k), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    rc = lib.oracle_rows(_p(z), DTYPES[dtype], R, V, float(T), k, _p(ids), _p(logp), _p(lse),
                         threads)
    if rc:
        raise ValueError(f"oracle_rows failed ({rc})")
    return ids, logp, lse


def tree_from_lists(ids, base, *, B, d, k, W, lam, beta, ngram: NGram | None, ctx,
                    invT: float = 1.0, off=None, threads: int = 0, lib=None):
    """The tree stage alone, from candidate lists ids/base [B, d, k].

    With the defaults (invT = 1, off = None) base holds log-probabilities."""
    lib = lib or load()
    N = lib.oracle_num_nodes(d, k, W)
    if N < 0:
        raise ValueError("invalid d/k/W")
    MW = (N + 31) // 32
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    base = np.ascontiguousarray(base, dtype=np.float64)
    offa = None if off is None else np.ascontiguousarray(off, dtype=np.float64)
    tok = np.zeros((B, N), dtype=np.int32)
    par = np.zeros((B, N), dtype=np.int32)
    pos = np.zeros((B, N), dtype=np.int32)
    mask = np.zeros((B, N, MW), dtype=np.uint32)
    sc = np.zeros((B, N), dtype=np.float64)
    gap = np.zeros((B, d), dtype=np.float64)
    n = ngram.n if ngram is not None else 0
    c = None if ctx is None else np.ascontiguousarray(ctx, dtype=np.int32)
    rc = lib.oracle_tree_from_lists(B, d, k, W, _p(ids), _p(base), float(invT), _p(offa), float(lam),
                                    float(beta), ngram.h if ngram is not None else None, n, _p(c),
                                    _p(tok), _p(par), _p(pos), _p(mask), _p(sc), _p(gap), threads)
    if rc:
        raise ValueError(f"oracle_tree_from_lists failed ({rc})")
    return dict(tokens=tok, parents=par, pos=pos, mask=mask, scores=sc, min_pos_gap=gap)


def tree_from_pairs(ids, base, pair, *, B, d, k, W, lam, invT: float = 1.0, off=None,
                    threads: int = 0, lib=None):
    """The tree stage with caller-supplied pair scores pair [B, d, k, k] as the
    continuity term: a child with column c of row j adds pair[b, j, c', c],
    c' its parent's column in row j-1 (0 at j = 0, the root)."""
    lib = lib or load()
    N = lib.oracle_num_nodes(d, k, W)
    if N < 0:
        raise ValueError("invalid d/k/W")
    MW = (N + 31) // 32
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    base = np.ascontiguousarray(base, dtype=np.float64)
    pr = np.ascontiguousarray(pair, dtype=np.float32)
    if pr.shape != (B, d, k, k):
        raise ValueError("pair must be [B, d, k, k]")
    offa = None if off is None else np.ascontiguousarray(off, dtype=np.float64)
    tok = np.zeros((B, N), dtype=np.int32)
    par = np.zeros((B, N), dtype=np.int32)
    pos = np.zeros((B, N), dtype=np.int32)
    mask = np.zeros((B, N, MW), dtype=np.uint32)
    sc = np.zeros((B, N), dtype=np.float64)
    gap = np.zeros((B, d), dtype=np.float64)
    rc = lib.oracle_tree_from_pairs(B, d, k, W, _p(ids), _p(base), float(invT), _p(offa), float(lam),
                                    _p(pr), _p(tok), _p(par), _p(pos), _p(mask), _p(sc), _p(gap),
                                    threads)
    if rc:
        raise ValueError(f"oracle_tree_from_pairs failed ({rc})")
    return dict(tokens=tok, parents=par, pos=pos, mask=mask, scores=sc, min_pos_gap=gap)


TRACE_DTYPE = np.dtype([("depth", "<i4"), ("parent", "<i4"), ("parent_rank", "<i4"), ("token", "<i4"),
                        ("column", "<i4"), ("found", "<i4"), ("node", "<i4"), ("pad", "<i4"),
                        ("g", "<f8"), ("Z", "<f8"), ("G", "<f8"), ("key", "<f8")])


def tree_trace(ids, base, *, d, k, W, lam, beta, ngram: NGram | None, ctx, invT: float = 1.0, off=None,
               lib=None) -> np.ndarray:
    """One tree (ids/base [d, k], ctx [n-1]) with every expanded child: a
    structured array (TRACE_DTYPE), per depth the whole sorted candidate table."""
    lib = lib or load()
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(d, k)
    base = np.ascontiguousarray(base, dtype=np.float64).reshape(d, k)
    offa = None if off is None else np.ascontiguousarray(off, dtype=np.float64).reshape(d)
    cap = 0
    width = 1
    for _ in range(d):
        cap += width * k
        width = min(width * k, W)
    out = np.zeros(cap, dtype=TRACE_DTYPE)
    n = ngram.n if ngram is not None else 0
    c = None if ctx is None else np.ascontiguousarray(ctx, dtype=np.int32)
    length = C.c_int64(0)
    rc = lib.oracle_tree_trace(d, k, W, _p(ids), _p(base), float(invT), _p(offa), float(lam), float(beta),
                               ngram.h if ngram is not None else None, n, _p(c), _p(out), cap,
                               C.byref(length))
    if rc:
        raise ValueError(f"oracle_tree_trace failed ({rc})")
    return out[:length.value]


def tree_build(case, ngram: NGram | None = None, threads: int = 0, use_table: bool = True, lib=None):
    """The whole path on a synth.Case: rows, then the tree.  Returns a dict of arrays."""
    lib = lib or load()
    B, d, V, k, W = case.B, case.d, case.V, case.k, case.W
    if use_table and case.n >= 2 and ngram is None:
        ngram = NGram(case.n, case.ng_keys, case.ng_vals, lib=lib)
    if not use_table:
        ngram = None
    N = lib.oracle_num_nodes(d, k, W)
    MW = (N + 31) // 32
    z = np.ascontiguousarray(case.logits)
    tok = np.zeros((B, N), dtype=np.int32)
    par = np.zeros((B, N), dtype=np.int32)
    pos = np.zeros((B, N), dtype=np.int32)
    mask = np.zeros((B, N, MW), dtype=np.uint32)
    sc = np.zeros((B, N), dtype=np.float64)
    gap = np.zeros((B, d), dtype=np.float64)
    rid = np.zeros((B, d, k), dtype=np.int32)
    rlp = np.zeros((B, d, k), dtype=np.float64)
    rlse = np.zeros((B, d), dtype=np.float64)
    n = ngram.n if ngram is not None else 0
    ctx = np.ascontiguousarray(case.ctx, dtype=np.int32)
    rc = lib.oracle_tree_build(_p(z), DTYPES[case.dtype], B, d, V, float(case.T), k, W,
                               float(case.lam), float(case.beta),
                               ngram.h if ngram is not None else None, n, _p(ctx),
                               _p(tok), _p(par), _p(pos), _p(mask), _p(sc), _p(gap),
                               _p(rid), _p(rlp), _p(rlse), threads)
    if rc:
        raise ValueError(f"oracle_tree_build failed ({rc})")
    return dict(tokens=tok, parents=par, pos=pos, mask=mask, scores=sc, min_pos_gap=gap,
                row_ids=rid, row_logp=rlp, row_lse=rlse, ngram=ngram)


def mask_from_parents(parents: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    par = np.ascontiguousarray(parents, dtype=np.int32)
    B, N = par.shape
    MW = (N + 31) // 32
    mask = np.zeros((B, N, MW), dtype=np.uint32)
    rc = lib.oracle_mask_from_parents(B, N, _p(par), _p(mask))
    if rc:
        raise ValueError(f"oracle_mask_from_parents failed ({rc})")
    return mask


def select_tree(tokens, parents, pos, scores, M: int, lib=None):
    """Verification tree of budget M chosen best-first from candidate trees
    [B, N] (see oracle_select_tree).  Returns index, tokens, parents, pos [B, M']
    and the ancestor masks [B, M', ceil(M'/32)] of the chosen trees, M' = min(M, N)."""
    lib = lib or load()
    par = np.ascontiguousarray(parents, dtype=np.int32)
    B, N = par.shape
    s = np.ascontiguousarray(scores, dtype=np.float64).reshape(B, N)
    Mp = min(int(M), N)
    index = np.zeros((B, Mp), dtype=np.int32)
    npar = np.zeros((B, Mp), dtype=np.int32)
    rc = lib.oracle_select_tree(B, N, int(M), _p(par), _p(s), _p(index), _p(npar))
    if rc:
        raise ValueError(f"oracle_select_tree failed ({rc})")
    tok = np.take_along_axis(np.asarray(tokens, dtype=np.int32).reshape(B, N), index, axis=1)
    dep = np.take_along_axis(np.asarray(pos, dtype=np.int32).reshape(B, N), index, axis=1)
    MW = (Mp + 31) // 32
    mask = np.zeros((B, Mp, MW), dtype=np.uint32)
    if Mp:
        rc = lib.oracle_mask_from_parents(B, Mp, _p(npar), _p(mask))
        if rc:
            raise ValueError(f"oracle_mask_from_parents failed ({rc})")
    return dict(index=index, tokens=tok, parents=npar, pos=dep, mask=mask)
