"""Continuity-aware draft-tree construction on one GB300 (sm_103a).

A thin binding over the C ABI in include/darttree.h (libdarttree.so, built
in-tree by ``build()``).  This module only marshals arguments: every step of
the path runs in the library's CUDA kernels, PyTorch supplies device memory
and streams.  Calls raise ``DartError`` when the library is missing or a call
fails; there is no fallback.

The computation (DART, Figure 3 caption; DARTree, Method / Tree
Construction), made precise:
  p_j = log_softmax(z_j / T); C_j = the k largest z_j (lower id first on ties);
  child score = parent + p_j[c] + lam * ngram(last n-1 tokens, c), or
  + lam * beta when the n-gram is missing; keep the W best children of the
  whole frontier (score, then lower parent index, then lower token id);
  emit tokens, parents (-1 at depth 1), depths and ancestor-or-self masks.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np

from ._build import LIB as _LIB_PATH, build as _build_lib

__all__ = [
    "DartError", "build", "lib", "NGramTable", "num_nodes", "mask_words", "workspace_bytes",
    "tree_build", "tree_build_noalloc", "tree_from_topk", "tree_from_rows", "row_topk", "mask_pack", "tree_select", "set_wait_limit", "device_error", "noalloc_device_error",
    "TreeBuilder",
    "DTYPE_CODES",
]

DART_OK = 0
DEVERR = {1: "bulk-copy wait timeout", 2: "row max mismatch", 4: "tree selection", 8: "bad parent",
          16: "score rises from a parent"}


class DartError(RuntimeError):
    pass


class _Table(C.Structure):
    _fields_ = [("n", C.c_int32), ("reserved", C.c_int32), ("capacity", C.c_uint64),
                ("slots", C.c_void_p)]


_lock = threading.Lock()
_handle = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libdarttree.so for sm_103a (nvcc) if it is missing or stale."""
    return _build_lib(force=force, verbose=verbose)


def _declare(L):
    P, i32, i64, u64, f32, sz = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_float, C.c_size_t
    T = C.POINTER(_Table)
    L.dart_tree_num_nodes.argtypes = [i32, i32, i32]
    L.dart_tree_num_nodes.restype = i32
    L.dart_tree_mask_words.argtypes = [i32]
    L.dart_tree_mask_words.restype = i32
    L.dart_tree_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.dart_tree_workspace_bytes.restype = sz
    L.dart_tree_build.argtypes = [P, i32, i32, i32, i32, f32, i32, i32, f32, f32, T, P,
                                  P, P, P, P, P, P, sz, P]
    L.dart_tree_build.restype = i32
    L.dart_tree_build_verify.argtypes = [P, i32, i32, i32, i64, i32, f32, i32, i32, f32, f32, T, P,
                                         P, P, P, P, P, i32, P, P, P, P, P, P, P, sz, P]
    L.dart_tree_build_verify.restype = i32
    L.dart_tree_build_noalloc.argtypes = [P, i32, i32, i32, i32, f32, i32, i32, f32, f32, T, P,
                                          P, P, P, P, P, P]
    L.dart_tree_build_noalloc.restype = i32
    L.dart_tree_from_topk.argtypes = [P, P, i32, i32, i32, i32, f32, f32, T, P, P, P, P, P, P, P]
    L.dart_tree_from_topk.restype = i32
    L.dart_tree_from_topk_pairs.argtypes = [P, P, P, i32, i32, i32, i32, f32, P, P, P, P, P, P]
    L.dart_tree_from_topk_pairs.restype = i32
    L.dart_tree_from_rows_pairs.argtypes = [i32, i32, i32, i32, f32, i32, i32, f32, P, P, P, P, P, P,
                                            P, sz, P]
    L.dart_tree_from_rows_pairs.restype = i32
    L.dart_row_topk.argtypes = [P, i32, i32, i32, f32, i32, P, P, P, P, sz, P]
    L.dart_row_topk.restype = i32
    L.dart_row_topk_strided.argtypes = [P, i32, i32, i64, i32, f32, i32, P, P, P, P, sz, P]
    L.dart_row_topk_strided.restype = i32
    L.dart_tree_build_strided.argtypes = [P, i32, i32, i32, i64, i32, f32, i32, i32, f32, f32, T, P,
                                          P, P, P, P, P, P, sz, P]
    L.dart_tree_build_strided.restype = i32
    L.dart_tree_plan_create.argtypes = [C.POINTER(P), P, i32, i32, i32, i64, i32, f32, i32, i32, f32, f32, T, P,
                                        P, P, P, P, P, P, sz]
    L.dart_tree_plan_create.restype = i32
    L.dart_tree_plan_launch.argtypes = [P, P]
    L.dart_tree_plan_launch.restype = i32
    L.dart_tree_plan_destroy.argtypes = [P]
    L.dart_tree_plan_destroy.restype = i32
    L.dart_row_pass.argtypes = [P, i32, i32, i64, i32, f32, i32, P, sz, P]
    L.dart_row_pass.restype = i32
    L.dart_row_finish.argtypes = [i32, i32, i64, i32, f32, i32, P, P, P, P, sz, P]
    L.dart_row_finish.restype = i32
    L.dart_mask_pack.argtypes = [P, i32, i32, P, P, P]
    L.dart_mask_pack.restype = i32
    L.dart_tree_select.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, P, P, P, P]
    L.dart_tree_select.restype = i32
    L.dart_ngram_capacity_for.argtypes = [u64]
    L.dart_ngram_capacity_for.restype = u64
    L.dart_ngram_table_pack_host.argtypes = [i32, P, P, u64, u64, P, C.POINTER(C.c_uint64)]
    L.dart_ngram_table_pack_host.restype = i32
    L.dart_ngram_lookup.argtypes = [T, P, i64, P, P, P]
    L.dart_ngram_lookup.restype = i32
    L.dart_probe_ex2.argtypes = [i32, i32, i32, P, P]
    L.dart_probe_ex2.restype = i32
    L.dart_probe_stream.argtypes = [P, u64, i32, i32, i32, i32, P, P, P]
    L.dart_probe_stream.restype = i32
    L.dart_set_wait_limit.argtypes = [i64]
    L.dart_set_wait_limit.restype = None
    L.dart_device_error.argtypes = [P, C.POINTER(C.c_uint32), P]
    L.dart_device_error.restype = i32
    L.dart_noalloc_device_error.argtypes = [C.POINTER(C.c_uint32), P]
    L.dart_noalloc_device_error.restype = i32
    L.dart_status_string.argtypes = [i32]
    L.dart_status_string.restype = C.c_char_p
    return L


def lib():
    """The loaded C library; raises DartError when it has not been built."""
    global _handle
    with _lock:
        if _handle is None:
            if not os.path.exists(_LIB_PATH):
                raise DartError(f"{_LIB_PATH} is missing: run draft_tree_construction_gb300.build()")
            _handle = _declare(C.CDLL(_LIB_PATH))
    return _handle


def _check(rc: int, what: str):
    if rc != DART_OK:
        msg = lib().dart_status_string(rc).decode()
        raise DartError(f"{what} failed: {msg} ({rc})")


# --------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def DTYPE_CODES():
    torch = _torch()
    return {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def _mask_dtypes():
    torch = _torch()
    return tuple(t for t in (torch.int32, getattr(torch, "uint32", None)) if t is not None)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _device_of(*named):
    """The one CUDA device that every given tensor lives on.

    named: (name, tensor-or-None) pairs.  Raises DartError for a tensor that
    is not on a CUDA device, or for tensors on two devices: the library takes
    device pointers of the current device, so each call runs with this device
    current (see _on_device)."""
    dev = None
    for name, t in named:
        if t is None:
            continue
        if not getattr(t, "is_cuda", False):
            raise DartError(f"{name} must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise DartError(f"{name} is on {t.device}, but the other arguments are on {dev}")
    return dev


def _on_device(dev):
    """Context manager that makes `dev` the current CUDA device for one call."""
    return _torch().cuda.device(dev)


def _stream_ptr(stream, dev=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if dev is not None and getattr(s, "device", dev) != dev:
        raise DartError(f"stream is on {s.device}, but the tensors are on {dev}")
    return C.c_void_p(s.cuda_stream)


def _check_tensor(t, name, dtype=None, shape=None, contiguous=True):
    """dtype (one dtype or a tuple), exact shape and contiguity of a tensor."""
    if t is None:
        return
    if dtype is not None:
        allowed = dtype if isinstance(dtype, tuple) else (dtype,)
        if t.dtype not in allowed:
            want = " or ".join(str(a) for a in allowed)
            raise DartError(f"{name} must be {want}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise DartError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise DartError(f"{name} must be contiguous")


def _need_cuda(t, name, dtype=None, contiguous=True, shape=None):
    if t is None:
        return
    _device_of((name, t))
    _check_tensor(t, name, dtype, shape, contiguous)


def _check_outputs(o, B, N, MW):
    """Caller-supplied output tensors of a tree: tokens, parents, pos int32
    [B, N]; mask int32 (or uint32) [B, N, MW]; scores float32 [B, N] or
    absent / None.  All contiguous."""
    torch = _torch()
    if not isinstance(o, dict):
        raise DartError("out must be a dict of tensors")
    for key in ("tokens", "parents", "pos", "mask"):
        if o.get(key) is None:
            raise DartError(f"out['{key}'] is missing")
    for key in ("tokens", "parents", "pos"):
        _check_tensor(o[key], f"out['{key}']", torch.int32, (B, N))
    _check_tensor(o["mask"], "out['mask']", _mask_dtypes(), (B, N, MW))
    _check_tensor(o.get("scores"), "out['scores']", torch.float32, (B, N))


def _check_ctx(table, ctx, B):
    """The committed context a table needs: int32 [B, n-1], contiguous."""
    if table is None:
        return
    if ctx is None:
        raise DartError("ctx is required with an n-gram table")
    _check_tensor(ctx, "ctx", _torch().int32, (B, table.n - 1))


def _check_workspace(ws, need):
    _check_tensor(ws, "workspace", contiguous=True)
    if ws.numel() * ws.element_size() < need:
        raise DartError(f"workspace holds {ws.numel() * ws.element_size()} bytes, {need} needed")


def _out_names(o):
    return [(f"out['{k}']", o.get(k)) for k in ("tokens", "parents", "pos", "mask", "scores")]


def num_nodes(d: int, k: int, W: int) -> int:
    return lib().dart_tree_num_nodes(d, k, W)


def mask_words(N: int) -> int:
    return lib().dart_tree_mask_words(N)


def workspace_bytes(B: int, d: int, V: int, dtype_code: int, k: int) -> int:
    return lib().dart_tree_workspace_bytes(B, d, V, dtype_code, k)


# ------------------------------------------------------------ n-gram model

class NGramTable:
    """Open-addressing n-gram table in device memory (format: include/darttree.h)."""

    def __init__(self, n: int, keys: np.ndarray, vals: np.ndarray, device="cuda",
                 capacity: int | None = None):
        torch = _torch()
        L = lib()
        keys = np.ascontiguousarray(keys, dtype=np.int32).reshape(-1, n)
        vals = np.ascontiguousarray(vals, dtype=np.float32).reshape(-1)
        M = keys.shape[0]
        cap = int(capacity) if capacity else int(L.dart_ngram_capacity_for(M))
        host = np.empty(cap * 16, dtype=np.uint8)
        distinct = C.c_uint64(0)
        _check(L.dart_ngram_table_pack_host(n, keys.ctypes.data_as(C.c_void_p),
                                            vals.ctypes.data_as(C.c_void_p), M, cap,
                                            host.ctypes.data_as(C.c_void_p), C.byref(distinct)),
               "dart_ngram_table_pack_host")
        self.n = n
        self.capacity = cap
        self.distinct = int(distinct.value)
        self.slots = torch.from_numpy(host).to(device)
        self.desc = _Table(n, 0, cap, self.slots.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.capacity * 16

    def lookup(self, keys, stream=None):
        """keys: CUDA int32 [Q, n] -> (vals float32 [Q], found bool [Q])."""
        torch = _torch()
        dev = _device_of(("keys", keys), ("table", self.slots))
        _check_tensor(keys, "keys", torch.int32)
        if keys.dim() != 2 or keys.shape[1] != self.n:
            raise DartError(f"keys must be [Q, {self.n}], got {tuple(keys.shape)}")
        Q = keys.shape[0]
        vals = torch.empty(Q, dtype=torch.float32, device=dev)
        found = torch.empty(Q, dtype=torch.int32, device=dev)
        with _on_device(dev):
            _check(lib().dart_ngram_lookup(C.byref(self.desc), _ptr(keys), Q, _ptr(vals), _ptr(found),
                                           _stream_ptr(stream, dev)), "dart_ngram_lookup")
        return vals, found.bool()


# ------------------------------------------------------------ the tree path

def _outputs(B, N, MW, device, scores: bool):
    torch = _torch()
    return dict(tokens=torch.empty((B, N), dtype=torch.int32, device=device),
                parents=torch.empty((B, N), dtype=torch.int32, device=device),
                pos=torch.empty((B, N), dtype=torch.int32, device=device),
                mask=torch.empty((B, N, MW), dtype=torch.int32, device=device),
                scores=torch.empty((B, N), dtype=torch.float32, device=device) if scores else None)


def _row_stride(logits) -> int:
    """Elements between row starts of a [..., V] tensor whose rows are evenly
    spaced with unit element stride (a contiguous tensor, or a view such as
    z[..., :V] of a padded one); raises otherwise."""
    shape, strides = logits.shape, logits.stride()
    V = shape[-1]
    if V > 1 and strides[-1] != 1:
        raise DartError("logits rows must have unit element stride")
    rows = 1
    for s_ in shape[:-1]:
        rows *= s_
    if rows <= 1:
        return V
    # the innermost row dimension of size > 1 fixes the stride; every outer one must continue it
    step = None
    expect = None
    for size, st in reversed(list(zip(shape[:-1], strides[:-1]))):
        if size == 1:
            continue
        if step is None:
            step, expect = st, st * size
        elif st != expect:
            raise DartError("logits rows must be evenly spaced")
        else:
            expect = st * size
    if step < V:
        raise DartError("logits rows overlap")
    return int(step)


def _table_args(table, ctx):
    if table is None:
        return None, None
    return C.byref(table.desc), _ptr(ctx)


def _tree_inputs(logits, k, W, table, ctx, out, extra=()):
    """Shared checks of tree_build / tree_build_noalloc: returns (dev, B, d, V, N, MW)."""
    codes = DTYPE_CODES()
    dev = _device_of(("logits", logits), ("ctx", ctx if table is not None else None),
                     ("table", table.slots if table is not None else None),
                     *(_out_names(out) if out is not None else ()), *extra)
    if logits.dtype not in codes or logits.dim() != 3:
        raise DartError("logits must be [B, d, V] float32, float16 or bfloat16")
    B, d, V = logits.shape
    N = num_nodes(d, k, W)
    if N < 0:
        raise DartError("invalid d/k/W")
    MW = mask_words(N)
    _check_ctx(table, ctx, B)
    if out is not None:
        _check_outputs(out, B, N, MW)
    return dev, B, d, V, N, MW


def _verify_outputs(B, Mp, device, scores: bool):
    torch = _torch()
    return dict(index=torch.empty((B, Mp), dtype=torch.int32, device=device),
                tokens=torch.empty((B, Mp), dtype=torch.int32, device=device),
                parents=torch.empty((B, Mp), dtype=torch.int32, device=device),
                pos=torch.empty((B, Mp), dtype=torch.int32, device=device),
                mask=torch.empty((B, Mp, (Mp + 31) // 32), dtype=torch.int32, device=device),
                scores=torch.empty((B, Mp), dtype=torch.float32, device=device) if scores else None)


def tree_build(logits, T: float, k: int, W: int, lam: float, beta: float,
               table: NGramTable | None = None, ctx=None, *, out: dict | None = None,
               workspace=None, stream=None, scores: bool = True, verify_budget: int | None = None) -> dict:
    """logits: CUDA [B, d, V] float32/float16/bfloat16 -> dict of CUDA outputs.

    The rows may be a view of a padded vocabulary (z[..., :V] of [B, d, V_pad]):
    only the V valid logits of each row are read.  mask is returned as int32
    storage holding the uint32 bit pattern.  T = 0 is greedy decoding: the
    tree is then scored with log_softmax(z), as at T = 1.  Every tensor
    (logits, ctx, the table, out, workspace) must be on one CUDA device; the
    call runs with that device current.  With verify_budget = M the same
    kernels also choose each tree's best-first verification tree of min(M, N)
    nodes (dart_tree_build_verify), returned under "verify" with the keys of
    tree_select."""
    torch = _torch()
    dev, B, d, V, N, MW = _tree_inputs(logits, k, W, table, ctx, out, (("workspace", workspace),))
    stride = _row_stride(logits)
    code = DTYPE_CODES()[logits.dtype]
    need = workspace_bytes(B, d, V, code, k)
    if verify_budget is not None and int(verify_budget) < 1:
        raise DartError("verify_budget must be >= 1")
    with _on_device(dev):
        o = out if out is not None else _outputs(B, N, MW, dev, scores)
        if workspace is not None:
            _check_workspace(workspace, need)
            ws = workspace
        else:
            ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=dev)
        outs = (_ptr(o["tokens"]), _ptr(o["parents"]), _ptr(o["pos"]), _ptr(o["mask"]), _ptr(o.get("scores")))
        if verify_budget is None:
            rc = lib().dart_tree_build_strided(_ptr(logits), B, d, V, stride, code, float(T), k, W,
                                               float(lam), float(beta), *_table_args(table, ctx), *outs,
                                               _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream, dev))
            what = "dart_tree_build_strided"
        else:
            M = int(verify_budget)
            v = _verify_outputs(B, min(M, N), dev, scores)
            rc = lib().dart_tree_build_verify(_ptr(logits), B, d, V, stride, code, float(T), k, W,
                                              float(lam), float(beta), *_table_args(table, ctx), *outs, M,
                                              _ptr(v["index"]), _ptr(v["tokens"]), _ptr(v["parents"]),
                                              _ptr(v["pos"]), _ptr(v["mask"]), _ptr(v["scores"]),
                                              _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream, dev))
            what = "dart_tree_build_verify"
            o["verify"] = v
    _check(rc, what)
    o["workspace"] = ws
    return o


def tree_build_noalloc(logits, T: float, k: int, W: int, lam: float, beta: float,
                       table: NGramTable | None = None, ctx=None, *, out: dict | None = None,
                       stream=None, scores: bool = True, check_errors: bool = False) -> dict:
    """tree_build for callers that cannot allocate device scratch: the library's
    fixed 16 MiB buffer stands in for the workspace (see dart_tree_build_noalloc
    in include/darttree.h for its limits and sharing rules).  logits must be
    contiguous.  With check_errors, the call then waits for the stream and
    raises DartError if the buffer's device error word is set."""
    dev, B, d, V, N, MW = _tree_inputs(logits, k, W, table, ctx, out)
    _check_tensor(logits, "logits")
    code = DTYPE_CODES()[logits.dtype]
    with _on_device(dev):
        o = out if out is not None else _outputs(B, N, MW, dev, scores)
        sp = _stream_ptr(stream, dev)
        rc = lib().dart_tree_build_noalloc(_ptr(logits), B, d, V, code, float(T), k, W,
                                           float(lam), float(beta), *_table_args(table, ctx),
                                           _ptr(o["tokens"]), _ptr(o["parents"]), _ptr(o["pos"]),
                                           _ptr(o["mask"]), _ptr(o.get("scores")), sp)
        _check(rc, "dart_tree_build_noalloc")
        if check_errors:
            flags = _noalloc_error(sp)
            if flags:
                raise DartError(f"dart_tree_build_noalloc: device error bits {flags:#x} "
                                f"({_deverr_names(flags)})")
    return o


def _noalloc_error(stream_ptr) -> int:
    flags = C.c_uint32(0)
    _check(lib().dart_noalloc_device_error(C.byref(flags), stream_ptr), "dart_noalloc_device_error")
    return int(flags.value)


def noalloc_device_error(device=None, stream=None) -> int:
    """Waits for the stream, then returns (and clears) the device error bits
    that dart_tree_build_noalloc calls on `device` (default: the current one)
    left in the library's internal buffer."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with _on_device(dev):
        return _noalloc_error(_stream_ptr(stream, dev))


def _deverr_names(flags: int) -> str:
    return ", ".join(v for b, v in DEVERR.items() if flags & b) or "unknown"


def tree_from_topk(ids, logp, W: int, lam: float, beta: float = 0.0, table: NGramTable | None = None,
                   ctx=None, *, pairs=None, out: dict | None = None, stream=None,
                   scores: bool = True) -> dict:
    """ids: CUDA int32 [B, d, k]; logp: CUDA float64 [B, d, k] -> dict of CUDA outputs.

    The continuity term is the n-gram table (with ctx), or `pairs`: CUDA
    float32 [B, d, k, k] caller scores of (parent's list position in row j-1,
    child's list position in row j), the root counting as position 0 for row
    0 (dart_tree_from_topk_pairs), or nothing."""
    torch = _torch()
    if pairs is not None and table is not None:
        raise DartError("give either an n-gram table or pair scores, not both")
    dev = _device_of(("ids", ids), ("logp", logp), ("ctx", ctx if table is not None else None),
                     ("table", table.slots if table is not None else None), ("pairs", pairs),
                     *(_out_names(out) if out is not None else ()))
    if ids.dim() != 3:
        raise DartError("ids must be [B, d, k]")
    _check_tensor(ids, "ids", torch.int32)
    _check_tensor(logp, "logp", torch.float64, tuple(ids.shape))
    B, d, k = ids.shape
    _check_tensor(pairs, "pairs", torch.float32, (B, d, k, k))
    N = num_nodes(d, k, W)
    if N < 0:
        raise DartError("invalid d/k/W")
    MW = mask_words(N)
    _check_ctx(table, ctx, B)
    if out is not None:
        _check_outputs(out, B, N, MW)
    with _on_device(dev):
        o = out if out is not None else _outputs(B, N, MW, dev, scores)
        outs = (_ptr(o["tokens"]), _ptr(o["parents"]), _ptr(o["pos"]), _ptr(o["mask"]), _ptr(o.get("scores")))
        if pairs is not None:
            rc = lib().dart_tree_from_topk_pairs(_ptr(ids), _ptr(logp), _ptr(pairs), B, d, k, W, float(lam),
                                                 *outs, _stream_ptr(stream, dev))
            what = "dart_tree_from_topk_pairs"
        else:
            rc = lib().dart_tree_from_topk(_ptr(ids), _ptr(logp), B, d, k, W, float(lam), float(beta),
                                           *_table_args(table, ctx), *outs, _stream_ptr(stream, dev))
            what = "dart_tree_from_topk"
    _check(rc, what)
    return o


def tree_from_rows(workspace, pairs, *, B: int, d: int, V: int, dtype, T: float, k: int, W: int,
                   lam: float, out: dict | None = None, stream=None, scores: bool = True) -> dict:
    """The tree stage on the candidate lists that row_topk left in `workspace`
    (rows = B * d, same V, dtype, T and k), with pair scores `pairs` (CUDA
    float32 [B, d, k, k], see tree_from_topk) as the continuity term
    (dart_tree_from_rows_pairs)."""
    torch = _torch()
    code = DTYPE_CODES()[dtype]
    dev = _device_of(("workspace", workspace), ("pairs", pairs),
                     *(_out_names(out) if out is not None else ()))
    if pairs is None:
        raise DartError("pairs is required")
    _check_tensor(pairs, "pairs", torch.float32, (B, d, k, k))
    _check_workspace(workspace, workspace_bytes(B, d, V, code, k))
    N = num_nodes(d, k, W)
    if N < 0:
        raise DartError("invalid d/k/W")
    MW = mask_words(N)
    if out is not None:
        _check_outputs(out, B, N, MW)
    with _on_device(dev):
        o = out if out is not None else _outputs(B, N, MW, dev, scores)
        rc = lib().dart_tree_from_rows_pairs(B, d, V, code, float(T), k, W, float(lam), _ptr(pairs),
                                             _ptr(o["tokens"]), _ptr(o["parents"]), _ptr(o["pos"]),
                                             _ptr(o["mask"]), _ptr(o.get("scores")), _ptr(workspace),
                                             workspace.numel() * workspace.element_size(),
                                             _stream_ptr(stream, dev))
    _check(rc, "dart_tree_from_rows_pairs")
    return o


def row_topk(logits, T: float, k: int, *, workspace=None, stream=None):
    """logits: CUDA [R, V] -> (ids int32 [R,k], logp float32 [R,k], lse float32 [R], workspace).

    The rows may be a view of a padded vocabulary (z[:, :V] of [R, V_pad])."""
    torch = _torch()
    codes = DTYPE_CODES()
    dev = _device_of(("logits", logits), ("workspace", workspace))
    if logits.dtype not in codes or logits.dim() != 2:
        raise DartError("logits must be [R, V] float32, float16 or bfloat16")
    R, V = logits.shape
    stride = _row_stride(logits)
    need = workspace_bytes(R, 1, V, codes[logits.dtype], k)
    with _on_device(dev):
        ids = torch.empty((R, k), dtype=torch.int32, device=dev)
        logp = torch.empty((R, k), dtype=torch.float32, device=dev)
        lse = torch.empty((R,), dtype=torch.float32, device=dev)
        if workspace is not None:
            _check_workspace(workspace, need)
            ws = workspace
        else:
            ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=dev)
        rc = lib().dart_row_topk_strided(_ptr(logits), R, V, stride, codes[logits.dtype], float(T), k,
                                         _ptr(ids), _ptr(logp), _ptr(lse), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream_ptr(stream, dev))
    _check(rc, "dart_row_topk_strided")
    return ids, logp, lse, ws


def _check_error_word(device_err):
    if device_err is not None:
        _check_tensor(device_err, "device_err", (_torch().int32,) + _mask_dtypes()[1:])
        if device_err.numel() < 1:
            raise DartError("device_err must hold at least one element")


def mask_pack(parents, *, device_err=None, stream=None):
    """parents: CUDA int32 [B, N] -> mask int32 [B, N, ceil(N/32)] (uint32 bits)."""
    torch = _torch()
    dev = _device_of(("parents", parents), ("device_err", device_err))
    if parents.dim() != 2:
        raise DartError("parents must be [B, N]")
    _check_tensor(parents, "parents", torch.int32)
    _check_error_word(device_err)
    B, N = parents.shape
    with _on_device(dev):
        out = torch.empty((B, N, (N + 31) // 32), dtype=torch.int32, device=dev)
        rc = lib().dart_mask_pack(_ptr(parents), B, N, _ptr(out), _ptr(device_err),
                                  _stream_ptr(stream, dev))
    _check(rc, "dart_mask_pack")
    return out


def tree_select(tokens, parents, pos, scores, M: int, *, device_err=None, stream=None) -> dict:
    """Verification tree of budget M chosen best-first from candidate trees.

    tokens, parents, pos: CUDA int32 [B, N]; scores: CUDA float32 [B, N] (as
    returned by tree_build).  Returns index, tokens, parents, pos (int32 [B, M']),
    mask (int32 [B, M', ceil(M'/32)], uint32 bits) and scores (float32 [B, M']),
    M' = min(M, N)."""
    torch = _torch()
    dev = _device_of(("tokens", tokens), ("parents", parents), ("pos", pos), ("scores", scores),
                     ("device_err", device_err))
    if parents.dim() != 2:
        raise DartError("tokens, parents, pos and scores must all be [B, N]")
    for t, name in ((tokens, "tokens"), (parents, "parents"), (pos, "pos")):
        _check_tensor(t, name, torch.int32, tuple(parents.shape))
    _check_tensor(scores, "scores", torch.float32, tuple(parents.shape))
    _check_error_word(device_err)
    if int(M) < 0:
        raise DartError("the budget M must be >= 0")
    B, N = parents.shape
    Mp = min(int(M), N)
    with _on_device(dev):
        out = dict(index=torch.empty((B, Mp), dtype=torch.int32, device=dev),
                   tokens=torch.empty((B, Mp), dtype=torch.int32, device=dev),
                   parents=torch.empty((B, Mp), dtype=torch.int32, device=dev),
                   pos=torch.empty((B, Mp), dtype=torch.int32, device=dev),
                   mask=torch.empty((B, Mp, (Mp + 31) // 32), dtype=torch.int32, device=dev),
                   scores=torch.empty((B, Mp), dtype=torch.float32, device=dev))
        rc = lib().dart_tree_select(_ptr(tokens), _ptr(parents), _ptr(pos), _ptr(scores), B, N, int(M),
                                    _ptr(out["index"]), _ptr(out["tokens"]), _ptr(out["parents"]),
                                    _ptr(out["pos"]), _ptr(out["mask"]), _ptr(out["scores"]),
                                    _ptr(device_err), _stream_ptr(stream, dev))
    _check(rc, "dart_tree_select")
    return out


def set_wait_limit(cycles: int) -> None:
    """SM clock cycles any one wait of the row pass may take before it gives up
    (<= 0 restores the default of about two seconds).  For tests of the timeout
    path."""
    lib().dart_set_wait_limit(int(cycles))


def device_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the workspace's device error bits."""
    dev = _device_of(("workspace", workspace))
    flags = C.c_uint32(0)
    with _on_device(dev):
        _check(lib().dart_device_error(_ptr(workspace), C.byref(flags), _stream_ptr(stream, dev)),
               "dart_device_error")
    return int(flags.value)


class TreeBuilder:
    """Fixed-shape driver: preallocated outputs and workspace, one C call per step.

    With graph=True (the default) the first call on a logits buffer records
    the path's launches once (dart_tree_plan_create) and every call on the same
    buffer replays them (dart_tree_plan_launch); a call on another buffer
    records a new plan.  graph=False calls dart_tree_build every time."""

    def __init__(self, B, d, V, dtype, T, k, W, lam, beta, table=None, ctx=None, device="cuda",
                 scores=True, graph=True):
        torch = _torch()
        self.shape = (B, d, V)
        self.dtype = dtype
        self.code = DTYPE_CODES()[dtype]
        self.T, self.k, self.W, self.lam, self.beta = float(T), k, W, float(lam), float(beta)
        self.N = num_nodes(d, k, W)
        if self.N < 0:
            raise DartError("invalid d/k/W")
        self.MW = mask_words(self.N)
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        _device_of(("ctx", ctx if table is not None else None),
                   ("table", table.slots if table is not None else None))
        _check_ctx(table, ctx, B)
        self.table, self.ctx = table, ctx
        with _on_device(self.device):
            self.out = _outputs(B, self.N, self.MW, self.device, scores)
            self.ws = torch.zeros(max(workspace_bytes(B, d, V, self.code, k), 1), dtype=torch.uint8,
                                  device=self.device)
        _device_of(("workspace", self.ws), ("ctx", ctx if table is not None else None))
        self.graph = graph
        self._plan = None          # (logits address, plan handle)

    def _drop_plan(self):
        if self._plan is not None:
            _check(lib().dart_tree_plan_destroy(self._plan[1]), "dart_tree_plan_destroy")
            self._plan = None

    def __del__(self):
        try:
            if self._plan is not None:
                _torch().cuda.synchronize(self.device)
                self._drop_plan()
        except Exception:
            pass

    def __call__(self, logits, stream=None):
        B, d, V = self.shape
        if _device_of(("logits", logits)) != self.device:
            raise DartError(f"logits is on {logits.device}, the builder on {self.device}")
        _check_tensor(logits, "logits", self.dtype, self.shape)
        # inside a caller's own graph capture the kernels are launched directly,
        # so that the caller's graph records them
        if self.graph and not _torch().cuda.is_current_stream_capturing():
            with _on_device(self.device):
                sp = _stream_ptr(stream, self.device)
                if self._plan is None or self._plan[0] != logits.data_ptr():
                    if self._plan is not None:
                        _torch().cuda.synchronize(self.device)   # launches of the old plan are done
                    self._drop_plan()
                    plan = C.c_void_p()
                    rc = lib().dart_tree_plan_create(C.byref(plan), _ptr(logits), B, d, V, V, self.code, self.T,
                                                     self.k, self.W, self.lam, self.beta,
                                                     *_table_args(self.table, self.ctx),
                                                     _ptr(self.out["tokens"]), _ptr(self.out["parents"]),
                                                     _ptr(self.out["pos"]), _ptr(self.out["mask"]),
                                                     _ptr(self.out.get("scores")), _ptr(self.ws), self.ws.numel())
                    _check(rc, "dart_tree_plan_create")
                    self._plan = (logits.data_ptr(), plan)
                rc = lib().dart_tree_plan_launch(self._plan[1], sp)
            _check(rc, "dart_tree_plan_launch")
            return self.out
        with _on_device(self.device):
            rc = lib().dart_tree_build(_ptr(logits), B, d, V, self.code, self.T, self.k, self.W,
                                       self.lam, self.beta, *_table_args(self.table, self.ctx),
                                       _ptr(self.out["tokens"]), _ptr(self.out["parents"]),
                                       _ptr(self.out["pos"]), _ptr(self.out["mask"]),
                                       _ptr(self.out.get("scores")), _ptr(self.ws),
                                       self.ws.numel(), _stream_ptr(stream, self.device))
        _check(rc, "dart_tree_build")
        return self.out
