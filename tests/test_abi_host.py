"""The C ABI without a GPU: symbols, argument checks, sizes, the host packer.

Every check here returns before any CUDA call, so it runs on a machine with
no GPU.  Fake device pointers are never dereferenced (the library rejects the
call first).  The n-gram packer is checked against an independent reading of
the slot format documented in include/darttree.h.
"""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import draft_tree_construction_gb300 as D

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "darttree.h")

OK, INVALID, WORKSPACE, FULL = 0, 1, 3, 7


@pytest.fixture(scope="module")
def L():
    D.build()
    return D.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dart_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", D._LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (dart_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_sizes(L):
    assert L.dart_tree_num_nodes(4, 4, 4) == 16
    assert L.dart_tree_num_nodes(8, 8, 8) == 64
    assert L.dart_tree_num_nodes(8, 8, 10) == 8 + 10 * 7
    assert L.dart_tree_num_nodes(8, 10, 16) == 10 + 16 * 7
    assert L.dart_tree_num_nodes(16, 16, 32) == 16 + 32 * 15
    assert L.dart_tree_num_nodes(0, 4, 4) == -1
    assert L.dart_tree_mask_words(496) == 16
    assert L.dart_tree_mask_words(1) == 1
    assert L.dart_tree_mask_words(-1) == -1
    assert L.dart_tree_workspace_bytes(64, 8, 151936, 2, 8) > 0
    assert L.dart_tree_workspace_bytes(64, 8, 151936, 5, 8) == 0
    assert L.dart_tree_workspace_bytes(64, 8, 151936, 2, 33) == 0
    assert L.dart_ngram_capacity_for(4096) == 8192
    assert L.dart_ngram_capacity_for(5000) == 16384
    assert L.dart_ngram_capacity_for(0) == 8
    assert L.dart_ngram_capacity_for(3) == 8


FAKE = 0x10000000          # 16- and 256-byte aligned, never dereferenced


def _build(L, **over):
    a = dict(logits=FAKE, B=2, d=4, V=1000, dtype=2, T=1.0, k=4, W=4, lam=0.5, beta=-10.0, table=None,
             ctx=None, tok=FAKE, par=FAKE, pos=FAKE, mask=FAKE, scores=None, ws=None, wsb=0, stream=None)
    a.update(over)
    v = lambda key: C.c_void_p(a[key]) if a[key] else None
    return L.dart_tree_build(v("logits"), a["B"], a["d"], a["V"], a["dtype"], a["T"], a["k"], a["W"],
                             a["lam"], a["beta"], a["table"], v("ctx"), v("tok"), v("par"), v("pos"),
                             v("mask"), v("scores"), v("ws"), a["wsb"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(d=0), INVALID), (dict(d=33), INVALID), (dict(V=1), INVALID), (dict(V=1 << 24), INVALID),
    (dict(k=0), INVALID), (dict(k=33), INVALID), (dict(k=5, V=4), INVALID), (dict(W=0), INVALID),
    (dict(W=65), INVALID), (dict(d=32, k=32, W=64), INVALID),       # N > 1024
    (dict(T=-1e-30), INVALID), (dict(T=-1.0), INVALID), (dict(T=float("nan")), INVALID),
    (dict(T=float("inf")), INVALID), (dict(lam=float("nan")), INVALID),
    (dict(beta=float("-inf")), INVALID), (dict(dtype=3), INVALID), (dict(B=-1), INVALID),
    (dict(logits=0), INVALID), (dict(logits=FAKE + 8), INVALID), (dict(tok=0), INVALID),
    (dict(mask=0), INVALID),
    (dict(ws=None, wsb=0), WORKSPACE), (dict(ws=FAKE + 16, wsb=1 << 30), WORKSPACE),
    (dict(ws=FAKE, wsb=100), WORKSPACE),
    (dict(B=0), OK), (dict(B=0, logits=0, tok=0), OK),
])
def test_tree_build_argument_checks(L, over, code):
    assert _build(L, **over) == code


def _table(n=3, cap=1024, slots=FAKE, reserved=0):
    return D._Table(n, reserved, cap, slots)


@pytest.mark.parametrize("tab,ctx,code", [
    (dict(n=1), FAKE, INVALID), (dict(n=5), FAKE, INVALID), (dict(cap=1000), FAKE, INVALID),
    (dict(cap=1), FAKE, INVALID), (dict(cap=4), FAKE, INVALID), (dict(slots=0), FAKE, INVALID),
    (dict(slots=FAKE + 4), FAKE, INVALID), (dict(slots=FAKE + 16), FAKE, INVALID),
    (dict(reserved=1), FAKE, INVALID), (dict(), 0, INVALID),
])
def test_table_argument_checks(L, tab, ctx, code):
    t = _table(**tab)
    assert _build(L, table=C.byref(t), ctx=ctx) == code


def test_other_entry_points_check_arguments(L):
    P = C.c_void_p
    assert L.dart_row_topk(P(FAKE), 4, 1, 2, 1.0, 1, None, None, None, None, 0, None) == INVALID
    assert L.dart_row_topk(P(FAKE), 4, 100, 2, -0.5, 4, None, None, None, None, 0, None) == INVALID
    # T = 0 (greedy) passes the argument checks: the missing workspace is what fails
    assert L.dart_row_topk(P(FAKE), 4, 100, 2, 0.0, 4, None, None, None, None, 0, None) == WORKSPACE
    assert L.dart_noalloc_device_error(None, None) == INVALID
    assert L.dart_row_topk(P(FAKE), 4, 100, 2, 1.0, 4, None, None, None, None, 0, None) == WORKSPACE
    assert L.dart_row_topk(None, 0, 100, 2, 1.0, 4, None, None, None, None, 0, None) == OK
    assert L.dart_tree_from_topk(None, None, 2, 4, 4, 4, 0.5, -1.0, None, None, None, None, None, None,
                                 None, None) == INVALID
    assert L.dart_tree_from_topk(None, None, 0, 4, 4, 4, 0.5, -1.0, None, None, None, None, None, None,
                                 None, None) == OK
    assert L.dart_mask_pack(None, 2, 10, None, None, None) == INVALID
    assert L.dart_mask_pack(None, 0, 10, None, None, None) == OK
    assert L.dart_ngram_lookup(None, None, 10, None, None, None) == INVALID
    # padded rows: the stride must reach V, and stays below 2^30
    assert L.dart_row_topk_strided(P(FAKE), 4, 100, 99, 2, 1.0, 4, None, None, None, None, 0, None) == INVALID
    assert L.dart_row_topk_strided(P(FAKE), 4, 100, 1 << 31, 2, 1.0, 4, None, None, None, None, 0,
                                   None) == INVALID
    assert L.dart_row_topk_strided(P(FAKE), 4, 100, 128, 2, 1.0, 4, None, None, None, None, 0,
                                   None) == WORKSPACE
    assert L.dart_tree_build_strided(P(FAKE), 2, 3, 100, 50, 2, 1.0, 4, 4, 0.5, -1.0, None, None, P(FAKE),
                                     P(FAKE), P(FAKE), P(FAKE), None, None, 0, None) == INVALID
    assert L.dart_probe_ex2(0, 64, 8, P(FAKE), None) == INVALID       # no blocks
    assert L.dart_probe_ex2(4, 48, 8, P(FAKE), None) == INVALID       # threads not a multiple of 32
    assert L.dart_probe_ex2(4, 64, 8, None, None) == INVALID          # no output
    ps = lambda src, mode, warps, stages: L.dart_probe_stream(src, 1 << 20, mode, 4, warps, stages, P(FAKE),
                                                               P(FAKE), None)
    assert ps(P(FAKE + 8), 1, 12, 3) == INVALID       # source not 16-byte aligned
    assert ps(P(FAKE), 8, 12, 3) == INVALID           # unknown mode bit
    assert ps(P(FAKE), 4, 12, 3) == INVALID           # interleaving is a bulk-ring mode
    assert ps(P(FAKE), 0, 17, 0) == INVALID           # direct loads: at most 16 warps
    assert ps(P(FAKE), 5, 12, 1) == INVALID           # a ring needs two stages
    assert ps(P(FAKE), 5, 16, 4) == INVALID           # 16 x 4 stages of 4 KiB exceed shared memory
    sel = lambda B, N, M, ptr: L.dart_tree_select(ptr, ptr, ptr, ptr, B, N, M, ptr, ptr, ptr, ptr, ptr,
                                                  None, None, None)
    assert sel(2, 0, 4, P(FAKE)) == INVALID          # no nodes
    assert sel(2, 1025, 4, P(FAKE)) == INVALID       # above the node limit
    assert sel(2, 16, -1, P(FAKE)) == INVALID        # negative budget
    assert sel(2, 16, 4, None) == INVALID            # missing buffers
    assert sel(0, 16, 4, None) == OK                 # nothing to do: no launch
    assert sel(2, 16, 0, None) == OK
    assert L.dart_device_error(None, None, None) == INVALID
    plan = C.c_void_p(12345)
    assert L.dart_tree_plan_create(None, P(FAKE), 2, 3, 100, 100, 2, 1.0, 4, 4, 0.5, -1.0, None, None, P(FAKE),
                                   P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), 1 << 30) == INVALID
    assert L.dart_tree_plan_create(C.byref(plan), P(FAKE), 2, 3, 100, 100, 2, 1.0, 4, 0, 0.5, -1.0, None, None,
                                   P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), 1 << 30) == INVALID
    assert plan.value is None                          # W = 0 refused before anything is captured
    assert L.dart_tree_plan_create(C.byref(plan), P(FAKE), 2, 3, 100, 100, 2, 1.0, 4, 4, 0.5, -1.0, None, None,
                                   P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), 16) == WORKSPACE
    assert L.dart_tree_plan_launch(None, None) == INVALID
    assert L.dart_tree_plan_destroy(None) == OK
    assert L.dart_status_string(1).decode() == "invalid argument"


# ------------------------------------------------------------ host packer

def _splitmix_fold(w0, w1, w2):
    """The key hash as the header describes it (splitmix64 output function)."""
    M64 = (1 << 64) - 1
    x = (w0 | (w1 << 32)) ^ ((w2 * 0x9E3779B97F4A7C15) & M64)
    x ^= x >> 30
    x = (x * 0xBF58476D1CE4E5B9) & M64
    x ^= x >> 27
    x = (x * 0x94D049BB133111EB) & M64
    x ^= x >> 31
    return x


def _key_words(tokens):
    v = 0
    for f, t in enumerate(tokens):
        v |= int(t) << (24 * f)
    return v & 0xFFFFFFFF, (v >> 32) & 0xFFFFFFFF, (v >> 64) & 0xFFFFFFFF


BUCKET_SLOTS = 2   # two 16-byte slots to a 32-byte bucket, as the header describes it


def _buckets(w, cap):
    """The key's two buckets, as the header describes them."""
    h = _splitmix_fold(*w)
    nb = cap // BUCKET_SLOTS
    b1, b2 = h & (nb - 1), (h >> 32) & (nb - 1)
    return b1, (b1 ^ 1 if b2 == b1 else b2)


def _find(slots, cap, tokens):
    w = _key_words(tokens)
    for b in _buckets(w, cap):
        for t in range(BUCKET_SLOTS):
            s = slots[BUCKET_SLOTS * b + t]
            if tuple(int(x) for x in s[:3]) == w:
                return True, s[3:4].view(np.float32)[0]
    return False, None


@pytest.mark.parametrize("n", [2, 3, 4])
def test_packer_against_documented_format(L, n):
    rng = np.random.default_rng(n)
    M = 3000
    keys = rng.integers(0, (1 << 24) - 1, size=(M, n)).astype(np.int32)
    keys[100:200] = keys[:100]                                   # repeats: first value wins
    vals = rng.uniform(-9, -1, size=M).astype(np.float32)
    cap = L.dart_ngram_capacity_for(M)
    slots = np.zeros((cap, 4), dtype=np.uint32)
    distinct = C.c_uint64(0)
    rc = L.dart_ngram_table_pack_host(n, keys.ctypes.data_as(C.c_void_p), vals.ctypes.data_as(C.c_void_p),
                                      M, cap, slots.ctypes.data_as(C.c_void_p), C.byref(distinct))
    assert rc == OK
    first = {}
    for key, v in zip(map(tuple, keys.tolist()), vals):
        first.setdefault(key, v)
    assert distinct.value == len(first)
    for key, v in first.items():
        ok, got = _find(slots, cap, key)
        assert ok and got == v
    for key in rng.integers(0, 1 << 20, size=(500, n)).tolist():
        if tuple(key) not in first:
            assert not _find(slots, cap, key)[0]
    # every other slot is empty
    assert int((slots[:, :3] != 0xFFFFFFFF).any(axis=1).sum()) == len(first)


def test_packer_at_half_load_displaces_and_keeps_every_key(L):
    """capacity / 2 distinct keys: some keys find both buckets full and move
    earlier keys to their other bucket; every key must stay findable."""
    rng = np.random.default_rng(11)
    cap = 4096
    M = cap // 2
    keys = rng.choice((1 << 24) - 1, size=(M, 3), replace=True).astype(np.int32)
    keys[:, 0] = np.arange(M)                                    # distinct keys
    vals = rng.uniform(-9, -1, size=M).astype(np.float32)
    slots = np.zeros((cap, 4), dtype=np.uint32)
    distinct = C.c_uint64(0)
    rc = L.dart_ngram_table_pack_host(3, keys.ctypes.data_as(C.c_void_p), vals.ctypes.data_as(C.c_void_p),
                                      M, cap, slots.ctypes.data_as(C.c_void_p), C.byref(distinct))
    assert rc == OK and distinct.value == M
    home = sum(1 for key in keys.tolist()
               if any(tuple(int(x) for x in slots[BUCKET_SLOTS * _buckets(_key_words(key), cap)[0] + t][:3])
                      == _key_words(key) for t in range(BUCKET_SLOTS)))
    assert home < M                                              # some keys sit in their second bucket
    for key, v in zip(keys.tolist(), vals):
        ok, got = _find(slots, cap, key)
        assert ok and got == v


def test_packer_refuses_overfull_and_bad_tokens(L):
    keys = np.arange(10, dtype=np.int32).reshape(5, 2)
    vals = np.zeros(5, dtype=np.float32)
    slots = np.zeros((8, 4), dtype=np.uint32)
    P = lambda a: a.ctypes.data_as(C.c_void_p)
    assert L.dart_ngram_table_pack_host(2, P(keys), P(vals), 5, 8, P(slots), None) == FULL
    assert L.dart_ngram_table_pack_host(2, P(keys), P(vals), 4, 8, P(slots), None) == OK
    bad = keys.copy()
    bad[2, 1] = (1 << 24) - 1
    assert L.dart_ngram_table_pack_host(2, P(bad), P(vals), 4, 8, P(slots), None) == INVALID
    bad[2, 1] = -5
    assert L.dart_ngram_table_pack_host(2, P(bad), P(vals), 4, 8, P(slots), None) == INVALID
    assert L.dart_ngram_table_pack_host(2, P(keys), P(vals), 4, 6, P(slots), None) == INVALID
    assert L.dart_ngram_table_pack_host(2, P(keys), P(vals), 2, 4, P(slots), None) == INVALID   # below 8 slots


def test_row_stride_of_views():
    torch = pytest.importorskip("torch")
    z = torch.zeros((3, 4, 130))
    assert D._row_stride(z) == 130
    assert D._row_stride(z[:, :, :100]) == 130          # a padded vocabulary
    assert D._row_stride(z[:, 1:2, :100]) == 130 * 4    # one row per sequence
    assert D._row_stride(z[:1, :1, :7]) == 7            # a single row
    assert D._row_stride(z.reshape(12, 130)[:, :128]) == 130
    assert D._row_stride(z[:, ::2, :100]) == 260        # every other row: still evenly spaced
    with pytest.raises(D.DartError):
        D._row_stride(z[:, :2, :100])                    # two rows of four: a gap after each pair
    with pytest.raises(D.DartError):
        D._row_stride(z[:, :, ::2])                      # elements not adjacent


def test_binding_rejects_host_tensors_and_bad_shapes():
    torch = pytest.importorskip("torch")
    z = torch.zeros((2, 3, 100))
    with pytest.raises(D.DartError):
        D.tree_build(z, 1.0, 4, 4, 0.5, -1.0)                 # host memory: no CPU fallback
    with pytest.raises(D.DartError):
        D.row_topk(z[0], 1.0, 4)
    t = torch.zeros((2, 5), dtype=torch.int32)
    with pytest.raises(D.DartError):
        D.tree_select(t, t, t, torch.zeros((2, 5)), 3)         # host memory


def test_noalloc_rejects_sizes_beyond_its_buffer(L):
    # 65,536 rows with k = 32 need far more workspace than the fixed 16 MiB
    # scratch; the call refuses before any CUDA call, so the fake pointers are
    # never touched
    B, d, V, k, W = 8192, 8, 4096, 32, 64
    need = L.dart_tree_workspace_bytes(B, d, V, 2, k)
    assert need > (16 << 20)
    assert L.dart_tree_num_nodes(d, k, W) <= 1024
    fake = C.c_void_p(0x10000000)
    rc = L.dart_tree_build_noalloc(fake, B, d, V, 2, 1.0, k, W, 0.25, -14.0, None, None,
                                   fake, fake, fake, fake, None, None)
    assert rc == WORKSPACE
