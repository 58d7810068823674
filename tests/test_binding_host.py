"""Argument checks of the Python binding, on the CPU (no GPU, no kernel launch).

The binding hands raw device pointers to the C ABI, which cannot see a
tensor's shape, dtype or device; these checks have to catch a wrong output
dict, context or device before the call.  Device placement is exercised with
stand-in objects that carry only the attributes the binding reads.
"""
import types

import pytest

torch = pytest.importorskip("torch")

import draft_tree_construction_gb300 as D
from draft_tree_construction_gb300 import DartError


def _fake(device, shape=(2, 3), dtype=None):
    """A stand-in for a CUDA tensor on `device` (never dereferenced)."""
    return types.SimpleNamespace(is_cuda=True, device=torch.device(device), shape=shape,
                                 dtype=dtype or torch.int32, is_contiguous=lambda: True)


def _outs(B, N, MW, scores=True):
    o = {k: torch.zeros((B, N), dtype=torch.int32) for k in ("tokens", "parents", "pos")}
    o["mask"] = torch.zeros((B, N, MW), dtype=torch.int32)
    o["scores"] = torch.zeros((B, N), dtype=torch.float32) if scores else None
    return o


def test_output_dict_is_checked():
    B, N, MW = 3, 40, 2
    D._check_outputs(_outs(B, N, MW), B, N, MW)
    D._check_outputs(_outs(B, N, MW, scores=False), B, N, MW)
    bad = []
    o = _outs(B, N, MW); o["tokens"] = torch.zeros((B, N), dtype=torch.int64); bad.append(o)
    o = _outs(B, N, MW); o["parents"] = torch.zeros((B, N - 1), dtype=torch.int32); bad.append(o)
    o = _outs(B, N, MW); o["pos"] = torch.zeros((N, B), dtype=torch.int32).t(); bad.append(o)
    o = _outs(B, N, MW); o["mask"] = torch.zeros((B, N, MW + 1), dtype=torch.int32); bad.append(o)
    o = _outs(B, N, MW); o["mask"] = torch.zeros((B, N, MW), dtype=torch.float32); bad.append(o)
    o = _outs(B, N, MW); o["scores"] = torch.zeros((B, N), dtype=torch.float64); bad.append(o)
    o = _outs(B, N, MW); del o["mask"]; bad.append(o)
    for o in bad:
        with pytest.raises(DartError):
            D._check_outputs(o, B, N, MW)
    with pytest.raises(DartError):
        D._check_outputs([1, 2], B, N, MW)


def test_context_shape_follows_the_table_order():
    table = types.SimpleNamespace(n=3)
    D._check_ctx(table, torch.zeros((4, 2), dtype=torch.int32), 4)
    D._check_ctx(None, None, 4)
    for ctx in (None, torch.zeros((4, 3), dtype=torch.int32), torch.zeros((3, 2), dtype=torch.int32),
                torch.zeros((4, 2), dtype=torch.int64), torch.zeros((2, 4), dtype=torch.int32).t()):
        with pytest.raises(DartError):
            D._check_ctx(table, ctx, 4)


def test_tensors_must_share_one_cuda_device():
    assert D._device_of(("a", _fake("cuda:1")), ("b", None), ("c", _fake("cuda:1"))) == \
        torch.device("cuda", 1)
    with pytest.raises(DartError, match="cuda:0"):
        D._device_of(("a", _fake("cuda:1")), ("b", _fake("cuda:0")))
    with pytest.raises(DartError, match="CUDA tensor"):
        D._device_of(("a", torch.zeros(3)))
    with pytest.raises(DartError, match="CUDA tensor"):
        D._device_of(("a", torch.empty(3, device="meta")))


def test_stream_must_be_on_the_tensors_device():
    s1 = types.SimpleNamespace(device=torch.device("cuda", 1), cuda_stream=0)
    assert D._stream_ptr(s1, torch.device("cuda", 1)).value is None      # NULL = default stream
    with pytest.raises(DartError, match="stream"):
        D._stream_ptr(s1, torch.device("cuda", 0))


def test_workspace_size_counts_bytes():
    D._check_workspace(torch.zeros(64, dtype=torch.float32), 256)
    with pytest.raises(DartError):
        D._check_workspace(torch.zeros(63, dtype=torch.float32), 256)
    with pytest.raises(DartError):
        D._check_workspace(torch.zeros((8, 64), dtype=torch.uint8).t(), 16)


def test_host_and_meta_tensors_are_refused_before_any_call():
    for dev in ("cpu", "meta"):
        z = torch.zeros((2, 3, 100), dtype=torch.float32, device=dev)
        with pytest.raises(DartError, match="CUDA tensor"):
            D.tree_build(z, 1.0, 4, 4, 0.0, 0.0)
        with pytest.raises(DartError, match="CUDA tensor"):
            D.tree_build_noalloc(z, 1.0, 4, 4, 0.0, 0.0)
        with pytest.raises(DartError, match="CUDA tensor"):
            D.row_topk(z[0], 1.0, 4)
        ids = torch.zeros((2, 3, 4), dtype=torch.int32, device=dev)
        with pytest.raises(DartError, match="CUDA tensor"):
            D.tree_from_topk(ids, ids.double(), 4, 0.0, 0.0)
        with pytest.raises(DartError, match="CUDA tensor"):
            D.mask_pack(ids[0])
