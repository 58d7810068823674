"""Padded vocabularies: rows row_stride > V elements apart (needs a GB300).

The logits are a view z[..., :V] of a [.., V_pad] buffer whose padding holds
values that would win every comparison (+1e30, +inf, NaN) if they were read.
Row results and whole trees must equal the oracle's on the contiguous valid
logits: ids bit-exact, log-probabilities and lse within 1e-5, trees exact.
"""
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


def _padded(case, pad, fill):
    """[B, d, V + pad] device buffer holding the case's logits, the padding set to fill."""
    z = parity.to_device(case)                      # [B, d, V] as stored
    big = torch.empty(z.shape[:-1] + (z.shape[-1] + pad,), dtype=z.dtype, device=z.device)
    big.fill_(fill)
    big[..., :z.shape[-1]] = z
    return big


CASES = [
    # dtype, V, pad, T, k, rows, recipe, fill
    ("bf16", 151936, 128, 1.0, 8, 8, ("normal_spike", 3.0, 12.0), 1e30),
    ("f16", 32000, 64, 1.0, 10, 40, ("normal_spike", 2.5, 10.0), float("inf")),
    ("f32", 7777, 1, 1.7, 16, 24, ("gumbel_zipf", 4.0, 1.2), float("nan")),
    ("bf16", 1001, 7, 1.3, 7, 37, ("normal", 3.0), 1e30),
    ("f16", 777, 3, 0.5, 32, 19, ("normal", 2.0), float("inf")),
    ("bf16", 1 << 20, 40, 1.0, 12, 3, ("normal", 3.0), 1e30),
    ("f32", 33, 31, 1.0, 5, 50, ("normal", 1.0), float("nan")),
]


@pytest.mark.parametrize("dtype,V,pad,T,k,rows,recipe,fill", CASES)
def test_row_topk_on_padded_rows(D, dtype, V, pad, T, k, rows, recipe, fill):
    case = synth.make_case(B=rows, d=1, V=V, dtype=dtype, T=T, k=k, W=1, n=0, M=0, lam=0, beta=0,
                           recipe=recipe, seed=V + pad)
    big = _padded(case, pad, fill).reshape(rows, V + pad)
    view = big[:, :V]
    ids, logp, lse, ws = D.row_topk(view, case.T, k)
    assert D.device_error(ws) == 0
    rid, rlogp, rlse = oracle.rows(case.logits, dtype, V, case.T, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.abs(logp.cpu().numpy().astype(np.float64) - rlogp).max() <= 1e-5
    assert np.abs(lse.cpu().numpy().astype(np.float64) - rlse).max() <= 1e-5


@pytest.mark.parametrize("cfg,over,pad", [
    (0, {}, 4),
    (2, dict(B=6, M=1 << 16), 128),
    (3, dict(B=24, M=1 << 16), 64),
    (2, dict(B=5, V=30011, M=1 << 14, dtype="f16"), 5),
])
def test_tree_build_on_padded_rows(D, cfg, over, pad):
    case = synth.make_config(cfg, seed=3, **over)
    fill = {"bf16": 1e30, "f16": float("inf"), "f32": float("nan")}[case.dtype]
    big = _padded(case, pad, fill)
    tab, ctx = parity.gpu_table(case)
    out = D.tree_build(big[..., :case.V], case.T, case.k, case.W, case.lam, case.beta, table=tab, ctx=ctx)
    assert D.device_error(out["workspace"]) == 0
    got = {key: v.cpu().numpy() for key, v in out.items() if key != "workspace" and v is not None}
    ref = oracle.tree_build(case)
    stats = parity.compare_all(case, got, ref, ref["ngram"])
    assert stats["exact"] == case.B
