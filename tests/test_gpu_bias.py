"""GPU parity with biases: b1 (b3) added before the activation in the column
epilogue, b2 added once after the g-sum in the row epilogue, and the bias
gradients (column sums over tokens) from the deterministic column-sum
kernel -- against the fp64 oracle with the same biases."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import cat_cols, cat_rows, rel_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def _run(tp, inp, bias, act, dtype):
    T, d = inp.X.shape
    mlp = tp.ShardedMLP(T, d, inp.d_i, act, dtype)
    cu = lambda xs: [x.cuda() for x in xs] if xs is not None else None
    X, dY = inp.X.cuda(), inp.dY.cuda()
    W1, W2, W3 = cu(inp.W1_i), cu(inp.W2_i), cu(inp.W3_i)
    b1, b3, b2 = cu(bias["b1_i"]), cu(bias["b3_i"]), bias["b2"].cuda()
    Y, saved, H = mlp.forward(X, W1, W2, W3, b1_i=b1, b3_i=b3, b2=b2)
    g = mlp.backward(X, W1, W2, saved, H, dY, W3, bias_grads=True)
    torch.cuda.synchronize()
    mlp.check()
    return Y, saved, H, g


def _check(tp, T, d, d_i, act, dtype, seed=11):
    inp = si.make_inputs(T, d, d_i, act, dtype, seed)
    bias = si.make_biases(d, d_i, act, dtype, seed)
    Y, saved, H, g = _run(tp, inp, bias, act, dtype)
    kw = dict(act=act, W3=inp.W3, b1=bias["b1"], b3=bias["b3"], b2=bias["b2"])
    f = oracle.forward(inp.X, inp.W1, inp.W2, **kw)
    b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, **kw)
    t = len(d_i)
    errs = {"Y": rel_err(to_np(Y), f["Y"]), "A": rel_err(cat_cols(saved[:t]), f["A"]),
            "H": rel_err(cat_cols(H), f["H"]), "dX": rel_err(to_np(g["dX"]), b["dX"]),
            "dW1": rel_err(cat_cols(g["dW1"]), b["dW1"]), "dW2": rel_err(cat_rows(g["dW2"]), b["dW2"]),
            "db1": rel_err(np.concatenate([to_np(x) for x in g["db1"]]), b["db1"]),
            "db2": rel_err(to_np(g["db2"]), b["db2"])}
    if act == "swiglu":
        errs["U"] = rel_err(cat_cols(saved[t:]), f["U"])
        errs["dW3"] = rel_err(cat_cols(g["dW3"]), b["dW3"])
        errs["db3"] = rel_err(np.concatenate([to_np(x) for x in g["db3"]]), b["db3"])
    tol = tol_for(dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"over tolerance {tol}: {bad} (all {errs})"
    return g


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("case", [(200, 72, (40, 136, 64)), (333, 200, (8, 96, 264, 152)), (1, 8, (8,)),
                                  (1024, 384, (512, 384, 640, 256))])
def test_bias_bf16(gpu_lib, act, case):
    _check(gpu_lib, *case, act, "bf16")


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bias_fp32(gpu_lib, act):
    _check(gpu_lib, 45, 36, (20, 44), act, "fp32")


def test_bias_grads_deterministic(gpu_lib):
    tp = gpu_lib
    inp = si.make_inputs(777, 256, (384, 128), "swiglu", "bf16", seed=3)
    bias = si.make_biases(256, (384, 128), "swiglu", "bf16", seed=3)
    g1 = _run(tp, inp, bias, "swiglu", "bf16")[3]
    g2 = _run(tp, inp, bias, "swiglu", "bf16")[3]
    for k in ("db1", "db3"):
        for x, y in zip(g1[k], g2[k]):
            assert torch.equal(x, y)
    assert torch.equal(g1["db2"], g2["db2"])


def test_bias_grads_empty_batch(gpu_lib):
    tp = gpu_lib
    d, d_i = 64, (64, 32)
    mlp = tp.ShardedMLP(0, d, d_i, "swiglu", "bf16")
    X = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    W = lambda r, c: torch.randn(r, c, device="cuda").to(torch.bfloat16)
    W1 = [W(d, w) for w in d_i]; W3 = [W(d, w) for w in d_i]; W2 = [W(w, d) for w in d_i]
    Y, saved, H = mlp.forward(X, W1, W2, W3)
    g = mlp.backward(X, W1, W2, saved, H, torch.empty(0, d, dtype=torch.bfloat16, device="cuda"), W3,
                     bias_grads=True)
    torch.cuda.synchronize()
    for x in g["db1"] + g["db3"] + [g["db2"]]:
        assert torch.count_nonzero(x) == 0


@pytest.mark.parametrize("name", ["C3", "C4"])
def test_bias_workload_sampled(gpu_lib, name):
    w = si.WORKLOADS[name]
    inp = si.make_workload_inputs(w)
    bias = si.make_biases(w.d, w.d_i, w.act, w.dtype)
    Y, saved, H, g = _run(gpu_lib, inp, bias, w.act, w.dtype)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 16, replace=False)]))
    units = np.unique(np.concatenate([[0, w.dff - 1], rng.choice(w.dff, 16, replace=False)]))
    kw = dict(act=w.act, W3=inp.W3, b1=bias["b1"], b3=bias["b3"])
    Yr, dXr = oracle.rows(inp.X, inp.W1, inp.W2, inp.dY, rows, b2=bias["b2"], **kw)
    c1, c3, c2, g1, g3 = oracle.wgrad_units(inp.X, inp.W1, inp.W2, inp.dY, units, with_bias_grads=True, **kw)
    errs = {"Y": rel_err(to_np(Y)[rows], Yr), "dX": rel_err(to_np(g["dX"])[rows], dXr),
            "dW1": rel_err(cat_cols(g["dW1"])[:, units].T, c1), "dW2": rel_err(cat_rows(g["dW2"])[units], c2),
            "db1": rel_err(np.concatenate([to_np(x) for x in g["db1"]])[units], g1),
            "db2": rel_err(to_np(g["db2"]), oracle.db2(inp.dY))}
    if w.act == "swiglu":
        errs["db3"] = rel_err(np.concatenate([to_np(x) for x in g["db3"]])[units], g3)
    bad = {k: v for k, v in errs.items() if not v <= 2e-2}
    assert not bad, f"{w.name}: {bad} (all {errs})"


@pytest.mark.parametrize("dtype,d,d_i", [
    ("bf16", 8192, (1024, 1024)),  # db2: 128-byte strips, 4 rows ahead; db1: 128-byte strips, 8 rows ahead
    ("bf16", 1536, (256, 256)),    # db2: 64-byte strips; db1: 32-byte strips
    ("fp32", 4096, (512, 512)),    # the same four launch shapes with 4-byte elements
    ("fp32", 768, (128, 128)),
])
def test_bias_colsum_launch_shapes(gpu_lib, dtype, d, d_i):
    """The column sums run in one of four launch shapes chosen by the number
    of columns (strip width 128, 64 or 32 bytes; 4 or 8 rows in flight); a few
    tokens and wide matrices reach each of them."""
    _check(gpu_lib, 16, d, d_i, "gelu", dtype, seed=29)
