"""Backward with recomputation (tpmlp_backward_recompute): H is not read;
the dgrad launch rewrites H_i from the saved pre-activations and the second
launch takes dW2 from it.  H is filled with NaN before the backward, so any
read of the forward's H would poison the gradients."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import cat_cols, cat_rows, rel_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def _fwd(tp, inp, act, dtype, bias=None, stream_k=None):
    T, d = inp.X.shape
    mlp = tp.ShardedMLP(T, d, inp.d_i, act, dtype)
    if stream_k is not None:
        tp.tpmlp_plan_set_stream_k(mlp.plan, stream_k)
    cu = lambda xs: [x.cuda() for x in xs] if xs is not None else None
    X, dY = inp.X.cuda(), inp.dY.cuda()
    W1, W2, W3 = cu(inp.W1_i), cu(inp.W2_i), cu(inp.W3_i)
    kw = {}
    if bias is not None:
        kw = dict(b1_i=cu(bias["b1_i"]), b3_i=cu(bias["b3_i"]), b2=bias["b2"].cuda())
    Y, saved, H = mlp.forward(X, W1, W2, W3, **kw)
    return mlp, X, dY, W1, W2, W3, Y, saved, H


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("dtype,stream_k", [("bf16", False), ("bf16", True), ("fp32", False)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_recompute_matches_oracle(gpu_lib, act, dtype, stream_k, with_bias):
    """stream_k: the stream-K tail forced on every launch (the H-writing dgrad
    epilogue and the f-sum launch carrying dW2 then run on split tiles)."""
    tp = gpu_lib
    T, d, d_i = (333, 200, (8, 96, 264, 152)) if dtype == "bf16" else (45, 36, (20, 44))
    inp = si.make_inputs(T, d, d_i, act, dtype, seed=17)
    bias = si.make_biases(d, d_i, act, dtype, seed=17) if with_bias else None
    mlp, X, dY, W1, W2, W3, Y, saved, H = _fwd(tp, inp, act, dtype, bias,
                                               stream_k=tp.STREAM_K_ALWAYS if stream_k else None)
    for h in H:
        h.fill_(float("nan"))
    g = mlp.backward(X, W1, W2, saved, H, dY, W3, bias_grads=with_bias, recompute=True)
    torch.cuda.synchronize()
    mlp.check()
    kw = dict(act=act, W3=inp.W3)
    if with_bias:
        kw.update(b1=bias["b1"], b3=bias["b3"], b2=bias["b2"])
    f = oracle.forward(inp.X, inp.W1, inp.W2, **kw)
    b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, **kw)
    errs = {"H": rel_err(cat_cols(H), f["H"]), "dX": rel_err(to_np(g["dX"]), b["dX"]),
            "dW1": rel_err(cat_cols(g["dW1"]), b["dW1"]), "dW2": rel_err(cat_rows(g["dW2"]), b["dW2"])}
    if act == "swiglu":
        errs["dW3"] = rel_err(cat_cols(g["dW3"]), b["dW3"])
    if with_bias:
        errs["db1"] = rel_err(np.concatenate([to_np(x) for x in g["db1"]]), b["db1"])
        errs["db2"] = rel_err(to_np(g["db2"]), b["db2"])
    tol = tol_for(dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"over tolerance {tol}: {bad} (all {errs})"


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_recompute_same_activation_gradients(gpu_lib, act):
    """dact, dX and dW1 (dW3) come from identical arithmetic in both modes.
    With the stream-K tail off: recompute moves the dW2 tiles into the second
    launch, and the tail cuts that launch's tiles differently."""
    tp = gpu_lib
    inp = si.make_inputs(1024, 384, (512, 384, 640, 256), act, "bf16", seed=23)
    mlp, X, dY, W1, W2, W3, Y, saved, H = _fwd(tp, inp, act, "bf16", stream_k=tp.STREAM_K_OFF)
    ref = mlp.backward(X, W1, W2, saved, H, dY, W3)
    H2 = [torch.full_like(h, float("nan")) for h in H]
    rec = mlp.backward(X, W1, W2, saved, H2, dY, W3, recompute=True)
    torch.cuda.synchronize()
    assert torch.equal(ref["dX"], rec["dX"])
    for k in ("dact", "dW1") + (("dW3",) if act == "swiglu" else ()):
        for x, y in zip(ref[k], rec[k]):
            assert torch.equal(x, y), k
    for x, y in zip(ref["dW2"], rec["dW2"]):
        assert rel_err(to_np(y), to_np(x)) <= 1e-2


@pytest.mark.parametrize("name", ["C4", "C5"])
def test_recompute_workload_sampled(gpu_lib, name):
    w = si.WORKLOADS[name]
    inp = si.make_workload_inputs(w)
    mlp, X, dY, W1, W2, W3, Y, saved, H = _fwd(gpu_lib, inp, w.act, w.dtype)
    for h in H:
        h.fill_(float("nan"))
    g = mlp.backward(X, W1, W2, saved, H, dY, W3, recompute=True)
    torch.cuda.synchronize()
    mlp.check()
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 12, replace=False)]))
    units = np.unique(np.concatenate([[0, w.dff - 1], rng.choice(w.dff, 12, replace=False)]))
    Yr, dXr = oracle.rows(inp.X, inp.W1, inp.W2, inp.dY, rows, act=w.act, W3=inp.W3)
    c1, c3, c2 = oracle.wgrad_units(inp.X, inp.W1, inp.W2, inp.dY, units, act=w.act, W3=inp.W3)
    errs = {"dX": rel_err(to_np(g["dX"])[rows], dXr), "dW1": rel_err(cat_cols(g["dW1"])[:, units].T, c1),
            "dW2": rel_err(cat_rows(g["dW2"])[units], c2)}
    if w.act == "swiglu":
        errs["dW3"] = rel_err(cat_cols(g["dW3"])[:, units].T, c3)
    bad = {k: v for k, v in errs.items() if not v <= 2e-2}
    assert not bad, f"{w.name}: {bad} (all {errs})"


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_recompute_sixteen_shards(gpu_lib, act, dtype):
    """The largest launch tables: the recompute f-sum launch carries dW2_i next
    to dW1_i, dW3_i and dX, 3t + 1 problems and 5t segments for SwiGLU at
    t = 16 (bf16: more tensor maps than one launch holds, so dW2 gets a launch
    of its own).  Compared with the oracle on every output."""
    tp = gpu_lib
    d_i = (8, 16, 8, 24, 8, 8, 16, 8, 8, 8, 32, 8, 8, 16, 8, 8) if dtype == "bf16" else (4, 8) * 8
    T, d = (150, 48) if dtype == "bf16" else (37, 20)
    inp = si.make_inputs(T, d, d_i, act, dtype, seed=31)
    mlp, X, dY, W1, W2, W3, Y, saved, H = _fwd(tp, inp, act, dtype)
    for h in H:
        h.fill_(float("nan"))
    g = mlp.backward(X, W1, W2, saved, H, dY, W3, recompute=True)
    torch.cuda.synchronize()
    mlp.check()
    f = oracle.forward(inp.X, inp.W1, inp.W2, act=act, W3=inp.W3)
    b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, act=act, W3=inp.W3)
    errs = {"Y": rel_err(to_np(Y), f["Y"]), "H": rel_err(cat_cols(H), f["H"]),
            "dX": rel_err(to_np(g["dX"]), b["dX"]), "dW1": rel_err(cat_cols(g["dW1"]), b["dW1"]),
            "dW2": rel_err(cat_rows(g["dW2"]), b["dW2"])}
    if act == "swiglu":
        errs["dW3"] = rel_err(cat_cols(g["dW3"]), b["dW3"])
    tol = tol_for(dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"over tolerance {tol}: {bad} (all {errs})"
