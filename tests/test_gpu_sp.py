"""GPU parity of the sequence-parallel layout (X and dY read from token
stripes, Y and dX written as stripes) against the fp64 oracle's SP form,
through the C ABI, and its equality with the dense layout: the stripes only
change where rows live, so on the same inputs the GPU results equal the dense
entry points' bit for bit (except db2, whose column sum walks the stripes in
another order)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import cat_cols, cat_rows, rel_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def _cut(M, rows):
    out, r = [], 0
    for n in rows:
        out.append(M[r:r + n].contiguous())
        r += n
    return out


def run_sp(tp, inp, act, dtype, rows, bias=None, stream_k=None):
    T, d = inp.X.shape
    mlp = tp.ShardedMLP(T, d, inp.d_i, act, dtype)
    if stream_k is not None:
        tp.tpmlp_plan_set_stream_k(mlp.plan, stream_k)
    mlp.set_sequence_stripes(rows)
    X_j = [x.cuda() for x in _cut(inp.X, rows)]
    dY_j = [x.cuda() for x in _cut(inp.dY, rows)]
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    W3 = [w.cuda() for w in inp.W3_i] if act == "swiglu" else None
    kw = {}
    if bias is not None:
        kw = {"b1_i": [b.cuda() for b in bias["b1_i"]], "b2": bias["b2"].cuda(),
              "b3_i": [b.cuda() for b in bias["b3_i"]] if act == "swiglu" else None}
    Y_j, saved, H = mlp.forward_sp(X_j, W1, W2, W3, **kw)
    g = mlp.backward_sp(X_j, W1, W2, saved, H, dY_j, W3, bias_grads=bias is not None)
    torch.cuda.synchronize()
    mlp.check()
    return Y_j, H, g


CASES = [
    ("gelu", (1000, 384, (256, 128)), [256, 384, 360]),
    ("swiglu", (1000, 256, (128, 64, 64)), [512, 488]),
    ("gelu", (1000, 256, (128, 64)), [0, 512, 0, 488]),
    ("swiglu", (300, 128, (64,)), [300]),
]


@pytest.mark.parametrize("stream_k", [None, "always"])
@pytest.mark.parametrize("act,shape,rows", CASES)
def test_sp_matches_oracle(gpu_lib, act, shape, rows, stream_k):
    """stream_k "always": the stream-K tail on every launch, so that parts
    start inside the MN-major token walks across the stripes."""
    T, d, d_i = shape
    inp = si.make_inputs(T, d, d_i, act, "bf16", seed=31)
    bias = si.make_biases(d, d_i, act, "bf16", seed=31)
    Y_j, H, g = run_sp(gpu_lib, inp, act, "bf16", rows, bias,
                       stream_k=gpu_lib.STREAM_K_ALWAYS if stream_k else None)
    W3 = inp.W3_i if act == "swiglu" else None
    b3 = bias["b3_i"] if act == "swiglu" else None
    Yr_j, H_r = oracle.forward_sp(_cut(inp.X, rows), inp.W1_i, inp.W2_i, act=act, W3_i=W3, b1_i=bias["b1_i"],
                                  b3_i=b3, b2=bias["b2"])
    br = oracle.backward_sp(_cut(inp.X, rows), inp.W1_i, inp.W2_i, _cut(inp.dY, rows), act=act, W3_i=W3,
                            b1_i=bias["b1_i"], b3_i=b3)
    tol = tol_for("bf16")
    assert [y.shape[0] for y in Y_j] == rows and [x.shape[0] for x in g["dX_stripes"]] == rows
    errs = {"Y": rel_err(cat_rows(Y_j), np.concatenate(Yr_j, 0)),
            "dX": rel_err(cat_rows(g["dX_stripes"]), np.concatenate(br["dX_j"], 0)),
            "H": rel_err(cat_cols(H), np.concatenate(H_r, 1)),
            "dW1": rel_err(cat_cols(g["dW1"]), np.concatenate(br["dW1_i"], 1)),
            "dW2": rel_err(cat_rows(g["dW2"]), np.concatenate(br["dW2_i"], 0)),
            "db1": rel_err(np.concatenate([to_np(x) for x in g["db1"]]), np.concatenate(br["db1_i"])),
            "db2": rel_err(to_np(g["db2"]), br["db2"])}
    if act == "swiglu":
        errs["dW3"] = rel_err(cat_cols(g["dW3"]), np.concatenate(br["dW3_i"], 1))
        errs["db3"] = rel_err(np.concatenate([to_np(x) for x in g["db3"]]), np.concatenate(br["db3_i"]))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{act} {shape} stripes {rows}: over {tol}: {bad} (all: {errs})"


def test_sp_fp32_path(gpu_lib):
    inp = si.make_inputs(300, 64, (32, 32), "gelu", "fp32", seed=4)
    rows = [128, 172]
    Y_j, H, g = run_sp(gpu_lib, inp, "gelu", "fp32", rows)
    Yr_j, _ = oracle.forward_sp(_cut(inp.X, rows), inp.W1_i, inp.W2_i, act="gelu")
    br = oracle.backward_sp(_cut(inp.X, rows), inp.W1_i, inp.W2_i, _cut(inp.dY, rows), act="gelu")
    tol = tol_for("fp32")
    assert rel_err(cat_rows(Y_j), np.concatenate(Yr_j, 0)) <= tol
    assert rel_err(cat_rows(g["dX_stripes"]), np.concatenate(br["dX_j"], 0)) <= tol
    assert rel_err(cat_cols(g["dW1"]), np.concatenate(br["dW1_i"], 1)) <= tol


@pytest.mark.parametrize("name", ["C5", "C4"])
def test_sp_equals_dense_layout_full_size(gpu_lib, name):
    """At the full workload with t stripes of T/t tokens (the pages' layout), the
    SP entry points give the dense entry points' results bit for bit."""
    tp = gpu_lib
    w = si.WORKLOADS[name]
    inp = si.make_workload_inputs(w)
    rows = [w.T // w.t] * w.t
    mlp = tp.ShardedMLP(w.T, w.d, w.d_i, w.act, w.dtype)
    X, dY = inp.X.cuda(), inp.dY.cuda()
    W1 = [x.cuda() for x in inp.W1_i]
    W2 = [x.cuda() for x in inp.W2_i]
    W3 = [x.cuda() for x in inp.W3_i] if w.act == "swiglu" else None
    Y, saved, H = mlp.forward(X, W1, W2, W3)
    g = mlp.backward(X, W1, W2, saved, H, dY, W3)
    torch.cuda.synchronize()
    mlp.set_sequence_stripes(rows)
    X_j = list(X.split(rows))
    dY_j = list(dY.split(rows))
    Y_j, saved_sp, H_sp = mlp.forward_sp([x.contiguous() for x in X_j], W1, W2, W3)
    g_sp = mlp.backward_sp([x.contiguous() for x in X_j], W1, W2, saved_sp, H_sp, [x.contiguous() for x in dY_j], W3)
    torch.cuda.synchronize()
    mlp.check()
    assert torch.equal(torch.cat(Y_j, 0), Y)
    assert torch.equal(torch.cat(g_sp["dX_stripes"], 0), g["dX"])
    for k in ("dW1", "dW2") + (("dW3",) if w.act == "swiglu" else ()):
        for a, b in zip(g_sp[k], g[k]):
            assert torch.equal(a, b), k
    for a, b in zip(H_sp, H):
        assert torch.equal(a, b)


def test_sp_argument_errors(gpu_lib):
    tp = gpu_lib
    mlp = tp.ShardedMLP(256, 64, (64,), "gelu", "bf16")
    W1 = [torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")]
    W2 = [torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")]
    X_j = [torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(tp.TpmlpError) as e:  # no stripes set on the plan
        mlp.forward_sp(X_j, W1, W2)
    assert e.value.status == 1
    mlp.set_sequence_stripes([128, 128])
    with pytest.raises(tp.TpmlpError) as e:  # a non-empty stripe without a buffer
        tp.tpmlp_forward_sp(mlp.plan, [X_j[0], 0], W1, None, W2, None, None, None, mlp.alloc_stripes(),
                            *mlp.alloc_forward()[1:], mlp.workspace)
    assert e.value.status == 1
