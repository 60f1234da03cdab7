"""GPU edge cases: empty batches, determinism, argument errors with a device
present, launch accounting, and the device status word."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import cat_cols, rel_err, run_gpu, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_empty_token_batch(gpu_lib, act, dtype):
    tp = gpu_lib
    d, d_i = 64, (64, 32)
    mlp = tp.ShardedMLP(0, d, d_i, act, dtype)
    td = mlp.tdtype
    X = torch.empty(0, d, dtype=td, device="cuda")
    W1 = [torch.randn(d, w, device="cuda").to(td) for w in d_i]
    W2 = [torch.randn(w, d, device="cuda").to(td) for w in d_i]
    W3 = [torch.randn(d, w, device="cuda").to(td) for w in d_i] if act == "swiglu" else None
    Y, saved, H = mlp.forward(X, W1, W2, W3)
    out = mlp.alloc_backward()
    for x in out[2] + out[4] + (out[3] or []):
        x.fill_(7)
    g = mlp.backward(X, W1, W2, saved, H, torch.empty(0, d, dtype=td, device="cuda"), W3, out=out)
    torch.cuda.synchronize()
    mlp.check()
    assert Y.shape == (0, d) and g["dX"].shape == (0, d)
    for x in g["dW1"] + g["dW2"] + (g["dW3"] or []):
        assert torch.count_nonzero(x) == 0


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bitwise_determinism(gpu_lib, act):
    inp = si.make_inputs(700, 256, (384, 256, 128), act, "bf16", seed=99)
    a = run_gpu(gpu_lib, inp, act, "bf16")
    b = run_gpu(gpu_lib, inp, act, "bf16")
    assert torch.equal(a["Y"], b["Y"]) and torch.equal(a["dX"], b["dX"])
    for k in ("dW1", "dW2", "H", "saved", "dact"):
        for x, y in zip(a[k], b[k]):
            assert torch.equal(x, y)


def test_launch_count(gpu_lib):
    tp = gpu_lib
    inp = si.make_inputs(256, 64, (64, 64), "gelu", "bf16")
    run_gpu(tp, inp, "gelu", "bf16")
    assert tp.tpmlp_last_launch_count() == 2  # the backward call: dgrad + fsum kernels


def test_status_word_clear_after_normal_runs(gpu_lib):
    tp = gpu_lib
    inp = si.make_inputs(300, 128, (128, 64), "swiglu", "bf16")
    g = run_gpu(tp, inp, "swiglu", "bf16")
    ws = g["mlp"].workspace
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_argument_errors_with_device(gpu_lib):
    tp = gpu_lib
    mlp = tp.ShardedMLP(64, 64, (64,), "gelu", "bf16")
    X = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    W1 = [torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")]
    W2 = [torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")]
    Y, saved, H = mlp.alloc_forward()
    # misaligned X (offset by one element = 2 bytes)
    raw = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(mlp.plan, raw.data_ptr() + 2, W1, None, W2, None, None, None, Y, saved, H, mlp.workspace)
    assert e.value.status == 3
    # null weight
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(mlp.plan, X, [0], None, W2, None, None, None, Y, saved, H, mlp.workspace)
    assert e.value.status == 1
    # null workspace
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(mlp.plan, X, W1, None, W2, None, None, None, Y, saved, H, 0)
    assert e.value.status == 1
    # SwiGLU plan without W3
    ms = tp.ShardedMLP(64, 64, (64,), "swiglu", "bf16")
    Ys, saveds, Hs = ms.alloc_forward()
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(ms.plan, X, W1, None, W2, None, None, None, Ys, saveds, Hs, ms.workspace)
    assert e.value.status == 1


def test_phase_entry_points_match_fused_calls(gpu_lib):
    """tpmlp_forward == forward_column + forward_row; tpmlp_backward == dgrad + fsum."""
    tp = gpu_lib
    inp = si.make_inputs(384, 128, (192, 64), "gelu", "bf16", seed=5)
    ref = run_gpu(tp, inp, "gelu", "bf16")
    mlp = ref["mlp"]
    X = inp.X.cuda(); dY = inp.dY.cuda()
    sl = si.shard_slices(inp.d_i)
    W1 = [inp.W1[:, a:b].contiguous().cuda() for a, b in sl]
    W2 = [inp.W2[a:b].contiguous().cuda() for a, b in sl]
    Y, saved, H = mlp.alloc_forward()
    tp.tpmlp_forward_column(mlp.plan, X, W1, None, None, None, saved, H, mlp.workspace)
    tp.tpmlp_forward_row(mlp.plan, W2, None, H, Y, mlp.workspace)
    dact, dX, dW1, dW3, dW2 = mlp.alloc_backward()
    tp.tpmlp_backward_dgrad(mlp.plan, W2, saved, H, dY, dact, dW2, None, mlp.workspace)
    tp.tpmlp_backward_fsum(mlp.plan, X, W1, None, dact, dX, dW1, None, None, None, mlp.workspace)
    torch.cuda.synchronize()
    assert torch.equal(Y, ref["Y"]) and torch.equal(dX, ref["dX"])
    for x, y in zip(dW1 + dW2, ref["dW1"] + ref["dW2"]):
        assert torch.equal(x, y)


def test_autograd_function(gpu_lib):
    tp = gpu_lib
    inp = si.make_inputs(256, 64, (96, 32), "swiglu", "bf16", seed=3)
    mlp = tp.ShardedMLP(256, 64, inp.d_i, "swiglu", "bf16")
    X = inp.X.cuda().requires_grad_(True)
    W1 = [w.cuda().requires_grad_(True) for w in inp.W1_i]
    W2 = [w.cuda().requires_grad_(True) for w in inp.W2_i]
    W3 = [w.cuda().requires_grad_(True) for w in inp.W3_i]
    Y = tp.TPMLPFunction.apply(mlp, X, *W1, *W2, *W3)
    Y.backward(inp.dY.cuda())
    b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, act="swiglu", W3=inp.W3)
    assert rel_err(to_np(X.grad), b["dX"]) <= 2e-2
    assert rel_err(np.concatenate([to_np(w.grad) for w in W1], 1), b["dW1"]) <= 2e-2
    assert rel_err(np.concatenate([to_np(w.grad) for w in W3], 1), b["dW3"]) <= 2e-2
