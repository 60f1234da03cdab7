"""Failure detection on the GPU without a fault: an injected stall (the
producers load nothing, or the stream-K parts are never published: a flag
nothing sets) makes a bounded wait run out; the kernel records a timeout in the workspace status word, all
roles leave, TMEM is freed and the context stays usable."""
import time

import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import cat_cols, rel_err, to_np

pytestmark = pytest.mark.gpu


def test_injected_stall_reports_timeout_and_context_survives(gpu_lib):
    tp = gpu_lib
    T, d, d_i = 512, 128, (128, 64)
    inp = si.make_inputs(T, d, d_i, "gelu", "bf16", seed=77)
    mlp = tp.ShardedMLP(T, d, d_i, "gelu", "bf16")
    X = inp.X.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    tp.tpmlp_plan_set_timeout(mlp.plan, 25)
    tp.tpmlp_plan_set_stall_injection(mlp.plan, True)
    Y, saved, H = mlp.alloc_forward()
    t0 = time.time()
    tp.tpmlp_forward(mlp.plan, X, W1, None, W2, None, None, None, Y, saved, H, mlp.workspace)  # asynchronous
    with pytest.raises(tp.TpmlpError) as e:
        mlp.check()
    assert e.value.status == 6  # TPMLP_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 10.0
    mlp.check()  # the status word was cleared
    # the context is intact: a normal run on the same plan gives the right answer
    tp.tpmlp_plan_set_stall_injection(mlp.plan, False)
    tp.tpmlp_plan_set_timeout(mlp.plan, 2000)
    Y, saved, H = mlp.forward(X, W1, W2)
    torch.cuda.synchronize()
    mlp.check()
    f = oracle.forward(inp.X, inp.W1, inp.W2)
    assert rel_err(to_np(Y), f["Y"]) <= 2e-2
    assert rel_err(cat_cols(H), f["H"]) <= 2e-2


def test_withheld_stream_k_parts_report_timeout_and_flags_clear(gpu_lib):
    """The stream-K tail forced on, and its parts never published (injection
    2): the owners' bounded waits on another pair's flags run out, the kernel
    records a timeout and leaves; tpmlp_check clears the status word and the
    flags, and the next run on the same workspace is right."""
    tp = gpu_lib
    T, d, d_i = 1000, 384, (256, 128)
    inp = si.make_inputs(T, d, d_i, "gelu", "bf16", seed=78)
    mlp = tp.ShardedMLP(T, d, d_i, "gelu", "bf16")
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_ALWAYS)
    X = inp.X.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    tp.tpmlp_plan_set_timeout(mlp.plan, 100)
    tp.tpmlp_plan_set_stall_injection(mlp.plan, 2)
    Y, saved, H = mlp.alloc_forward()
    t0 = time.time()
    tp.tpmlp_forward(mlp.plan, X, W1, None, W2, None, None, None, Y, saved, H, mlp.workspace)
    with pytest.raises(tp.TpmlpError) as e:
        mlp.check()
    assert e.value.status == 6  # TPMLP_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 10.0
    mlp.check()
    tp.tpmlp_plan_set_stall_injection(mlp.plan, False)
    tp.tpmlp_plan_set_timeout(mlp.plan, 2000)
    Y, saved, H = mlp.forward(X, W1, W2)
    torch.cuda.synchronize()
    mlp.check()
    f = oracle.forward(inp.X, inp.W1, inp.W2)
    assert rel_err(to_np(Y), f["Y"]) <= 2e-2
    assert rel_err(cat_cols(H), f["H"]) <= 2e-2


def test_timeout_setter_validates(gpu_lib):
    tp = gpu_lib
    mlp = tp.ShardedMLP(64, 64, (64,), "gelu", "bf16")
    with pytest.raises(tp.TpmlpError):
        tp.tpmlp_plan_set_timeout(mlp.plan, 0)
