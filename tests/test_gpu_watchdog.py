"""Failure detection on the GPU without a fault: an injected stall (the
producers load nothing: a barrier nothing completes) makes a bounded wait run
out; the kernel records a timeout in the workspace status word, all roles
leave, TMEM is freed and the context stays usable.  The stream-K tail has no
cross-pair wait at all: late parts (injection 2) change nothing."""
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


def test_late_stream_k_parts_still_give_the_same_result(gpu_lib):
    """The stream-K tail forced on, and every part of a split tile but its first
    delayed by 20 ms (injection 2), as CTA pairs that are not resident, or run
    late behind another kernel, would be: nobody waits for them; the last part
    to arrive adds all parts in K order.  The outputs equal, bit for bit, a run
    without the delay (the order of the sum is fixed), match the oracle, and
    the status stays clean."""
    tp = gpu_lib
    T, d, d_i = 1000, 384, (256, 128)
    inp = si.make_inputs(T, d, d_i, "gelu", "bf16", seed=78)
    mlp = tp.ShardedMLP(T, d, d_i, "gelu", "bf16")
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_ALWAYS)
    X, dY = inp.X.cuda(), inp.dY.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    Y0, saved0, H0 = mlp.forward(X, W1, W2)
    g0 = mlp.backward(X, W1, W2, saved0, H0, dY)
    torch.cuda.synchronize()
    mlp.check()
    assert tp.tpmlp_last_split_tiles(tp.LAUNCH_BWD_FSUM), "the f-sum launch was expected to split tiles"
    tp.tpmlp_plan_set_stall_injection(mlp.plan, 2)
    Y, saved, H = mlp.forward(X, W1, W2)
    g = mlp.backward(X, W1, W2, saved, H, dY)
    torch.cuda.synchronize()
    mlp.check()  # no timeout: nobody waited for the late parts
    tp.tpmlp_plan_set_stall_injection(mlp.plan, False)
    assert torch.equal(Y, Y0) and torch.equal(g["dX"], g0["dX"])
    for k in ("dW1", "dW2", "dact"):
        for a, b in zip(g[k], g0[k]):
            assert torch.equal(a, b), k
    for a, b in zip(H, H0):
        assert torch.equal(a, b)
    f = oracle.forward(inp.X, inp.W1, inp.W2)
    b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY)
    assert rel_err(to_np(Y), f["Y"]) <= 2e-2
    assert rel_err(to_np(g["dX"]), b["dX"]) <= 2e-2
    assert rel_err(cat_cols(g["dW1"]), b["dW1"]) <= 2e-2


def test_stale_ticket_counts_do_not_change_the_result(gpu_lib):
    """Ticket counts left in the workspace by an aborted launch (simulated by
    filling the counter block with garbage on the host) read as zero in the
    next launch, whose counts carry a new epoch: the outputs equal a clean
    run's bit for bit."""
    tp = gpu_lib
    T, d, d_i = 1000, 384, (256, 128)
    inp = si.make_inputs(T, d, d_i, "gelu", "bf16", seed=79)
    mlp = tp.ShardedMLP(T, d, d_i, "gelu", "bf16")
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_ALWAYS)
    X, dY = inp.X.cuda(), inp.dY.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    Y0, saved0, H0 = mlp.forward(X, W1, W2)
    g0 = mlp.backward(X, W1, W2, saved0, H0, dY)
    torch.cuda.synchronize()
    mlp.check()
    gen = torch.Generator(device="cpu").manual_seed(5)
    mlp.workspace[256:8192] = torch.randint(0, 256, (8192 - 256,), generator=gen, dtype=torch.uint8).cuda()
    Y, saved, H = mlp.forward(X, W1, W2)
    g = mlp.backward(X, W1, W2, saved, H, dY)
    torch.cuda.synchronize()
    mlp.check()
    assert torch.equal(Y, Y0) and torch.equal(g["dX"], g0["dX"])
    for k in ("dW1", "dW2", "dact"):
        for a, b in zip(g[k], g0[k]):
            assert torch.equal(a, b), k


def test_timeout_setter_validates(gpu_lib):
    tp = gpu_lib
    mlp = tp.ShardedMLP(64, 64, (64,), "gelu", "bf16")
    with pytest.raises(tp.TpmlpError):
        tp.tpmlp_plan_set_timeout(mlp.plan, 0)
