"""The workspace-free row-parallel GEMM entry point.

tpmlp_forward_row_noalloc serves callers that cannot allocate device memory
(code handed only its input and output buffers by a framework that owns the
allocator, or callers that must not call cudaMalloc because it synchronises
the device): its scratch status word is a library-owned static device array
instead of a caller workspace.  Through the C ABI, two calls in a row must
give the output of the workspace entry point tpmlp_forward_row within the
bf16 tolerance of the parity tests.  Further cases: the oracle's Y for bf16
and fp32 plans, T = 0, a ragged multi-wave shape where the workspace entry
point cuts a stream-K tail (the static-scratch call never does, so it must
equal the workspace call with the tail off bit for bit), and a bounded wait
that runs out: the call itself reports the timeout, and the next call clears
the static status word and succeeds.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import BF16_TOL, rel_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def _setup(tp, T, d, d_i, act, dtype, seed):
    inp = si.make_inputs(T, d, d_i, act, dtype, seed=seed)
    mlp = tp.ShardedMLP(T, d, d_i, act, dtype)
    X = inp.X.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    W3 = [w.cuda() for w in inp.W3_i] if act == "swiglu" else None
    Y_ref, saved, H = mlp.alloc_forward()
    tp.tpmlp_forward_column(mlp.plan, X, W1, W3, None, None, saved, H, mlp.workspace)
    return inp, mlp, W2, Y_ref, H


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_forward_row_noalloc_matches_workspace_entry_point(gpu_lib, act):
    tp = gpu_lib
    inp, mlp, W2, Y_ref, H = _setup(tp, 1000, 384, (512, 136, 384), act, "bf16", 2024)
    tp.tpmlp_forward_row(mlp.plan, W2, None, H, Y_ref, mlp.workspace)
    torch.cuda.synchronize()
    mlp.check()
    ref = to_np(Y_ref)
    for call in range(2):
        Y = torch.full_like(Y_ref, float("nan"))
        tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
        torch.cuda.synchronize()
        err = rel_err(to_np(Y), ref)
        assert err <= BF16_TOL, f"call {call}: max|err| / max|ref| = {err}"
        assert torch.isfinite(Y).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_forward_row_noalloc_matches_oracle(gpu_lib, act, dtype):
    tp = gpu_lib
    T, d, d_i = (333, 200, (8, 96, 264, 152)) if dtype == "bf16" else (45, 36, (20, 44))
    inp, mlp, W2, Y_ref, H = _setup(tp, T, d, d_i, act, dtype, 41)
    f = oracle.forward(inp.X, inp.W1, inp.W2, act=act, W3=inp.W3)
    for call in range(2):
        Y = torch.full_like(Y_ref, float("nan"))
        tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
        torch.cuda.synchronize()
        err = rel_err(to_np(Y), f["Y"])
        assert err <= tol_for(dtype), f"call {call}: max|err| / max|ref| = {err}"


def test_forward_row_noalloc_zero_tokens(gpu_lib):
    tp = gpu_lib
    mlp = tp.ShardedMLP(0, 64, (64, 128), "gelu", "bf16")
    W2 = [torch.randn(w, 64, device="cuda").bfloat16() for w in (64, 128)]
    Y, _, H = mlp.alloc_forward()
    tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
    tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
    assert tp.tpmlp_last_launch_count() == 0


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_forward_row_noalloc_equals_round_robin_bitwise(gpu_lib, act):
    """A ragged shape with several waves of tiles: the workspace call with the
    stream-K tail forced on splits tiles; the static-scratch call never does,
    and equals the workspace call with the tail off bit for bit."""
    tp = gpu_lib
    inp, mlp, W2, Y_ref, H = _setup(tp, 2000, 520, (1024, 136), act, "bf16", 55)
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_ALWAYS)
    Y_sk = torch.empty_like(Y_ref)
    tp.tpmlp_forward_row(mlp.plan, W2, None, H, Y_sk, mlp.workspace)
    assert tp.tpmlp_last_split_tiles(tp.LAUNCH_FWD_ROW), "the workspace call was expected to split tiles"
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_OFF)
    tp.tpmlp_forward_row(mlp.plan, W2, None, H, Y_ref, mlp.workspace)
    torch.cuda.synchronize()
    mlp.check()
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_ALWAYS)  # ignored by the static-scratch call
    for call in range(2):
        Y = torch.full_like(Y_ref, float("nan"))
        tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
        assert not tp.tpmlp_last_split_tiles(tp.LAUNCH_FWD_ROW)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y_ref), f"call {call}"
    assert rel_err(to_np(Y_sk), to_np(Y_ref)) <= BF16_TOL


def test_forward_row_noalloc_reports_timeout_then_recovers(gpu_lib):
    """Stall injection 1 (the producers load nothing) with a 25 ms bound: the
    call itself returns TPMLP_ERR_DEVICE_TIMEOUT from the static status word;
    the next call, injection off, clears the word and gives the right Y."""
    tp = gpu_lib
    inp, mlp, W2, Y_ref, H = _setup(tp, 512, 128, (128, 64), "gelu", "bf16", 77)
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_OFF)
    tp.tpmlp_forward_row(mlp.plan, W2, None, H, Y_ref, mlp.workspace)
    torch.cuda.synchronize()
    mlp.check()
    tp.tpmlp_plan_set_timeout(mlp.plan, 25)
    tp.tpmlp_plan_set_stall_injection(mlp.plan, 1)
    Y = torch.full_like(Y_ref, float("nan"))
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
    assert e.value.status == 6  # TPMLP_ERR_DEVICE_TIMEOUT
    tp.tpmlp_plan_set_stall_injection(mlp.plan, 0)
    tp.tpmlp_plan_set_timeout(mlp.plan, 2000)
    for call in range(2):
        Y = torch.full_like(Y_ref, float("nan"))
        tp.tpmlp_forward_row_noalloc(mlp.plan, W2, H, Y)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y_ref), f"call {call}"
