"""The workspace-free row-parallel GEMM entry point.

tpmlp_forward_row_noalloc serves callers that cannot allocate device memory
(code handed only its input and output buffers by a framework that owns the
allocator, or callers that must not call cudaMalloc because it synchronises
the device): its scratch status word is a library-owned static device array
instead of a caller workspace.  Through the C ABI, two calls in a row must
give the output of the workspace entry point tpmlp_forward_row within the
bf16 tolerance of the parity tests.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import pytest
import torch

import synthetic_inputs as si
from gpu_helpers import BF16_TOL, rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_forward_row_noalloc_matches_workspace_entry_point(gpu_lib, act):
    tp = gpu_lib
    T, d, d_i = 1000, 384, (512, 136, 384)
    inp = si.make_inputs(T, d, d_i, act, "bf16", seed=2024)
    mlp = tp.ShardedMLP(T, d, d_i, act, "bf16")
    X = inp.X.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    W3 = [w.cuda() for w in inp.W3_i] if act == "swiglu" else None
    Y_ref, saved, H = mlp.alloc_forward()
    tp.tpmlp_forward_column(mlp.plan, X, W1, W3, None, None, saved, H, mlp.workspace)
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
