"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import synthetic_inputs as si

BF16_TOL = 2e-2  # max|err| <= 2e-2 * max|ref| (bf16 storage, fp32 accumulation)
FP32_TOL = 1e-4  # max|err| <= 1e-4 * max|ref| (fp32 storage and accumulation)


def tol_for(dtype: str) -> float:
    return BF16_TOL if dtype == "bf16" else FP32_TOL


def rel_err(got, ref) -> float:
    """max|got - ref| / max|ref| (0 when both are all zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    diff = float(np.max(np.abs(got - ref)))
    if scale == 0.0:
        return diff
    return diff / scale


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu", torch.float64).numpy()


def run_gpu(tp, inp: si.Inputs, act: str, dtype: str, d_i=None, device="cuda", stream_k=None):
    """Forward + backward through the binding.  Returns a dict of device tensors.
    stream_k: the plan's stream-K mode (None: the default, automatic)."""
    d_i = tuple(d_i if d_i is not None else inp.d_i)
    T, d = inp.X.shape
    mlp = tp.ShardedMLP(T, d, d_i, act, dtype, device=device)
    if stream_k is not None:
        tp.tpmlp_plan_set_stream_k(mlp.plan, stream_k)
    X = inp.X.to(device)
    dY = inp.dY.to(device)
    sl = si.shard_slices(d_i)
    W1_i = [inp.W1[:, a:b].contiguous().to(device) for a, b in sl]
    W2_i = [inp.W2[a:b, :].contiguous().to(device) for a, b in sl]
    W3_i = [inp.W3[:, a:b].contiguous().to(device) for a, b in sl] if act == "swiglu" else None
    Y, saved, H = mlp.forward(X, W1_i, W2_i, W3_i)
    g = mlp.backward(X, W1_i, W2_i, saved, H, dY, W3_i)
    torch.cuda.synchronize()
    mlp.check()
    out = {"Y": Y, "H": H, "saved": saved, "dX": g["dX"], "dW1": g["dW1"], "dW2": g["dW2"], "dW3": g["dW3"],
           "dact": g["dact"], "mlp": mlp}
    return out


def cat_cols(ts):
    return torch.cat([t.to("cpu", torch.float64) for t in ts], dim=1).numpy()


def cat_rows(ts):
    return torch.cat([t.to("cpu", torch.float64) for t in ts], dim=0).numpy()
