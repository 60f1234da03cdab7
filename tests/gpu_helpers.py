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


# ---------------------------------------------------------------- tile-complete samples
# The tensor-core launches compute 256 x 256 output tiles (SwiGLU forward:
# 256 x 128), each drained by 16 epilogue warps of 32 rows (two CTAs x four
# TMEM lane quarters, two column halves).  A sampled token row is compared
# over all of its columns, so it checks every N-tile of its 256-row band in
# the outputs indexed by tokens (Y, dX, A/G/U, H, dA/dU); a sampled hidden
# unit j is compared over a whole column of dW1/dW3 and a whole row of dW2, so
# it checks every tile of its 256-wide band of the shard in those outputs.

TILE = 256
WARP_ROWS = 32


def tile_rows(T: int, seed: int = 7, per_band: int = 1):
    """Token rows with at least `per_band` in every 256-row band.  Band b's
    first row sits in the 32-row warp slot (b mod 8), so the bands together
    reach every epilogue warp's rows; further rows of a band go to the next
    slots.  Also the first and the last row.  Sorted, unique."""
    rng = np.random.default_rng(seed)
    rows = {0, T - 1}
    for b in range((T + TILE - 1) // TILE):
        for k in range(per_band):
            lo = b * TILE + ((b + k) % (TILE // WARP_ROWS)) * WARP_ROWS
            hi = min(lo + WARP_ROWS, T)
            if lo >= T:  # ragged last band: any of its rows
                lo, hi = b * TILE, T
            rows.add(int(rng.integers(lo, hi)))
    return np.array(sorted(rows), dtype=np.int64)


def band_rows(T: int, band: int):
    """One row in each of the eight 32-row warp slots of a 256-row band (that exist)."""
    out = [band * TILE + s * WARP_ROWS + (s * 5) % WARP_ROWS for s in range(TILE // WARP_ROWS)]
    return [r for r in out if r < T]


def tile_units(d_i, seed: int = 7):
    """Hidden units with one in every 256-wide band of every shard, plus each
    shard's first and last unit.  Sorted, unique, global unit indices."""
    import synthetic_inputs as si
    rng = np.random.default_rng(seed)
    units = set()
    for lo, hi in si.shard_slices(d_i):
        units.update((lo, hi - 1))
        for b0 in range(lo, hi, TILE):
            units.add(int(rng.integers(b0, min(b0 + TILE, hi))))
    return np.array(sorted(units), dtype=np.int64)


def rows_of(ts, rows):
    """Rows of a list of per-shard [T x d_i] device tensors, side by side (fp64 numpy)."""
    idx = torch.as_tensor(rows, device=ts[0].device)
    return torch.cat([t.index_select(0, idx).to(torch.float64) for t in ts], dim=1).cpu().numpy()


def dev_rel_err(got: torch.Tensor, ref: torch.Tensor) -> float:
    """rel_err of two device tensors without leaving the device (fp32 arithmetic)."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.numel() == 0:
        return 0.0
    g, r = got.float(), ref.float()
    scale = float(r.abs().max())
    diff = float((g - r).abs().max())
    return diff if scale == 0.0 else diff / scale
