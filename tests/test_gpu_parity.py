"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: max|err| <= 2e-2 * max|ref| per output tensor for bf16 storage with fp32
accumulation, 1e-4 * max|ref| for fp32 (the bounds stated for this block).
Small cases are compared element by element on every output; the full-size
workloads are compared on sampled token rows (Y, dX) and sampled hidden
units (columns of dW1 / dW3, rows of dW2), each computed by the oracle from
its own definition, in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import (TILE, band_rows, cat_cols, cat_rows, dev_rel_err, rel_err, rows_of, run_gpu,
                         tile_rows, tile_units, to_np, tol_for)

pytestmark = pytest.mark.gpu


def _full_compare(tp, T, d, d_i, act, dtype, seed=1234, check_intermediates=True, stream_k=None):
    inp = si.make_inputs(T, d, d_i, act, dtype, seed)
    g = run_gpu(tp, inp, act, dtype, stream_k=stream_k)
    f = oracle.forward(inp.X, inp.W1, inp.W2, act=act, W3=inp.W3)
    b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, act=act, W3=inp.W3)
    tol = tol_for(dtype)
    errs = {
        "Y": rel_err(to_np(g["Y"]), f["Y"]),
        "dX": rel_err(to_np(g["dX"]), b["dX"]),
        "dW1": rel_err(cat_cols(g["dW1"]), b["dW1"]),
        "dW2": rel_err(cat_rows(g["dW2"]), b["dW2"]),
    }
    if act == "swiglu":
        errs["dW3"] = rel_err(cat_cols(g["dW3"]), b["dW3"])
    if check_intermediates:
        t = len(d_i)
        errs["H"] = rel_err(cat_cols(g["H"]), f["H"])
        errs["A"] = rel_err(cat_cols(g["saved"][:t]), f["A"])
        errs["dA"] = rel_err(cat_cols(g["dact"][:t]), b["dA"])
        if act == "swiglu":
            errs["U"] = rel_err(cat_cols(g["saved"][t:]), f["U"])
            errs["dU"] = rel_err(cat_cols(g["dact"][t:]), b["dU"])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"over tolerance {tol}: {bad} (all: {errs})"
    return errs


# ------------------------------------------------------------- small, ragged, every tail

SMALL_CASES = [
    # T, d, d_i: tiles of 128 x 256 with ragged tails in M, N and K, unequal shards
    (200, 72, (40, 136, 64)),
    (128, 256, (256,)),
    (333, 200, (8, 96, 264, 152)),
    (64, 64, (64, 64)),
    (257, 136, (120, 392)),
    (1, 8, (8,)),
    (37, 24, (8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8, 8)),  # 16 shards of width 8
]


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("case", SMALL_CASES, ids=[f"T{c[0]}_d{c[1]}_t{len(c[2])}" for c in SMALL_CASES])
def test_small_bf16_all_outputs(gpu_lib, act, case):
    T, d, d_i = case
    _full_compare(gpu_lib, T, d, d_i, act, "bf16")


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_multi_wave_bf16(gpu_lib, act):
    # more tiles than SMs in every launch, several K blocks per shard
    _full_compare(gpu_lib, 1024, 384, (512, 384, 640, 256), act, "bf16")


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("case", [(32, 64, (128, 128)), (45, 36, (20, 44)), (130, 100, (64, 36, 100))])
def test_fp32_path(gpu_lib, act, case):
    T, d, d_i = case
    _full_compare(gpu_lib, T, d, d_i, act, "fp32")


# ------------------------------------------------------------- stream-K tail
# Cases whose launches cut tiles into parts spread over many pairs: parts
# that start inside a later shard's segment (row and dX launches), ragged K
# blocks, partial tiles, SwiGLU tiles in both MMA forms (merged N = 256 for
# full tiles, split for partial ones).
SK_CASES = [
    (1024, 384, (512, 384, 640, 256)),
    (333, 200, (8, 96, 264, 152)),
    (257, 136, (120, 392)),
    (2000, 520, (1024, 136)),
    (640, 1000, (256, 256, 256, 256)),
]


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("case", SK_CASES, ids=[f"T{c[0]}_d{c[1]}_t{len(c[2])}" for c in SK_CASES])
def test_stream_k_always_bf16_all_outputs(gpu_lib, act, case):
    T, d, d_i = case
    _full_compare(gpu_lib, T, d, d_i, act, "bf16", stream_k=gpu_lib.STREAM_K_ALWAYS)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("case", SK_CASES, ids=[f"T{c[0]}_d{c[1]}_t{len(c[2])}" for c in SK_CASES])
def test_stream_k_balance_bf16_all_outputs(gpu_lib, act, case):
    """Every launch spread evenly over the pairs: ranges that end inside one
    tile, cover whole tiles and start inside another (two parts per range),
    the weight-gradient tiles placed after the short ones."""
    T, d, d_i = case
    _full_compare(gpu_lib, T, d, d_i, act, "bf16", stream_k=gpu_lib.STREAM_K_BALANCE)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_stream_k_deterministic_and_within_bound_of_round_robin(gpu_lib, act):
    """The parts of a split tile are added in a fixed order: two runs agree bit
    for bit.  Against plain round robin (one K loop per tile) only the fp32
    summation order differs."""
    T, d, d_i = 1024, 384, (512, 384, 640, 256)
    inp = si.make_inputs(T, d, d_i, act, "bf16", seed=77)
    runs = [run_gpu(gpu_lib, inp, act, "bf16", stream_k=m)
            for m in (gpu_lib.STREAM_K_ALWAYS, gpu_lib.STREAM_K_ALWAYS, gpu_lib.STREAM_K_OFF,
                      gpu_lib.STREAM_K_BALANCE, gpu_lib.STREAM_K_BALANCE)]
    keys = ("Y", "dX")
    lists = ("dW1", "dW2", "H", "saved", "dact") + (("dW3",) if act == "swiglu" else ())
    for k in keys:
        assert torch.equal(runs[0][k], runs[1][k]), k
        assert torch.equal(runs[3][k], runs[4][k]), k
        assert rel_err(to_np(runs[0][k]), to_np(runs[2][k])) <= 1e-2, k
        assert rel_err(to_np(runs[3][k]), to_np(runs[2][k])) <= 1e-2, k
    for k in lists:
        for a, b, c, e, f in zip(runs[0][k], runs[1][k], runs[2][k], runs[3][k], runs[4][k]):
            assert torch.equal(a, b), k
            assert torch.equal(e, f), k
            assert rel_err(to_np(a), to_np(c)) <= 1e-2, k
            assert rel_err(to_np(e), to_np(c)) <= 1e-2, k


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_deal_of_short_tiles(gpu_lib, act):
    """A dgrad launch whose three K = T weight-gradient tiles (64 K blocks)
    come first leaves, on 76 pairs, pairs 0-2 a long tile ahead; the planner
    deals the first round of the 96 short tiles to pairs 3-75 (the Deal walk's
    head phase).  Every output element against the oracle: a tile that the
    walk skipped would show (that each tile is dealt exactly once is checked
    on the host, test_deal_cpu)."""
    _full_compare(gpu_lib, 8192, 256, (256, 256, 256), act, "bf16", seed=41)


def test_config_C1_fp32(gpu_lib):
    w = si.WORKLOADS["C1"]
    _full_compare(gpu_lib, w.T, w.d, w.d_i, w.act, w.dtype)


# ------------------------------------------------------------- full-size workloads (sampled)
# Tile-complete samples (gpu_helpers.tile_rows / tile_units): a token row in
# every 256-row band, cycling over the eight 32-row epilogue-warp slots, and a
# hidden unit in every 256-wide band of every shard; each sampled row is
# compared over all of its columns and each unit over a whole column of dW1
# (dW3) and row of dW2, so every output tile of every launch is checked.
# Tiles the stream-K tail split in the run (tpmlp_last_split_tiles) get a row
# in each of their eight warp slots (or their units, for weight gradients).

def _split_samples(tp, w, g, rows, units):
    """Add rows / units covering every tile the stream-K schedule split in the
    last four launches.  A split tile is identified by its output tensor (the
    address the launch reports).  Returns (rows, units, split) with
    split = {launch: tiles}."""
    offs = [lo for lo, _ in si.shard_slices(w.d_i)]
    token_out = {g["Y"].data_ptr(), g["dX"].data_ptr()} | {x.data_ptr() for x in g["saved"] + g["dact"]}
    dw_rows = {x.data_ptr(): i for i, x in enumerate(g["dW2"])}                    # rows are shard units
    dw_cols = {x.data_ptr(): i for i, x in enumerate(g["dW1"] + (g["dW3"] or []))}  # columns are shard units
    split = {k: tp.tpmlp_last_split_tiles(k) for k in
             (tp.LAUNCH_FWD_COLUMN, tp.LAUNCH_FWD_ROW, tp.LAUNCH_BWD_DGRAD, tp.LAUNCH_BWD_FSUM)}
    add_r, add_u = [], []
    t = len(w.d_i)
    for tiles in split.values():
        for _, m0, n0, out in tiles:
            if out in token_out:
                add_r += band_rows(w.T, m0 // TILE)
            elif out in dw_rows:
                i = dw_rows[out]
                lo, hi = offs[i], offs[i] + w.d_i[i]
                add_u += [u for u in (lo + m0, lo + m0 + 97, lo + m0 + 255) if u < hi]
            elif out in dw_cols:
                i = dw_cols[out] % t
                lo, hi = offs[i], offs[i] + w.d_i[i]
                add_u += [u for u in (lo + n0, lo + n0 + 131, lo + n0 + 255) if u < hi]
            else:
                raise AssertionError(f"split tile of an unknown output {out:#x}")
    rows = np.union1d(rows, np.asarray(add_r, dtype=np.int64))
    units = np.union1d(units, np.asarray(add_u, dtype=np.int64))
    return rows, units, split


def _sampled_compare(tp, w: si.Workload, seed=1234, extra_rows=(), stream_k=None, rows=None, units=None,
                     intermediates=True, tile_complete=True):
    inp = si.make_workload_inputs(w, seed)
    g = run_gpu(tp, inp, w.act, w.dtype, stream_k=stream_k)
    if rows is None:
        rows = tile_rows(w.T)
    rows = np.union1d(rows, np.asarray(extra_rows, dtype=np.int64))
    if units is None:
        units = tile_units(w.d_i)
    rows, units, split = _split_samples(tp, w, g, rows, units)
    Yr, dXr, inter = oracle.rows(inp.X, inp.W1, inp.W2, inp.dY, rows, act=w.act, W3=inp.W3, intermediates=True)
    c1, c3, c2 = oracle.wgrad_units(inp.X, inp.W1, inp.W2, inp.dY, units, act=w.act, W3=inp.W3)
    t = len(w.d_i)
    ridx = torch.as_tensor(rows, device=g["Y"].device)
    Y = g["Y"].index_select(0, ridx).double().cpu().numpy()
    dX = g["dX"].index_select(0, ridx).double().cpu().numpy()
    dW1 = cat_cols(g["dW1"])[:, units].T
    dW2 = cat_rows(g["dW2"])[units, :]
    tol = tol_for(w.dtype)
    errs = {"Y": rel_err(Y, Yr), "dX": rel_err(dX, dXr), "dW1": rel_err(dW1, c1), "dW2": rel_err(dW2, c2)}
    if w.act == "swiglu":
        errs["dW3"] = rel_err(cat_cols(g["dW3"])[:, units].T, c3)
    if intermediates:  # the saved pre-activations, H and the activation gradients
        errs["A"] = rel_err(rows_of(g["saved"][:t], rows), inter["A"])
        errs["H"] = rel_err(rows_of(g["H"], rows), inter["H"])
        errs["dA"] = rel_err(rows_of(g["dact"][:t], rows), inter["dA"])
        if w.act == "swiglu":
            errs["U"] = rel_err(rows_of(g["saved"][t:], rows), inter["U"])
            errs["dU"] = rel_err(rows_of(g["dact"][t:], rows), inter["dU"])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name}: over tolerance {tol}: {bad} (all: {errs})"
    if tile_complete:  # every 256-row band and every 256-wide band of every shard was compared
        assert set(rows // TILE) == set(range((w.T + TILE - 1) // TILE))
        for lo, hi in si.shard_slices(w.d_i):
            assert set((units[(units >= lo) & (units < hi)] - lo) // TILE) == set(range((hi - lo + TILE - 1) // TILE))
    # properties that hold at any size: finite outputs everywhere
    for k in ("Y", "dX"):
        assert torch.isfinite(g[k]).all()
    for k in ("dW1", "dW2", "H", "saved", "dact"):
        assert all(torch.isfinite(x).all() for x in g[k])
    return g, errs, split


@pytest.mark.parametrize("name", ["C2t1", "C2t2", "C2t4", "C3", "C4", "C5"])
def test_workload_sampled_parity(gpu_lib, name):
    _, _, split = _sampled_compare(gpu_lib, si.WORKLOADS[name])
    if name == "C5":
        # the default (automatic) stream-K mode splits the row launch's last
        # wave at this size; its tiles were among the compared ones
        assert split[gpu_lib.LAUNCH_FWD_ROW], "expected the row launch's last wave to be split"


def test_stream_k_soak_bitwise(gpu_lib):
    """60 forward + backward steps with the stream-K tail forced on (parts of
    many tiles exchanged between pairs through the workspace every launch):
    every step's outputs equal the first step's bit for bit -- a lost or
    early-read partial, or a stale flag from the previous launch, would show
    up as a difference."""
    tp = gpu_lib
    T, d, d_i = 1024, 384, (512, 384, 640, 256)
    inp = si.make_inputs(T, d, d_i, "swiglu", "bf16", seed=5)
    mlp = tp.ShardedMLP(T, d, d_i, "swiglu", "bf16")
    tp.tpmlp_plan_set_stream_k(mlp.plan, tp.STREAM_K_ALWAYS)
    X, dY = inp.X.cuda(), inp.dY.cuda()
    W1 = [w.cuda() for w in inp.W1_i]
    W2 = [w.cuda() for w in inp.W2_i]
    W3 = [w.cuda() for w in inp.W3_i]
    ref = None
    for step in range(60):
        Y, saved, H = mlp.forward(X, W1, W2, W3)
        g = mlp.backward(X, W1, W2, saved, H, dY, W3)
        got = [Y, g["dX"], *g["dW1"], *g["dW2"], *g["dW3"]]
        if ref is None:
            torch.cuda.synchronize()
            ref = [x.clone() for x in got]
            continue
        for i, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(a, b), f"step {step}: output {i} differs"
    torch.cuda.synchronize()
    mlp.check()


@pytest.mark.parametrize("name", ["C2t4", "C4"])
def test_workload_sampled_parity_stream_k_always(gpu_lib, name):
    """The stream-K tail on every launch of the workload (C4: SwiGLU with
    merged N = 256 MMAs; C2: tiles split across many pairs)."""
    _sampled_compare(gpu_lib, si.WORKLOADS[name], stream_k=gpu_lib.STREAM_K_ALWAYS)


@pytest.mark.parametrize("name", ["C3", "C4"])
def test_workload_sampled_parity_stream_k_balance(gpu_lib, name):
    """Every launch of a large workload spread evenly over the pairs (auto mode
    spreads only launches whose weight-gradient operands fit in L2, as C2's)."""
    _sampled_compare(gpu_lib, si.WORKLOADS[name], stream_k=gpu_lib.STREAM_K_BALANCE)


def _run_for_invariance(tp, inp, act, d_i):
    g = run_gpu(tp, inp, act, "bf16", d_i=d_i)
    out = {"Y": g["Y"], "dX": g["dX"], "dW1": torch.cat(g["dW1"], 1), "dW2": torch.cat(g["dW2"], 0),
           "H": torch.cat(g["H"], 1), "A": torch.cat(g["saved"], 1), "dA": torch.cat(g["dact"], 1)}
    if act == "swiglu":
        out["dW3"] = torch.cat(g["dW3"], 1)
    return out


# (workload, shard layouts of the same full weights)
INVARIANCE = [
    ("C2t1", [(3072,), (1536,) * 2, (768,) * 4]),
    ("C3", [(1536, 2560, 2048, 2048), (2048,) * 4, (8192,)]),
    ("C4", [(1376,) * 8, (5504,) * 2, (11008,)]),
    ("C5", [(1536,) * 8, (6144,) * 2, (12288,)]),
]


@pytest.mark.parametrize("name,layouts", INVARIANCE, ids=[c[0] for c in INVARIANCE])
def test_shard_count_invariance(gpu_lib, name, layouts):
    """The same full weights cut into different shard layouts (t = 1, 2, 4 or 8,
    equal or unequal widths) give the same outputs, activations and gradients
    within the bf16 bound, compared in full on the device (every element).  For
    SwiGLU the saved pre-activations are [G | U] side by side."""
    w = si.WORKLOADS[name]
    inp = si.make_workload_inputs(w)
    outs = [_run_for_invariance(gpu_lib, inp, w.act, d_i) for d_i in layouts]
    for a in range(len(outs)):
        for b in range(a + 1, len(outs)):
            for k in outs[0]:
                e = dev_rel_err(outs[b][k], outs[a][k])
                assert e <= 2e-2, f"{name}: d_i={layouts[a]} vs d_i={layouts[b]}: {k} differs by {e}"
    del outs
    torch.cuda.empty_cache()


def test_tensors_beyond_2_pow_31_elements(gpu_lib):
    """T = 2^21 + 96 tokens (ragged against the 256-row tiles) with one shard
    of 1536: A, H and dA hold 3.2e9 elements each, so element offsets pass
    2^31 (32-bit index arithmetic anywhere would show up).  Sampled rows include
    those where the offset into A / H / dA crosses 2^31."""
    w = si.Workload("large gelu bf16 T=2^21+96 d=256 t=1x1536", 2 ** 21 + 96, 256, (1536,), "gelu", "bf16")
    cross = (2 ** 31) // 1536
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0], rng.choice(w.T, 12, replace=False)])
    units = np.concatenate([[0, 1535], rng.choice(1536, 8, replace=False)])
    _sampled_compare(gpu_lib, w, extra_rows=(cross - 1, cross, cross + 1, 2 ** 21 + 95), rows=rows, units=units,
                     tile_complete=False)
    torch.cuda.empty_cache()
