"""GPU parity of the attention projections (QKV column-parallel by heads, the
row-parallel output projection with the g-sum, and their backward with the
f-sum) against the fp64 oracle, through the C ABI.

Small and ragged shapes are compared element by element on every output;
the full-size workloads (the Megatron 8.3B attention shape, Llama 3 405B at
t = 8 with grouped-query widths) on sampled token rows (QKV, Z, dO, dX) and
sampled weight columns (dW_QKV, rows of dWO), each computed by the oracle on
the corresponding sub-problem: the projections are row-separable in the
tokens and the weight gradients column-separable, which the oracle's own
pins check.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from gpu_helpers import cat_cols, cat_rows, rel_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def run_attn(tp, a: si.AttnInputs, dtype: str, device="cuda", stream_k=None):
    T, d = a.X.shape
    m = tp.ShardedAttentionProj(T, d, a.dq_i, a.dkv_i, dtype, device=device)
    if stream_k is not None:
        tp.tpmlp_plan_set_stream_k(m.plan, stream_k)
    X = a.X.to(device)
    Wqkv = [w.to(device) for w in a.Wqkv_i]
    O = [o.to(device) for o in a.O_i]
    WO = [w.to(device) for w in a.WO_i]
    dZ = a.dZ.to(device)
    dQKV = [g.to(device) for g in a.dQKV_i]
    out = {"QKV": m.qkv_forward(X, Wqkv)}
    out["Z"] = m.out_forward(WO, O)
    out["dO"], out["dWO"] = m.out_backward(WO, O, dZ)
    out["dX"], out["dWqkv"] = m.qkv_backward(X, Wqkv, dQKV)
    torch.cuda.synchronize()
    m.check()
    out["m"] = m
    return out


def split_qkv(mats, dq_i, dkv_i):
    """Per-shard [q | k | v] column blocks -> full Q, K, V (fp64 numpy)."""
    q = [x[:, :a] for x, a in zip(mats, dq_i)]
    k = [x[:, a:a + b] for x, a, b in zip(mats, dq_i, dkv_i)]
    v = [x[:, a + b:] for x, a, b in zip(mats, dq_i, dkv_i)]
    return cat_cols(q), cat_cols(k), cat_cols(v)


def _full_compare(tp, T, d, dq_i, dkv_i, dtype, seed=1234, stream_k=None):
    a = si.make_attn_inputs(T, d, dq_i, dkv_i, dtype, seed)
    g = run_attn(tp, a, dtype, stream_k=stream_k)
    f = oracle.attn_forward(a.X, a.WQ, a.WK, a.WV, a.O, a.WO)
    b = oracle.attn_backward(a.X, a.WQ, a.WK, a.WV, a.O, a.WO, a.dZ, a.dQ, a.dK, a.dV)
    Q, K, V = split_qkv(g["QKV"], dq_i, dkv_i)
    dWQ, dWK, dWV = split_qkv(g["dWqkv"], dq_i, dkv_i)
    errs = {"Q": rel_err(Q, f["Q"]), "K": rel_err(K, f["K"]), "V": rel_err(V, f["V"]),
            "Z": rel_err(to_np(g["Z"]), f["Z"]), "dO": rel_err(cat_cols(g["dO"]), b["dO"]),
            "dWO": rel_err(cat_rows(g["dWO"]), b["dWO"]), "dX": rel_err(to_np(g["dX"]), b["dX"]),
            "dWQ": rel_err(dWQ, b["dWQ"]), "dWK": rel_err(dWK, b["dWK"]), "dWV": rel_err(dWV, b["dWV"])}
    tol = tol_for(dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"T={T} d={d} dq={dq_i} dkv={dkv_i} {dtype}: over {tol}: {bad} (all: {errs})"
    return g, errs


SMALL = [
    (1000, 384, (256, 128, 64), (64, 32, 64)),  # grouped-query widths, ragged T, unequal shards
    (300, 128, (64, 64), (64, 64)),             # plain multi-head, two shards
    (257, 256, (128,), (16,)),                  # one shard, one narrow key/value head
    (96, 64, (8,) * 16, (8,) * 16),             # the most shards a plan takes
]


@pytest.mark.parametrize("case", SMALL)
def test_attn_small_bf16_all_outputs(gpu_lib, case):
    _full_compare(gpu_lib, *case, "bf16")


@pytest.mark.parametrize("case", SMALL[:3])
def test_attn_small_stream_k_always(gpu_lib, case):
    _full_compare(gpu_lib, *case, "bf16", stream_k=gpu_lib.STREAM_K_ALWAYS)


def test_attn_multi_wave_bf16(gpu_lib):
    """More tiles than resident CTA pairs in every launch, with a ragged tail."""
    _full_compare(gpu_lib, 4100, 1024, (256,) * 4, (64,) * 4, "bf16")


@pytest.mark.parametrize("case", [(130, 64, (32, 16), (8, 16)), (64, 128, (64,), (64,))])
def test_attn_fp32_path(gpu_lib, case):
    _full_compare(gpu_lib, *case, "fp32")


def test_attn_shard_count_invariance(gpu_lib):
    """12 heads of 64 (GPT-2 small's attention) split over t = 1, 2, 4 shards:
    the same full weights give the same outputs within the bf16 bound."""
    outs = {}
    for t in (1, 2, 4):
        dq = (768 // t,) * t
        g, _ = _full_compare(gpu_lib, 2048, 768, dq, dq, "bf16", seed=77)
        outs[t] = {"Z": to_np(g["Z"]), "dX": to_np(g["dX"]), "dWO": cat_rows(g["dWO"]),
                   "QKV": np.concatenate(split_qkv(g["QKV"], dq, dq), 1)}
        del g
        torch.cuda.empty_cache()
    for x, y in ((1, 2), (1, 4), (2, 4)):
        for k in outs[1]:
            e = rel_err(outs[y][k], outs[x][k])
            assert e <= 2e-2, f"t={x} vs t={y}: {k} differs by {e}"


def _sampled_compare(tp, w: si.AttnWorkload, nrows=16, ncols=16, seed=1234):
    a = si.make_attn_workload_inputs(w, seed)
    g = run_attn(tp, a, w.dtype)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, nrows, replace=False)]))
    dq, dkv = sum(w.dq_i), sum(w.dkv_i)
    cq = np.unique(np.concatenate([[0, dq - 1], rng.choice(dq, ncols, replace=False)]))
    ckv = np.unique(np.concatenate([[0, dkv - 1], rng.choice(dkv, ncols, replace=False)]))
    for lo, hi in si.shard_slices(w.dq_i):  # shard boundaries
        cq = np.union1d(cq, [lo, hi - 1])
    for lo, hi in si.shard_slices(w.dkv_i):
        ckv = np.union1d(ckv, [lo, hi - 1])
    r = torch.as_tensor(rows)
    fr = oracle.attn_forward(a.X[r], a.WQ, a.WK, a.WV, a.O[r], a.WO)
    br = oracle.attn_backward(a.X[r], a.WQ, a.WK, a.WV, a.O[r], a.WO, a.dZ[r], a.dQ[r], a.dK[r], a.dV[r])
    q, kv = torch.as_tensor(cq), torch.as_tensor(ckv)
    bc = oracle.attn_backward(a.X, a.WQ[:, q], a.WK[:, kv], a.WV[:, kv], a.O[:, q], a.WO[q], a.dZ, a.dQ[:, q],
                              a.dK[:, kv], a.dV[:, kv])
    Q, K, V = split_qkv([x[r.to(x.device)] for x in g["QKV"]], w.dq_i, w.dkv_i)
    dWQ, dWK, dWV = split_qkv(g["dWqkv"], w.dq_i, w.dkv_i)
    errs = {"Q": rel_err(Q, fr["Q"]), "K": rel_err(K, fr["K"]), "V": rel_err(V, fr["V"]),
            "Z": rel_err(to_np(g["Z"])[rows], fr["Z"]), "dX": rel_err(to_np(g["dX"])[rows], br["dX"]),
            "dO": rel_err(cat_cols(g["dO"])[rows], br["dO"]), "dWQ": rel_err(dWQ[:, cq], bc["dWQ"]),
            "dWK": rel_err(dWK[:, ckv], bc["dWK"]), "dWV": rel_err(dWV[:, ckv], bc["dWV"]),
            "dWO": rel_err(cat_rows(g["dWO"])[cq], bc["dWO"])}
    tol = tol_for(w.dtype)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name}: over tolerance {tol}: {bad} (all: {errs})"
    # properties that hold at any size: finite outputs everywhere
    assert torch.isfinite(g["Z"]).all() and torch.isfinite(g["dX"]).all()
    for k in ("QKV", "dO", "dWO", "dWqkv"):
        assert all(torch.isfinite(x).all() for x in g[k])
    return errs


@pytest.mark.parametrize("name", ["A1", "A2"])
def test_attn_workload_sampled_parity(gpu_lib, name):
    _sampled_compare(gpu_lib, si.ATTN_WORKLOADS[name])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_attn_empty_token_batch(gpu_lib, dtype):
    tp = gpu_lib
    d, dq, dkv = 64, (64, 32), (16, 32)
    m = tp.ShardedAttentionProj(0, d, dq, dkv, dtype)
    td = m.tdtype
    X = torch.empty(0, d, dtype=td, device="cuda")
    Wqkv = [torch.randn(d, q + 2 * k, device="cuda").to(td) for q, k in zip(dq, dkv)]
    WO = [torch.randn(q, d, device="cuda").to(td) for q in dq]
    O = [torch.empty(0, q, dtype=td, device="cuda") for q in dq]
    QKV = m.qkv_forward(X, Wqkv)
    Z = m.out_forward(WO, O)
    dO, dWO = m.out_backward(WO, O, torch.empty(0, d, dtype=td, device="cuda"))
    dWO_pre = [x.fill_(7) for x in dWO]
    dO, dWO = m.out_backward(WO, O, torch.empty(0, d, dtype=td, device="cuda"), out=(dO, dWO_pre))
    dQKV = [torch.empty(0, q + 2 * k, dtype=td, device="cuda") for q, k in zip(dq, dkv)]
    dWqkv = [torch.full((d, q + 2 * k), 7.0, dtype=td, device="cuda") for q, k in zip(dq, dkv)]
    dX, dWqkv = m.qkv_backward(X, Wqkv, dQKV, out=(torch.empty(0, d, dtype=td, device="cuda"), dWqkv))
    torch.cuda.synchronize()
    m.check()
    assert Z.shape == (0, d) and dX.shape == (0, d) and all(q.shape[0] == 0 for q in QKV)
    for x in dWO + dWqkv:
        assert torch.count_nonzero(x) == 0


def test_attn_determinism_and_launch_count(gpu_lib):
    tp = gpu_lib
    a = si.make_attn_inputs(700, 256, (128, 64), (32, 64), "bf16", seed=5)
    g1 = run_attn(tp, a, "bf16")
    assert tp.tpmlp_last_launch_count() == 1  # the QKV backward: one launch
    g2 = run_attn(tp, a, "bf16")
    assert torch.equal(g1["Z"], g2["Z"]) and torch.equal(g1["dX"], g2["dX"])
    for k in ("QKV", "dO", "dWO", "dWqkv"):
        for x, y in zip(g1[k], g2[k]):
            assert torch.equal(x, y)


def test_attn_argument_errors_with_device(gpu_lib):
    tp = gpu_lib
    m = tp.ShardedAttentionProj(64, 64, (64,), (64,), "bf16")
    X = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    QKV = [torch.empty(64, 192, dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(tp.TpmlpError) as e:  # null weight
        tp.tpmlp_attn_qkv_forward(m.plan, X, [0], QKV, m.workspace)
    assert e.value.status == 1
    raw = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    Wqkv = [torch.zeros(64, 192, dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(tp.TpmlpError) as e:  # X not 16-byte aligned
        tp.tpmlp_attn_qkv_forward(m.plan, raw.data_ptr() + 2, Wqkv, QKV, m.workspace)
    assert e.value.status == 3
    mlp = tp.ShardedMLP(64, 64, (64,), "gelu", "bf16")
    with pytest.raises(tp.TpmlpError) as e:  # MLP plan at an attention entry point
        tp.tpmlp_attn_qkv_forward(mlp.plan, X, Wqkv, QKV, mlp.workspace)
    assert e.value.status == 1
