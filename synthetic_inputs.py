"""Seeded synthetic inputs for the t-sharded MLP workloads.

This module holds no arithmetic of the method: it only draws random tensors,
rounds them once to the storage dtype and cuts the full weights into per-shard
slices.  It is the one module that both the oracle-based tests and the CUDA
path's callers (tests, bench) share.

Recipe (the pages' GPT-2 / BERT / Llama-style shapes; no dataset is used):
  * torch.Generator on the CPU, base seed 1234; sub-seeds +0 X, +1 W1, +2 W3,
    +3 W2, +4 dY;
  * X, dY ~ N(0, 1); W1, W3, W2 ~ N(0, 0.02) (standard deviation 0.02), drawn
    in fp32 and rounded once (round-to-nearest-even) to the config dtype;
  * shard i of W1/W3 is the column slice [o_i, o_i + d_i) of the one drawn
    matrix, shard i of W2 the row slice, so the full weights are the same
    for every shard count t.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

BASE_SEED = 1234


@dataclass(frozen=True)
class Workload:
    name: str
    T: int  # tokens = b * s
    d: int  # hidden
    d_i: tuple  # shard widths, sum = d_ff
    act: str  # "gelu" | "swiglu"
    dtype: str  # "bf16" | "fp32"
    b: int = 0
    s: int = 0
    note: str = ""

    @property
    def dff(self) -> int:
        return int(sum(self.d_i))

    @property
    def t(self) -> int:
        return len(self.d_i)


def _eq(dff: int, t: int) -> tuple:
    assert dff % t == 0
    return tuple([dff // t] * t)


# The five workloads of the pages' shapes.
WORKLOADS = {
    "C1": Workload("C1 gelu fp32 b=2 s=16 d=64 dff=256 t=2", 32, 64, _eq(256, 2), "gelu", "fp32", 2, 16),
    "C2t1": Workload("C2 gelu bf16 GPT-2-small b=8 s=1024 d=768 dff=3072 t=1", 8192, 768, _eq(3072, 1), "gelu",
                     "bf16", 8, 1024),
    "C2t2": Workload("C2 gelu bf16 GPT-2-small b=8 s=1024 d=768 dff=3072 t=2", 8192, 768, _eq(3072, 2), "gelu",
                     "bf16", 8, 1024),
    "C2t4": Workload("C2 gelu bf16 GPT-2-small b=8 s=1024 d=768 dff=3072 t=4", 8192, 768, _eq(3072, 4), "gelu",
                     "bf16", 8, 1024),
    "C3": Workload("C3 gelu bf16 b=4 s=2048 d=2048 dff=8192 t=4 unequal [1536,2560,2048,2048]", 8192, 2048,
                   (1536, 2560, 2048, 2048), "gelu", "bf16", 4, 2048),
    "C4": Workload("C4 swiglu bf16 b=4 s=2048 d=4096 dff=11008 t=8x1376", 8192, 4096, _eq(11008, 8), "swiglu",
                   "bf16", 4, 2048),
    "C5": Workload("C5 gelu bf16 b=8 s=2048 d=3072 dff=12288 t=8x1536", 16384, 3072, _eq(12288, 8), "gelu",
                   "bf16", 8, 2048),
}


def torch_dtype(dtype: str):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]


@dataclass
class Inputs:
    """Full (unsharded) tensors on the CPU in the storage dtype, plus shard views."""
    X: torch.Tensor
    W1: torch.Tensor
    W3: Optional[torch.Tensor]
    W2: torch.Tensor
    dY: torch.Tensor
    d_i: tuple
    W1_i: List[torch.Tensor] = field(default_factory=list)
    W3_i: Optional[List[torch.Tensor]] = None
    W2_i: List[torch.Tensor] = field(default_factory=list)


def _randn(shape, seed, std=1.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def shard_slices(d_i):
    off, out = 0, []
    for w in d_i:
        out.append((off, off + int(w)))
        off += int(w)
    return out


def make_inputs(T: int, d: int, d_i, act: str = "gelu", dtype: str = "bf16", seed: int = BASE_SEED,
                x_scale: float = 1.0, w_std: float = 0.02) -> Inputs:
    """Draw X, W1, (W3), W2, dY with the recipe above and cut the shards."""
    td = torch_dtype(dtype)
    dff = int(sum(d_i))
    X = (_randn((T, d), seed + 0) * x_scale).to(td)
    W1 = _randn((d, dff), seed + 1, w_std).to(td)
    W3 = _randn((d, dff), seed + 2, w_std).to(td) if act == "swiglu" else None
    W2 = _randn((dff, d), seed + 3, w_std).to(td)
    dY = _randn((T, d), seed + 4).to(td)
    inp = Inputs(X=X, W1=W1, W3=W3, W2=W2, dY=dY, d_i=tuple(int(v) for v in d_i))
    for lo, hi in shard_slices(d_i):
        inp.W1_i.append(W1[:, lo:hi].contiguous())
        inp.W2_i.append(W2[lo:hi, :].contiguous())
    if W3 is not None:
        inp.W3_i = [W3[:, lo:hi].contiguous() for lo, hi in shard_slices(d_i)]
    return inp


def make_workload_inputs(w: Workload, seed: int = BASE_SEED) -> Inputs:
    return make_inputs(w.T, w.d, w.d_i, w.act, w.dtype, seed)


def small_int_inputs(T: int, d: int, d_i, act: str, seed: int = 7, lo: int = -3, hi: int = 3) -> Inputs:
    """Integer-valued fp64 inputs in [lo, hi] (for exact sharded/unsharded identities)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    dff = int(sum(d_i))

    def ri(*shape):
        return torch.randint(lo, hi + 1, shape, generator=g).to(torch.float64)

    X, W1, W3, W2, dY = ri(T, d), ri(d, dff), ri(d, dff), ri(dff, d), ri(T, d)
    if act != "swiglu":
        W3 = None
    inp = Inputs(X=X, W1=W1, W3=W3, W2=W2, dY=dY, d_i=tuple(int(v) for v in d_i))
    for a, b in shard_slices(d_i):
        inp.W1_i.append(W1[:, a:b].contiguous())
        inp.W2_i.append(W2[a:b, :].contiguous())
    if W3 is not None:
        inp.W3_i = [W3[:, a:b].contiguous() for a, b in shard_slices(d_i)]
    return inp


def make_biases(d: int, d_i, act: str = "gelu", dtype: str = "bf16", seed: int = BASE_SEED, std: float = 0.5):
    """Optional biases: b1 (and b3 for SwiGLU) [d_ff] cut into shards, b2 [d];
    N(0, std), sub-seeds +5 b1, +6 b3, +7 b2, rounded once to the dtype."""
    td = torch_dtype(dtype)
    dff = int(sum(d_i))
    b1 = _randn((dff,), seed + 5, std).to(td)
    b3 = _randn((dff,), seed + 6, std).to(td) if act == "swiglu" else None
    b2 = _randn((d,), seed + 7, std).to(td)
    sl = shard_slices(d_i)
    return {"b1": b1, "b3": b3, "b2": b2, "b1_i": [b1[lo:hi].contiguous() for lo, hi in sl],
            "b3_i": [b3[lo:hi].contiguous() for lo, hi in sl] if b3 is not None else None}


# ---------------------------------------------------------------- attention projections

@dataclass(frozen=True)
class AttnWorkload:
    name: str
    T: int
    d: int
    dq_i: tuple   # per-shard query width (query heads x head size)
    dkv_i: tuple  # per-shard key/value width (key/value heads x head size)
    dtype: str
    b: int = 0
    s: int = 0

    @property
    def t(self) -> int:
        return len(self.dq_i)

    @property
    def n_i(self) -> tuple:
        return tuple(q + 2 * kv for q, kv in zip(self.dq_i, self.dkv_i))


# The pages' attention shapes: the Megatron GPT-2 8.3B row (hidden 3072, 32 heads of size 96, TP = 8: four
# heads per shard) and Llama 3 405B at TP = 8 (hidden 16384; 16 query heads and one key/value head of size
# 128 per shard).
ATTN_WORKLOADS = {
    "A1": AttnWorkload("A1 attn-proj bf16 GPT-2 8.3B b=8 s=2048 d=3072 32 heads x 96 t=8 (4 heads/shard)", 16384,
                       3072, (384,) * 8, (384,) * 8, "bf16", 8, 2048),
    "A2": AttnWorkload("A2 attn-proj bf16 Llama-3-405B b=1 s=8192 d=16384 GQA 128q/8kv x 128 t=8", 8192, 16384,
                       (2048,) * 8, (128,) * 8, "bf16", 1, 8192),
}


@dataclass
class AttnInputs:
    """Full tensors (CPU, storage dtype) and the per-shard layout of the
    library: W_QKV,i = [WQ_i | WK_i | WV_i] (columns), O_i, WO_i (rows) and
    dQKV_i = [dQ_i | dK_i | dV_i]."""
    X: torch.Tensor
    WQ: torch.Tensor
    WK: torch.Tensor
    WV: torch.Tensor
    O: torch.Tensor
    WO: torch.Tensor
    dZ: torch.Tensor
    dQ: torch.Tensor
    dK: torch.Tensor
    dV: torch.Tensor
    dq_i: tuple
    dkv_i: tuple
    Wqkv_i: List[torch.Tensor] = field(default_factory=list)
    O_i: List[torch.Tensor] = field(default_factory=list)
    WO_i: List[torch.Tensor] = field(default_factory=list)
    dQKV_i: List[torch.Tensor] = field(default_factory=list)


def make_attn_inputs(T: int, d: int, dq_i, dkv_i, dtype: str = "bf16", seed: int = BASE_SEED,
                     w_std: float = 0.02) -> AttnInputs:
    """Sub-seeds +20 X, +21 WQ, +22 WK, +23 WV, +24 O, +25 WO, +26 dZ, +27 dQ, +28 dK, +29 dV.
    X, O and the gradients ~ N(0, 1); weights ~ N(0, w_std); rounded once to the dtype.
    O stands in for the attention core's output and dQ, dK, dV for its input
    gradients: the core itself is not part of the projections."""
    td = torch_dtype(dtype)
    dq, dkv = int(sum(dq_i)), int(sum(dkv_i))
    r = lambda shape, k, std=1.0: _randn(shape, seed + k, std).to(td)
    a = AttnInputs(X=r((T, d), 20), WQ=r((d, dq), 21, w_std), WK=r((d, dkv), 22, w_std), WV=r((d, dkv), 23, w_std),
                   O=r((T, dq), 24), WO=r((dq, d), 25, w_std), dZ=r((T, d), 26), dQ=r((T, dq), 27),
                   dK=r((T, dkv), 28), dV=r((T, dkv), 29), dq_i=tuple(int(v) for v in dq_i),
                   dkv_i=tuple(int(v) for v in dkv_i))
    for (q0, q1), (k0, k1) in zip(shard_slices(dq_i), shard_slices(dkv_i)):
        a.Wqkv_i.append(torch.cat([a.WQ[:, q0:q1], a.WK[:, k0:k1], a.WV[:, k0:k1]], 1).contiguous())
        a.O_i.append(a.O[:, q0:q1].contiguous())
        a.WO_i.append(a.WO[q0:q1].contiguous())
        a.dQKV_i.append(torch.cat([a.dQ[:, q0:q1], a.dK[:, k0:k1], a.dV[:, k0:k1]], 1).contiguous())
    return a


def make_attn_workload_inputs(w: AttnWorkload, seed: int = BASE_SEED) -> AttnInputs:
    return make_attn_inputs(w.T, w.d, w.dq_i, w.dkv_i, w.dtype, seed)
