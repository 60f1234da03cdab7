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
