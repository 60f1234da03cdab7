"""Benchmark: forward + backward of the t-sharded Megatron MLP block on GB300.

One step = the whole hot path over one batch: the column-parallel GEMM with
the fused activation, the row-parallel GEMM with the g-sum, the dgrad GEMM
with act' fused (plus dW2), and the dX GEMM with the f-sum (plus dW1 / dW3).
The default workload is the largest GeLU configuration, T = b*s = 16384
tokens, d = 3072, d_ff = 12288 in t = 8 shards of 1536 (the north-star
target names the largest configurations).

Prints one JSON line (rank 0).  Multi-GPU: one process per GPU (torchrun),
each GPU runs its own replica of the workload (the block's shards all live on
one GPU; replicas only, no collective on the data path), barrier + max over
ranks around the timed region, value = total FLOPs of all ranks / time.

--impl reference times the fp64 CPU oracle instead (on the host cores, a
bounded token sample of the same workload): there is no other implementation
of this block to run.

--workload A1 / A2 measures the attention block's projections instead: one
step = the column-parallel QKV projection, the row-parallel output projection
with the g-sum, the output projection's backward (dO, dWO) and the QKV
backward with the f-sum (dX, dW_QKV); the attention core between them is not
part of the library and is not run (its output O and input gradients dQKV are
seeded inputs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = "TP-sharded MLP fwd+bwd TFLOP/s on 1 GB300 (% of dense BF16 peak)"
ATTN_METRIC = "TP-sharded attention projections fwd+bwd TFLOP/s on 1 GB300 (% of dense BF16 peak)"
UNIT = "TFLOP/s"
STREAM_K_MODES = {"off": 0, "auto": 1, "always": 2}
L2_BYTES = 129 * 1000 * 1000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def flops_fwd_bwd(w: si.Workload, T: int | None = None) -> int:
    """Algorithmic FLOPs: 12 T d dff (GeLU), 18 T d dff (SwiGLU); no padding, no recompute."""
    per = 18 if w.act == "swiglu" else 12
    return per * (w.T if T is None else T) * w.d * w.dff


def phase_flops(w: si.Workload) -> dict:
    """Algorithmic FLOPs of each of the four launches of a step."""
    g = 2 * w.T * w.d * w.dff
    if w.act == "swiglu":
        return {"fwd_column": 2 * g, "fwd_row": g, "bwd_dgrad": 2 * g, "bwd_fsum": 4 * g}
    return {"fwd_column": g, "fwd_row": g, "bwd_dgrad": 2 * g, "bwd_fsum": 2 * g}


def attn_phase_flops(w: si.AttnWorkload, T: int | None = None, n_i=None, dq_i=None) -> dict:
    """Algorithmic FLOPs of the four attention-projection launches (N = sum of
    the fused QKV widths, dq = sum of the query widths)."""
    T = w.T if T is None else T
    N = sum(w.n_i if n_i is None else n_i)
    dq = sum(w.dq_i if dq_i is None else dq_i)
    return {"qkv_fwd": 2 * T * w.d * N, "out_fwd": 2 * T * dq * w.d, "out_bwd": 4 * T * dq * w.d,
            "qkv_bwd": 4 * T * w.d * N}


def phase_bytes(w: si.Workload) -> dict:
    """Algorithmic HBM bytes of each launch of a step (bf16 = 2 bytes): every
    input read once and every output written once.  GeLU (SwiGLU adds W3, U,
    dU, dW3): column X, W1 -> A, H; row H, W2 -> Y; dgrad dY, W2, A, H -> dA,
    dW2; f-sum dA, W1, X -> dX, dW1."""
    e = 2 if w.dtype == "bf16" else 4
    T, d, f = w.T, w.d, w.dff
    n = 2 if w.act == "swiglu" else 1  # pre-activations / activation gradients per hidden unit
    return {"fwd_column": e * (T * d + n * d * f + n * T * f + T * f),
            "fwd_row": e * (T * f + f * d + T * d),
            "bwd_dgrad": e * (T * d + f * d + n * T * f + T * f + n * T * f + f * d),
            "bwd_fsum": e * (n * T * f + n * d * f + T * d + T * d + n * d * f)}


def attn_phase_bytes(w: si.AttnWorkload) -> dict:
    """Algorithmic HBM bytes of the four attention-projection launches (bf16),
    every input read and every output written once (N = sum of the fused QKV
    widths, dq = sum of the query widths)."""
    T, d, N, dq = w.T, w.d, sum(w.n_i), sum(w.dq_i)
    return {"qkv_fwd": 2 * (T * d + d * N + T * N), "out_fwd": 2 * (T * dq + dq * d + T * d),
            "out_bwd": 2 * (T * d + dq * d + T * dq + T * dq + dq * d),
            "qkv_bwd": 2 * (T * N + d * N + T * d + T * d + d * N)}


def peak_regime(peaks: dict, peak_src: str, elapsed_ms: float, clocks) -> dict:
    """The bf16 tensor peak the timed region ran in: the burst figure (a kernel
    timed alone, clocks free to boost), unless the region lasted a second or
    more with the power cap active in the clock samples, which is the
    sustained regime the measured sustained figure was taken in."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", [])
    regime = "sustained" if (elapsed_ms >= 1000.0 and capped) else "burst"
    return {"regime": regime, "peak": sus if regime == "sustained" else burst, "burst": burst, "sustained": sus,
            "hbm_gbs": float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), "source": peak_src,
            "why": (f"timed region {elapsed_ms:.0f} ms, power cap "
                    f"{'seen' if capped else 'not seen'} in the clock samples")}


def make_roofline(dom: str, flops: dict, nbytes: dict, per_phase: dict, ms_per_step: float, pk: dict, clocks,
                  traffic):
    """Dominant-launch roofline (TFLOP/s against the regime's bf16 peak), both
    peaks' fractions beside it, and the whole step's: the slower of its FLOPs
    at the tensor peak and its algorithmic bytes at the measured HBM bandwidth,
    against the measured step time."""
    achieved = flops[dom] / (per_phase[dom] / 1e3) / 1e12
    sm = clocks.get("sm_mhz") if clocks else None
    t_tensor = sum(flops.values()) / (pk["peak"] * 1e12) * 1e3
    t_hbm = sum(nbytes.values()) / (pk["hbm_gbs"] * 1e9) * 1e3
    per = {}
    for k, ms in per_phase.items():
        if flops.get(k):
            a = flops[k] / (ms / 1e3) / 1e12
            per[k] = {"ms": ms, "tflops": a, "frac": a / pk["peak"],
                      "gbs_algorithmic": nbytes.get(k, 0) / (ms / 1e3) / 1e9}
    return {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": pk["peak"], "unit": "TFLOP/s",
            "frac": achieved / pk["peak"], "traffic": traffic, "algorithmic_bytes": nbytes.get(dom),
            "regime": pk["regime"], "regime_why": pk["why"], "sm_mhz_median": sm,
            "frac_of_burst": achieved / pk["burst"], "frac_of_sustained": achieved / pk["sustained"],
            "peak_note": f"{pk['source']} bf16 peaks: burst {pk['burst']}, sustained {pk['sustained']} TFLOP/s",
            "step": {"bound": "tensor" if t_tensor >= t_hbm else "hbm", "tensor_ms": t_tensor, "hbm_ms": t_hbm,
                     "measured_ms": ms_per_step, "frac": max(t_tensor, t_hbm) / ms_per_step,
                     "flops": sum(flops.values()), "algorithmic_bytes": sum(nbytes.values())},
            "per_launch": per}


def parity_rows(T: int, seed: int = 11):
    """Token rows for the parity check of the timed results: one in every
    256-row tile band (at the 32-row epilogue-warp slot b mod 8), the first
    and the last row."""
    import numpy as np
    rng = np.random.default_rng(seed)
    rows = {0, T - 1}
    for b in range((T + 255) // 256):
        lo = b * 256 + (b % 8) * 32
        hi = min(lo + 32, T)
        if lo >= T:
            lo, hi = b * 256, T
        rows.add(int(rng.integers(lo, hi)))
    return sorted(rows)


def _rec(ev, i, stream):
    """Record event i of a step's event list, if the list has one there."""
    if ev is not None and ev[i] is not None:
        ev[i].record(stream)


def pick_dominant(step, names, dev, drop=()):
    """Per-launch timing that does not slow the timed steps: three untimed
    steps after the warm-up, with an event between every launch, give each
    phase's duration and pick the longest; the timed steps then carry events
    only around that one (dominant_events).  Returns (phase ms, name, index)."""
    import torch
    pre = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(3)]
    for ev in pre:
        step(ev)
    torch.cuda.synchronize(dev)
    phase = {n: statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in pre) for i, n in enumerate(names)}
    for n in drop:
        phase.pop(n, None)
    dom = max(phase, key=phase.get)
    return phase, dom, names.index(dom)


def dominant_events(steps, nphase, di):
    """Per-step event lists with events only at the dominant launch's two ends."""
    import torch
    out = []
    for _ in range(steps):
        ev = [None] * (nphase + 1)
        ev[di] = torch.cuda.Event(enable_timing=True)
        ev[di + 1] = torch.cuda.Event(enable_timing=True)
        out.append(ev)
    return out


PHASE_NOTE = ("the dominant launch: mean over the timed steps, whose only per-launch events bracket it; "
              "the others: three untimed steps after the warm-up")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ("tc_gemm.cu", "tc_gemm_common.cuh", "ptx.cuh", "act.cuh", "tpmlp_internal.h",
                  "tpmlp_api.cu")


def kernel_sources_sha256() -> str:
    """Hash of the sources that define the tensor-core kernel and its launches."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "megatron_tensor_transformer_column_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/dram_traffic.json when they were taken
    with the current kernel sources on this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    for r in rec.get("records", []):
        if (r.get("kernel") == kernel and r.get("workload") == workload
                and r.get("sources_sha256") == kernel_sources_sha256()):
            return r.get("dram_bytes_per_launch")
    return None


def attn_workload_config(w: si.AttnWorkload, extra=None):
    cfg = {"workload": w.name, "T": w.T, "b": w.b, "s": w.s, "d": w.d, "t": w.t, "dq_i": list(w.dq_i),
           "dkv_i": list(w.dkv_i), "n_i": list(w.n_i),
           "l2": "no flush: every launch reads more than the 129 MB L2"}
    if extra:
        cfg.update(extra)
    return cfg


def workload_config(w: si.Workload, extra=None):
    cfg = {"workload": w.name, "T": w.T, "b": w.b, "s": w.s, "d": w.d, "d_ff": w.dff, "t": w.t,
           "d_i": list(w.d_i), "act": w.act,
           "l2": "no flush: every launch reads more than the 129 MB L2 (inputs of one step ~1.9 GB)"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle leg

class OracleLeg:
    """The fp64 oracle timed on a bounded sample of the workload: the first
    `tokens` tokens and the first `shards` shards (a sub-block of the same
    weights; its FLOPs are 12 (SwiGLU: 18) * tokens * d * sum of those d_i).
    Inputs are converted to fp64 once, outside the timed calls."""

    def __init__(self, w: si.Workload, max_tokens: int, seed: int = si.BASE_SEED):
        import numpy as np
        self.w = w
        inp = si.make_inputs(max_tokens, w.d, w.d_i, w.act, w.dtype, seed)
        f64 = lambda t: None if t is None else np.ascontiguousarray(t.double().numpy())
        self.X, self.dY = f64(inp.X), f64(inp.dY)
        self.W1, self.W2, self.W3 = f64(inp.W1), f64(inp.W2), f64(inp.W3)

    def flops(self, tokens: int, shards: int) -> int:
        per = 18 if self.w.act == "swiglu" else 12
        return per * tokens * self.w.d * sum(self.w.d_i[:shards])

    def step(self, tokens: int, shards: int) -> float:
        import oracle
        n = sum(self.w.d_i[:shards])
        W1, W2 = self.W1[:, :n], self.W2[:n]
        W3 = self.W3[:, :n] if self.W3 is not None else None
        t0 = time.perf_counter()
        oracle.forward(self.X[:tokens], W1, W2, act=self.w.act, W3=W3)
        oracle.backward(self.X[:tokens], W1, W2, self.dY[:tokens], act=self.w.act, W3=W3)
        return time.perf_counter() - t0


class AttnOracleLeg:
    """The fp64 oracle of the attention projections on a bounded sample: the
    first `tokens` tokens with the full weights (all shards).  Inputs are
    converted to fp64 once, outside the timed calls."""

    def __init__(self, w: si.AttnWorkload, max_tokens: int, seed: int = si.BASE_SEED):
        import numpy as np
        import torch
        self.w = w
        a = si.make_attn_inputs(max_tokens, w.d, w.dq_i, w.dkv_i, w.dtype, seed)
        f64 = lambda t: np.ascontiguousarray(t.to(torch.float64).numpy())
        self.X, self.WQ, self.WK, self.WV = f64(a.X), f64(a.WQ), f64(a.WK), f64(a.WV)
        self.O, self.WO, self.dZ = f64(a.O), f64(a.WO), f64(a.dZ)
        self.dQ, self.dK, self.dV = f64(a.dQ), f64(a.dK), f64(a.dV)

    def flops(self, tokens: int, shards: int) -> int:
        return sum(attn_phase_flops(self.w, tokens).values())

    def step(self, tokens: int, shards: int = 0) -> float:
        import oracle
        n = tokens
        t0 = time.perf_counter()
        oracle.attn_forward(self.X[:n], self.WQ, self.WK, self.WV, self.O[:n], self.WO)
        oracle.attn_backward(self.X[:n], self.WQ, self.WK, self.WV, self.O[:n], self.WO, self.dZ[:n], self.dQ[:n],
                             self.dK[:n], self.dV[:n])
        return time.perf_counter() - t0


def oracle_threads() -> int:
    import oracle
    return oracle.num_threads()


def cpu_baseline(w: si.Workload, tokens: int):
    leg = OracleLeg(w, tokens)
    dt = leg.step(tokens, w.t)
    v = leg.flops(tokens, w.t) / dt / 1e12
    return {"value": v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"fp64 oracle forward+backward on the first {tokens} of {w.T} tokens with all {w.t} shards "
                      f"(full weights), one call of {dt:.1f} s; TFLOP/s = algorithmic FLOPs of that sample / time"}


def check_timed_results(w: si.Workload, got: dict, tol: float = 2e-2):
    """Part of the CPU leg: the last timed step's Y and dX on tile-complete
    sampled rows, and its dW1 / dW2 on one hidden unit per shard, against the
    fp64 oracle (each row or unit from its own definition).  Errors are
    max|err| / max|ref| over the sample, passed at the bf16 bound."""
    import numpy as np
    import oracle
    inp = si.make_workload_inputs(w)
    t0 = time.perf_counter()
    Yr, dXr = oracle.rows(inp.X, inp.W1, inp.W2, inp.dY, got["rows"], act=w.act, W3=inp.W3)
    c1, _, c2 = oracle.wgrad_units(inp.X, inp.W1, inp.W2, inp.dY, got["units"], act=w.act, W3=inp.W3)
    dt = time.perf_counter() - t0

    def rel(a, b):
        b = np.asarray(b, dtype=np.float64)
        return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - b)) / max(np.max(np.abs(b)), 1e-300))

    errs = {"Y": rel(got["Y"], Yr), "dX": rel(got["dX"], dXr), "dW1": rel(got["dW1"], c1), "dW2": rel(got["dW2"], c2)}
    return {"max_err_over_max_ref": errs, "tol": tol, "pass": all(v <= tol for v in errs.values()),
            "sample": f"last timed step: Y, dX on {len(got['rows'])} token rows (one in every 256-row tile band), "
                      f"dW1 columns / dW2 rows of {len(got['units'])} hidden units (one per shard); "
                      f"oracle {dt:.1f} s"}


def attn_cpu_baseline(w: si.AttnWorkload, tokens: int):
    leg = AttnOracleLeg(w, tokens)
    dt = leg.step(tokens)
    v = leg.flops(tokens, w.t) / dt / 1e12
    return {"value": v, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"fp64 oracle attention projections forward+backward on the first {tokens} of {w.T} tokens "
                      f"(full weights, all {w.t} shards), one call of {dt:.1f} s; TFLOP/s = algorithmic FLOPs of "
                      f"that sample / time"}


def run_reference_attn(args, w: si.AttnWorkload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    leg = AttnOracleLeg(w, 64)
    budget = 150.0 / (args.steps + args.warmup)
    t1 = leg.step(1)
    t8 = leg.step(8)
    per_tok = max(1e-9, (t8 - t1) / 7)
    tokens = 1
    for tk in (64, 32, 16, 8, 4, 2, 1):
        if t1 + (tk - 1) * per_tok <= budget:
            tokens = tk
            break
    for _ in range(args.warmup):
        leg.step(tokens)
    times = [leg.step(tokens) for _ in range(args.steps)]
    total = sum(times)
    value = leg.flops(tokens, w.t) * len(times) / total / 1e12
    sample = (f"per step: fp64 oracle attention projections forward+backward on the first {tokens} of {w.T} "
              f"tokens (full weights); TFLOP/s = algorithmic FLOPs of the sample / time")
    line = {"impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) X/O/gradients, N(0,0.02) W)", "config": attn_workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, w: si.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    leg = OracleLeg(w, 64)
    # size the per-step sample so the whole run stays within ~150 s
    budget = 150.0 / (args.steps + args.warmup)
    t11 = leg.step(1, 1)
    t81 = leg.step(8, 1)
    per_tok = max(0.0, (t81 - t11) / 7)
    shards, tokens = 1, 1
    for sh in range(w.t, 0, -1):
        if sh * t11 <= budget:
            shards = sh
            break
    for tk in (64, 32, 16, 8, 4, 2, 1):
        if shards * (t11 + (tk - 1) * per_tok) <= budget:
            tokens = tk
            break
    for _ in range(args.warmup):
        leg.step(tokens, shards)
    times = [leg.step(tokens, shards) for _ in range(args.steps)]
    total = sum(times)
    value = leg.flops(tokens, shards) * len(times) / total / 1e12
    sample = (f"per step: fp64 oracle forward+backward on the first {tokens} of {w.T} tokens and the first "
              f"{shards} of {w.t} shards (d_ff slice {sum(w.d_i[:shards])}); TFLOP/s = algorithmic FLOPs of the "
              f"sample / time")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) X/dY, N(0,0.02) W)", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg

def run_ours(args, w: si.Workload):
    import torch
    import megatron_tensor_transformer_column_gb300 as tp

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tp.load()

    inp = si.make_workload_inputs(w)
    td = si.torch_dtype(w.dtype)
    mlp = tp.ShardedMLP(w.T, w.d, w.d_i, w.act, w.dtype, device=dev)
    tp.tpmlp_plan_set_stream_k(mlp.plan, STREAM_K_MODES[args.stream_k])
    sw = w.act == "swiglu"
    X = inp.X.to(dev)
    dY = inp.dY.to(dev)
    W1 = [x.to(dev) for x in inp.W1_i]
    W2 = [x.to(dev) for x in inp.W2_i]
    W3 = [x.to(dev) for x in inp.W3_i] if sw else None
    Y, saved, H = mlp.alloc_forward()
    dact, dX, dW1, dW3, dW2 = mlp.alloc_backward()
    stream = torch.cuda.current_stream(dev)
    plan, wsp = mlp.plan, mlp.workspace
    b1 = b3 = b2 = db1 = db3 = db2 = None
    if args.bias:  # b1 (b3) before the activation, b2 after the g-sum, and their gradients
        bias = si.make_biases(w.d, w.d_i, w.act, w.dtype)
        b1 = [x.to(dev) for x in bias["b1_i"]]
        b3 = [x.to(dev) for x in bias["b3_i"]] if sw else None
        b2 = bias["b2"].to(dev)
        db1, db3, db2 = mlp.alloc_bias_grads()

    def step(ev=None):
        if args.recompute:  # backward with H recomputed from the pre-activations (H treated as scratch)
            _rec(ev, 0, stream)
            tp.tpmlp_forward_column(plan, X, W1, W3, b1, b3, saved, H, wsp, stream)
            _rec(ev, 1, stream)
            tp.tpmlp_forward_row(plan, W2, b2, H, Y, wsp, stream)
            _rec(ev, 2, stream)
            _rec(ev, 3, stream)
            tp.tpmlp_backward_recompute(plan, X, W1, W3, W2, saved, H, dY, dact, dX, dW1, dW3, dW2, db1, db3, db2,
                                        wsp, stream)
            _rec(ev, 4, stream)
            return
        _rec(ev, 0, stream)
        tp.tpmlp_forward_column(plan, X, W1, W3, b1, b3, saved, H, wsp, stream)
        _rec(ev, 1, stream)
        tp.tpmlp_forward_row(plan, W2, b2, H, Y, wsp, stream)
        _rec(ev, 2, stream)
        tp.tpmlp_backward_dgrad(plan, W2, saved, H, dY, dact, dW2, db2, wsp, stream)
        _rec(ev, 3, stream)
        tp.tpmlp_backward_fsum(plan, X, W1, W3, dact, dX, dW1, dW3, db1, db3, wsp, stream)
        _rec(ev, 4, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    mlp.check(stream)

    names = ["fwd_column", "fwd_row", "bwd_dgrad", "bwd_fsum"]
    if args.recompute:
        names = ["fwd_column", "fwd_row", "bwd_none", "bwd_recompute"]
    per_phase, dom, di = pick_dominant(step, names, dev, drop=("bwd_none",))

    # ---- timed region: K steps, CUDA events on the launching stream
    evs = dominant_events(args.steps, len(names), di)
    barrier(ws)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    barrier(ws)
    mlp.check(stream)
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    ms_per_step = elapsed_ms / args.steps
    per_phase[dom] = statistics.mean(ev[di].elapsed_time(ev[di + 1]) for ev in evs)
    total_flops = flops_fwd_bwd(w) * ws
    value = total_flops * args.steps / (elapsed_ms / 1e3) / 1e12

    # ---- the last timed step's results on sampled rows / units, for the
    # parity check of the CPU leg (copied out before anything else runs)
    rows = parity_rows(w.T)
    units = [lo + (hi - lo) // 3 for lo, hi in si.shard_slices(w.d_i)]
    ridx = torch.as_tensor(rows, device=dev)
    offs = [lo for lo, _ in si.shard_slices(w.d_i)]
    shard_of = lambda u: max(i for i, o in enumerate(offs) if o <= u)
    timed = {"rows": rows, "units": units,
             "Y": Y.index_select(0, ridx).double().cpu().numpy(),
             "dX": dX.index_select(0, ridx).double().cpu().numpy(),
             "dW1": torch.stack([dW1[shard_of(u)][:, u - offs[shard_of(u)]] for u in units]).double().cpu().numpy(),
             "dW2": torch.stack([dW2[shard_of(u)][u - offs[shard_of(u)], :] for u in units]).double().cpu().numpy()}

    # ---- end to end through the public API, host buffers (pinned), copies timed
    e2e = run_e2e(args, w, tp, mlp, inp, dev, stream, ws)

    peaks, peak_src = load_peaks()
    pk = peak_regime(peaks, peak_src, elapsed_ms, clocks)
    pf = phase_flops(w)
    pb = phase_bytes(w)
    if args.recompute:
        pf = {"fwd_column": pf["fwd_column"], "fwd_row": pf["fwd_row"], "bwd_none": 0,
              "bwd_recompute": pf["bwd_dgrad"] + pf["bwd_fsum"]}
        pb = {"fwd_column": pb["fwd_column"], "fwd_row": pb["fwd_row"], "bwd_none": 0,
              "bwd_recompute": pb["bwd_dgrad"] + pb["bwd_fsum"]}
    roofline = make_roofline(dom, pf, pb, per_phase, ms_per_step, pk, clocks,
                             None if (args.bias or args.recompute) else measured_traffic(dom, w.name))
    peak_sus, peak_burst = pk["sustained"], pk["burst"]
    if rank != 0:
        return 0
    cpu = None
    parity = None
    if ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.oracle_tokens)
        if not args.bias:
            parity = check_timed_results(w, timed)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) X/dY, N(0,0.02) W, rounded once to bf16)",
        "config": workload_config(w, {"parallelism": f"replicas x{ws} (t={w.t} shards on each GPU)", "stream_k": args.stream_k,
                                      **({"bias": "b1/b3 before the activation, b2 after the g-sum, with db"}
                                         if args.bias else {}),
                                      **({"recompute": "backward recomputes H from the saved pre-activations"}
                                         if args.recompute else {})}),
        "pct_of_peak": {"sustained": value / ws / peak_sus, "burst": value / ws / peak_burst, "source": peak_src},
        "tokens_per_s": w.T * ws * args.steps / (elapsed_ms / 1e3),
        "phase_ms": per_phase,
        "phase_ms_note": PHASE_NOTE,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": (6 if args.bias else 4) * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


class E2EPipeline:
    """End-to-end steps through the public API with host buffers.

    Every step copies its activations in from pinned host memory (H2D) and its
    results back (D2H); the model's weights stay resident on the device (they
    are state, not per-step input, and their gradients are consumed by the
    optimizer on the device).  The copies run on two more streams (uploads,
    downloads: one copy engine each) into double buffers: the inputs of step
    k+1 upload and the results of step k-1 download while step k computes, as
    a training loop's data loader would.  All of it is inside the timed region
    (CUDA events on the compute stream, which waits for the last downloads at
    the end)."""

    def __init__(self, dev, stream, host_in, host_out_like):
        import torch
        self.torch = torch
        self.stream = stream
        self.copy = torch.cuda.Stream(dev)  # uploads
        self.down = torch.cuda.Stream(dev)  # downloads
        self.h_in = [x.contiguous().pin_memory() for x in host_in]
        self.d_in = [[torch.empty_like(x, device=dev) for x in self.h_in] for _ in range(2)]
        self.h_out = [torch.empty_like(o, device="cpu").pin_memory() for o in host_out_like]
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.out_ready = [torch.cuda.Event() for _ in range(2)]
        self.in_free = [torch.cuda.Event() for _ in range(2)]
        self.out_free = [torch.cuda.Event() for _ in range(2)]
        self.h2d = sum(x.numel() * x.element_size() for x in self.h_in)
        self.d2h = sum(x.numel() * x.element_size() for x in self.h_out)

    def upload(self, slot):
        with self.torch.cuda.stream(self.copy):
            self.copy.wait_event(self.in_free[slot])
            for d_, h_ in zip(self.d_in[slot], self.h_in):
                d_.copy_(h_, non_blocking=True)
            self.in_ready[slot].record(self.copy)

    def run(self, n, compute):
        """compute(inputs, slot) enqueues one step on the compute stream and
        returns its device results."""
        for e in self.in_free + self.out_free:
            e.record(self.stream)
        self.upload(0)
        for k in range(n):
            slot = k & 1
            if k + 1 < n:
                self.upload(slot ^ 1)
            self.stream.wait_event(self.in_ready[slot])
            self.stream.wait_event(self.out_free[slot])  # step k-2's results in this slot are read back
            outs = compute(self.d_in[slot], slot)
            self.in_free[slot].record(self.stream)
            self.out_ready[slot].record(self.stream)
            with self.torch.cuda.stream(self.down):
                self.down.wait_event(self.out_ready[slot])
                for h_, d_ in zip(self.h_out, outs):
                    h_.copy_(d_, non_blocking=True)
                self.out_free[slot].record(self.down)
        done = self.torch.cuda.Event()
        done.record(self.down)
        self.stream.wait_event(done)


def run_e2e(args, w, tp, mlp, inp, dev, stream, ws):
    """Same metric through tpmlp_forward / tpmlp_backward with X and dY copied in
    from pinned host memory and Y and dX read back every step (E2EPipeline)."""
    import torch
    sw = w.act == "swiglu"
    W1 = [x.to(dev) for x in inp.W1_i]
    W2 = [x.to(dev) for x in inp.W2_i]
    W3 = [x.to(dev) for x in inp.W3_i] if sw else None
    bufs = [(mlp.alloc_forward(), mlp.alloc_backward()) for _ in range(2)]
    pipe = E2EPipeline(dev, stream, [inp.X, inp.dY], [bufs[0][0][0], bufs[0][1][1]])

    def compute(d_in, slot):
        X, dY = d_in
        (Y, saved, H), (dact, dX, dW1, dW3, dW2) = bufs[slot]
        tp.tpmlp_forward(mlp.plan, X, W1, W3, W2, None, None, None, Y, saved, H, mlp.workspace, stream)
        tp.tpmlp_backward(mlp.plan, X, W1, W3, W2, saved, H, dY, dact, dX, dW1, dW3, dW2, None, None, None,
                          mlp.workspace, stream)
        return [Y, dX]

    pipe.run(2, compute)
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 20))
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.run(n, compute)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    mlp.check(stream)
    return {"value": flops_fwd_bwd(w) * ws * n / (ms / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": pipe.h2d,
            "d2h_bytes_per_step": pipe.d2h, "steps": n, "ms_per_step": ms / n,
            "api": "tpmlp_forward + tpmlp_backward; X and dY uploaded from pinned host memory and Y, dX read back "
                   "every step on copy streams overlapped with the previous/next step; weights resident"}


def run_ours_attn(args, w: si.AttnWorkload):
    import torch
    import megatron_tensor_transformer_column_gb300 as tp

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tp.load()

    a = si.make_attn_workload_inputs(w)
    m = tp.ShardedAttentionProj(w.T, w.d, w.dq_i, w.dkv_i, w.dtype, device=dev)
    tp.tpmlp_plan_set_stream_k(m.plan, STREAM_K_MODES[args.stream_k])
    X, dZ = a.X.to(dev), a.dZ.to(dev)
    Wqkv = [x.to(dev) for x in a.Wqkv_i]
    O = [x.to(dev) for x in a.O_i]
    WO = [x.to(dev) for x in a.WO_i]
    dQKV = [x.to(dev) for x in a.dQKV_i]
    QKV = [torch.empty(w.T, n, dtype=X.dtype, device=dev) for n in w.n_i]
    Z = torch.empty(w.T, w.d, dtype=X.dtype, device=dev)
    dO = [torch.empty(w.T, q, dtype=X.dtype, device=dev) for q in w.dq_i]
    dWO = [torch.empty(q, w.d, dtype=X.dtype, device=dev) for q in w.dq_i]
    dX = torch.empty(w.T, w.d, dtype=X.dtype, device=dev)
    dWqkv = [torch.empty(w.d, n, dtype=X.dtype, device=dev) for n in w.n_i]
    stream = torch.cuda.current_stream(dev)
    plan, wsp = m.plan, m.workspace

    def step(ev=None):
        calls = (lambda: tp.tpmlp_attn_qkv_forward(plan, X, Wqkv, QKV, wsp, stream),
                 lambda: tp.tpmlp_attn_out_forward(plan, WO, O, Z, wsp, stream),
                 lambda: tp.tpmlp_attn_out_backward(plan, WO, O, dZ, dO, dWO, wsp, stream),
                 lambda: tp.tpmlp_attn_qkv_backward(plan, X, Wqkv, dQKV, dX, dWqkv, wsp, stream))
        for i, c in enumerate(calls):
            _rec(ev, i, stream)
            c()
        _rec(ev, 4, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    m.check(stream)
    names = ["qkv_fwd", "out_fwd", "out_bwd", "qkv_bwd"]
    per_phase, dom, di = pick_dominant(step, names, dev)
    evs = dominant_events(args.steps, len(names), di)
    barrier(ws)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    barrier(ws)
    m.check(stream)
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), ws, dev)
    per_phase[dom] = statistics.mean(ev[di].elapsed_time(ev[di + 1]) for ev in evs)
    pf = attn_phase_flops(w)
    step_flops = sum(pf.values())
    value = step_flops * ws * args.steps / (elapsed_ms / 1e3) / 1e12

    # ---- end to end: the per-step activations (X, the attention core's O, dZ
    # and dQKV) uploaded and the results (QKV, Z, dO, dX) read back every step,
    # overlapped with compute; weights and their gradients stay on the device
    outs2 = [([torch.empty_like(x) for x in QKV], torch.empty_like(Z), [torch.empty_like(x) for x in dO],
              torch.empty_like(dX)) for _ in range(2)]
    pipe = E2EPipeline(dev, stream, [a.X, a.dZ, *a.O_i, *a.dQKV_i], [*QKV, Z, *dO, dX])
    nsh = w.t

    def compute(d_in, slot):
        Xs, dZs = d_in[0], d_in[1]
        Os, dQKVs = d_in[2:2 + nsh], d_in[2 + nsh:]
        QKVs, Zs, dOs, dXs = outs2[slot]
        tp.tpmlp_attn_qkv_forward(plan, Xs, Wqkv, QKVs, wsp, stream)
        tp.tpmlp_attn_out_forward(plan, WO, Os, Zs, wsp, stream)
        tp.tpmlp_attn_out_backward(plan, WO, Os, dZs, dOs, dWO, wsp, stream)
        tp.tpmlp_attn_qkv_backward(plan, Xs, Wqkv, dQKVs, dXs, dWqkv, wsp, stream)
        return [*QKVs, Zs, *dOs, dXs]

    pipe.run(2, compute)
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 20))
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.run(n, compute)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    m.check(stream)
    e2e = {"value": step_flops * ws * n / (ms / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": pipe.h2d,
           "d2h_bytes_per_step": pipe.d2h, "steps": n, "ms_per_step": ms / n,
           "api": "tpmlp_attn_* (four calls); X, O, dZ, dQKV uploaded from pinned host memory and QKV, Z, dO, dX "
                  "read back every step on copy streams overlapped with compute; weights resident"}

    peaks, peak_src = load_peaks()
    pk = peak_regime(peaks, peak_src, elapsed_ms, clocks)
    roofline = make_roofline(dom, pf, attn_phase_bytes(w), per_phase, elapsed_ms / args.steps, pk, clocks,
                             measured_traffic(dom, w.name))
    peak_sus, peak_burst = pk["sustained"], pk["burst"]
    if rank != 0:
        return 0
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        cpu = attn_cpu_baseline(w, args.oracle_tokens)
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) X/O/dZ/dQKV, N(0,0.02) W, rounded once to bf16)",
        "config": attn_workload_config(w, {"parallelism": f"replicas x{ws} (t={w.t} shards on each GPU)", "stream_k": args.stream_k}),
        "pct_of_peak": {"sustained": value / ws / peak_sus, "burst": value / ws / peak_burst, "source": peak_src},
        "tokens_per_s": w.T * ws * args.steps / (elapsed_ms / 1e3),
        "phase_ms": per_phase, "phase_ms_note": PHASE_NOTE, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 4 * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_ours_sp(args, w: si.Workload):
    """The same step in the sequence-parallel layout: X and dY read from t token
    stripes, Y and dX written as stripes (tpmlp_forward_sp / tpmlp_backward_sp)."""
    import torch
    import megatron_tensor_transformer_column_gb300 as tp

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tp.load()
    if w.T % w.t or (w.T // w.t) % 128:
        raise SystemExit(f"{w.name}: T/t must be a multiple of 128 tokens for the stripe layout")
    rows = [w.T // w.t] * w.t
    inp = si.make_workload_inputs(w)
    sw = w.act == "swiglu"
    mlp = tp.ShardedMLP(w.T, w.d, w.d_i, w.act, w.dtype, device=dev)
    tp.tpmlp_plan_set_stream_k(mlp.plan, STREAM_K_MODES[args.stream_k])
    mlp.set_sequence_stripes(rows)
    X_j = [x.contiguous().to(dev) for x in inp.X.split(rows)]
    dY_j = [x.contiguous().to(dev) for x in inp.dY.split(rows)]
    W1 = [x.to(dev) for x in inp.W1_i]
    W2 = [x.to(dev) for x in inp.W2_i]
    W3 = [x.to(dev) for x in inp.W3_i] if sw else None
    Y_j = mlp.alloc_stripes()
    dX_j = mlp.alloc_stripes()
    _, saved, H = mlp.alloc_forward()
    dact, _, dW1, dW3, dW2 = mlp.alloc_backward()
    stream = torch.cuda.current_stream(dev)
    plan, wsp = mlp.plan, mlp.workspace

    def step(ev=None):
        _rec(ev, 0, stream)
        tp.tpmlp_forward_sp(plan, X_j, W1, W3, W2, None, None, None, Y_j, saved, H, wsp, stream)
        _rec(ev, 1, stream)
        tp.tpmlp_backward_sp(plan, X_j, W1, W3, W2, saved, H, dY_j, dact, dX_j, dW1, dW3, dW2, None, None, None, wsp,
                             stream)
        _rec(ev, 2, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    mlp.check(stream)
    names = ["forward_sp", "backward_sp"]
    per_phase, dom, di = pick_dominant(step, names, dev)
    evs = dominant_events(args.steps, len(names), di)
    barrier(ws)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    barrier(ws)
    mlp.check(stream)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
    per_phase[dom] = statistics.mean(ev[di].elapsed_time(ev[di + 1]) for ev in evs)
    pf = phase_flops(w)
    pflops = {"forward_sp": pf["fwd_column"] + pf["fwd_row"], "backward_sp": pf["bwd_dgrad"] + pf["bwd_fsum"]}
    value = flops_fwd_bwd(w) * ws * args.steps / (elapsed_ms / 1e3) / 1e12

    # end to end: the X and dY stripes uploaded and the Y and dX stripes read
    # back every step, overlapped with compute; weights stay on the device
    outs2 = [(mlp.alloc_stripes(), mlp.alloc_stripes()) for _ in range(2)]
    pipe = E2EPipeline(dev, stream, [*inp.X.split(rows), *inp.dY.split(rows)], [*Y_j, *dX_j])
    ns = len(rows)

    def compute(d_in, slot):
        Xs, dYs = d_in[:ns], d_in[ns:]
        Ys, dXs = outs2[slot]
        tp.tpmlp_forward_sp(plan, Xs, W1, W3, W2, None, None, None, Ys, saved, H, wsp, stream)
        tp.tpmlp_backward_sp(plan, Xs, W1, W3, W2, saved, H, dYs, dact, dXs, dW1, dW3, dW2, None, None, None, wsp,
                             stream)
        return [*Ys, *dXs]

    pipe.run(2, compute)
    torch.cuda.synchronize(dev)
    n = max(3, min(args.steps, 20))
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.run(n, compute)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    mlp.check(stream)
    e2e = {"value": flops_fwd_bwd(w) * ws * n / (ms / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": pipe.h2d,
           "d2h_bytes_per_step": pipe.d2h, "steps": n, "ms_per_step": ms / n,
           "api": "tpmlp_forward_sp + tpmlp_backward_sp; X and dY stripes uploaded from pinned host memory and Y, "
                  "dX stripes read back every step on copy streams overlapped with compute; weights resident"}
    peaks, peak_src = load_peaks()
    pk = peak_regime(peaks, peak_src, elapsed_ms, clocks)
    pb = phase_bytes(w)
    pbytes = {"forward_sp": pb["fwd_column"] + pb["fwd_row"], "backward_sp": pb["bwd_dgrad"] + pb["bwd_fsum"]}
    roofline = make_roofline(dom, pflops, pbytes, per_phase, elapsed_ms / args.steps, pk, clocks, None)
    roofline["kernel"] = dom + " (two launches: dgrad + f-sum, or column + row)"
    peak_sus, peak_burst = pk["sustained"], pk["burst"]
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) X/dY, N(0,0.02) W, rounded once to bf16)",
        "config": workload_config(w, {"parallelism": f"replicas x{ws} (t={w.t} shards on each GPU)", "stream_k": args.stream_k,
                                      "layout": f"sequence-parallel: {w.t} token stripes of {rows[0]}"}),
        "pct_of_peak": {"sustained": value / ws / peak_sus, "burst": value / ws / peak_burst, "source": peak_src},
        "tokens_per_s": w.T * ws * args.steps / (elapsed_ms / 1e3),
        "phase_ms": per_phase, "phase_ms_note": PHASE_NOTE, "roofline": roofline, "cpu_baseline": None, "e2e": e2e,
        "gpu_launches": 4 * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="C5", choices=sorted(si.WORKLOADS) + sorted(si.ATTN_WORKLOADS))
    ap.add_argument("--oracle-tokens", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bias", action="store_true", help="include the optional biases and their gradients")
    ap.add_argument("--recompute", action="store_true", help="backward recomputes H instead of reading it")
    ap.add_argument("--stream-k", choices=sorted(STREAM_K_MODES), default="auto",
                    help="stream-K tail of the launches (auto: where it shortens the busiest pair's work)")
    ap.add_argument("--sp", action="store_true",
                    help="sequence-parallel layout: X, dY in and Y, dX out as t token stripes of T/t tokens")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.workload in si.ATTN_WORKLOADS:
        w = si.ATTN_WORKLOADS[args.workload]
        return run_reference_attn(args, w) if args.impl == "reference" else run_ours_attn(args, w)
    w = si.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.sp:
        return run_ours_sp(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
