"""Host logic of the benchmark, on CPU: algorithmic FLOP and byte counts, the
choice of the peak the roofline divides by, the step roofline, the parity
rows and the parity check of the timed results (against the oracle)."""
import numpy as np
import pytest

import bench
import oracle
import synthetic_inputs as si


def test_phase_bytes_hand_count_C5():
    w = si.WORKLOADS["C5"]
    T, d, f = 16384, 3072, 12288
    b = bench.phase_bytes(w)
    assert b["fwd_column"] == 2 * (T * d + d * f + 2 * T * f)   # X, W1 -> A, H
    assert b["fwd_row"] == 2 * (T * f + f * d + T * d)          # H, W2 -> Y
    assert b["bwd_dgrad"] == 2 * (T * d + f * d + 3 * T * f + f * d)  # dY, W2, A, H -> dA, dW2
    assert b["bwd_fsum"] == 2 * (T * f + d * f + 2 * T * d + d * f)   # dA, W1, X -> dX, dW1
    assert abs(sum(b.values()) / 1e9 - 3.77) < 0.01


def test_phase_bytes_swiglu_counts_both_projections():
    w = si.WORKLOADS["C4"]
    T, d, f = w.T, w.d, w.dff
    b = bench.phase_bytes(w)
    assert b["fwd_column"] == 2 * (T * d + 2 * d * f + 3 * T * f)  # X, W1, W3 -> G, U, H
    assert b["bwd_fsum"] == 2 * (2 * T * f + 2 * d * f + 2 * T * d + 2 * d * f)
    assert sum(bench.phase_flops(w).values()) == bench.flops_fwd_bwd(w) == 18 * T * d * f


def test_peak_regime():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
    capped = {"sm_mhz": 1600, "reasons": ["sw_power_cap"]}
    free = {"sm_mhz": 2070, "reasons": []}
    assert bench.peak_regime(peaks, "measured", 85.0, capped)["regime"] == "burst"      # short region
    assert bench.peak_regime(peaks, "measured", 5000.0, free)["regime"] == "burst"      # no cap seen
    assert bench.peak_regime(peaks, "measured", 5000.0, None)["regime"] == "burst"      # no samples
    r = bench.peak_regime(peaks, "measured", 5000.0, capped)
    assert r["regime"] == "sustained" and r["peak"] == 1700.0


def test_roofline_fields():
    w = si.WORKLOADS["C5"]
    pf, pb = bench.phase_flops(w), bench.phase_bytes(w)
    per_phase = {"fwd_column": 0.73, "fwd_row": 0.67, "bwd_dgrad": 1.46, "bwd_fsum": 1.31}
    pk = bench.peak_regime({"bf16_tflops": 1899.7, "bf16_tflops_sustained": 1696.5, "hbm_gbs": 6773.9},
                           "measured", 85.0, {"sm_mhz": 2058, "reasons": ["sw_power_cap"]})
    r = bench.make_roofline("bwd_dgrad", pf, pb, per_phase, 4.26, pk, {"sm_mhz": 2058}, None)
    assert r["peak"] == 1899.7 and r["regime"] == "burst"
    assert r["achieved"] == pytest.approx(4 * 16384 * 3072 * 12288 / 1.46e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / 1899.7)
    assert r["frac_of_sustained"] == pytest.approx(r["achieved"] / 1696.5)
    st = r["step"]
    assert st["bound"] == "tensor"
    assert st["tensor_ms"] == pytest.approx(12 * 16384 * 3072 * 12288 / 1899.7e12 * 1e3)
    assert st["frac"] == pytest.approx(st["tensor_ms"] / 4.26)
    assert set(r["per_launch"]) == set(per_phase)


def test_parity_rows_cover_every_band():
    for T in (8192, 16384, 1000, 257):
        rows = np.array(bench.parity_rows(T))
        assert rows.min() == 0 and rows.max() == T - 1
        assert set(rows // 256) == set(range((T + 255) // 256))


def test_timed_result_check_passes_and_catches_a_wrong_row():
    w = si.Workload("tiny", 300, 64, (64, 128), "gelu", "bf16")
    inp = si.make_workload_inputs(w)
    rows = bench.parity_rows(w.T)
    units = [10, 100]
    Yr, dXr = oracle.rows(inp.X, inp.W1, inp.W2, inp.dY, rows)
    c1, _, c2 = oracle.wgrad_units(inp.X, inp.W1, inp.W2, inp.dY, units)
    got = {"rows": rows, "units": units, "Y": Yr.copy(), "dX": dXr.copy(), "dW1": c1.copy(), "dW2": c2.copy()}
    r = bench.check_timed_results(w, got)
    assert r["pass"] and max(r["max_err_over_max_ref"].values()) < 1e-12
    got["dX"][3, 5] += 0.5 * np.abs(dXr).max()
    r = bench.check_timed_results(w, got)
    assert not r["pass"] and r["max_err_over_max_ref"]["dX"] > 0.4
