"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties an oracle function to something the pages or the mathematics
fix: tabulated values of the normal and logistic functions, hand-worked
examples, the split identities the pages state (exact on small integers),
central finite differences, an independent numpy implementation, and, last,
planted mistakes compiled into copies of the oracle that these pins must
catch.
"""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import np_oracle
import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([float(v) for v in line.split()])
    return rows


def _fixture(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if "=" not in line:
            continue
        k, v = (p.strip() for p in line.split("=", 1))
        out[k] = np.array([[float(x) for x in row.split()] for row in v.split(";")])
    return out


# ---------------------------------------------------------------- closed forms

def check_normal_table(o):
    """max relative error of GeLU and GeLU' against the normal-table values."""
    err = 0.0
    for x, P, Z in _table("normal_table.txt"):
        for xs, Ps in ((x, P), (-x, 1.0 - P)):
            g = o.act_value("gelu", xs)
            gp = o.act_grad("gelu", xs)
            err = max(err, abs(g - xs * Ps) / max(1.0, abs(xs * Ps)))
            err = max(err, abs(gp - (Ps + xs * Z)) / max(1.0, abs(Ps + xs * Z)))
    return err


def test_gelu_matches_normal_table():
    assert check_normal_table(oracle.default()) < 2e-15


def test_swish_matches_logistic_table():
    for g, s in _table("logistic_table.txt"):
        assert abs(oracle.act_value("swiglu", g) - g * s) < 2e-15
        assert abs(oracle.act_grad("swiglu", g) - (s + g * s * (1 - s))) < 2e-15


def test_activation_special_values():
    assert oracle.act_value("gelu", 0.0) == 0.0
    assert oracle.act_grad("gelu", 0.0) == 0.5
    assert oracle.act_value("swiglu", 0.0) == 0.0
    assert oracle.act_grad("swiglu", 0.0) == 0.5
    rng = np.random.default_rng(3)
    for x in rng.normal(0, 3, 50):
        # GeLU(x) - GeLU(-x) = x (P(x) + P(-x) = 1); the same holds for Swish.
        assert abs(oracle.act_value("gelu", x) - oracle.act_value("gelu", -x) - x) < 1e-14 * max(1, abs(x))
        assert abs(oracle.act_value("swiglu", x) - oracle.act_value("swiglu", -x) - x) < 1e-14 * max(1, abs(x))
    assert abs(oracle.act_value("gelu", 12.0) - 12.0) < 1e-15 * 12
    assert abs(oracle.act_value("gelu", -12.0)) < 1e-30
    assert oracle.act_value("relu", -2.0) == 0.0 and oracle.act_grad("relu", 3.0) == 1.0


# ---------------------------------------------------------------- worked examples

def test_hand_worked_identity_example_unsharded_and_sharded():
    f = _fixture("tiny_mlp_identity_t2.txt")
    fw = oracle.forward(f["X"], f["W1"], f["W2"], act="identity")
    bw = oracle.backward(f["X"], f["W1"], f["W2"], f["dY"], act="identity")
    assert np.array_equal(fw["Y"], f["Y"])
    assert np.array_equal(bw["dX"], f["dX"])
    assert np.array_equal(bw["dW1"], f["dW1"])
    assert np.array_equal(bw["dW2"], f["dW2"])
    W1_i = [f["W1"][:, 0:2], f["W1"][:, 2:4]]
    W2_i = [f["W2"][0:2], f["W2"][2:4]]
    Y, _ = oracle.forward_sharded(f["X"], W1_i, W2_i, act="identity")
    b = oracle.backward_sharded(f["X"], W1_i, W2_i, f["dY"], act="identity")
    assert np.array_equal(Y, f["Y"])
    assert np.array_equal(b["dX"], f["dX"])
    assert np.array_equal(np.concatenate(b["dW1_i"], 1), f["dW1"])
    assert np.array_equal(np.concatenate(b["dW2_i"], 0), f["dW2"])


def test_hand_worked_gelu_example():
    f = _fixture("tiny_mlp_gelu.txt")
    fw = oracle.forward(f["X"], f["W1"], f["W2"])
    bw = oracle.backward(f["X"], f["W1"], f["W2"], f["dY"])
    for got, want in ((fw["Y"], f["Y"]), (bw["dX"], f["dX"]), (bw["dW1"], f["dW1"]), (bw["dW2"], f["dW2"])):
        np.testing.assert_allclose(got, want, rtol=0, atol=4e-16)


# ---------------------------------------------------------------- split identities

def test_column_identity_is_bitwise():
    """[act(X W1_i)]_i equals act(X W1) bit for bit (same dot products, same order)."""
    rng = np.random.default_rng(11)
    T, d, d_i = 9, 13, [5, 8, 3]
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, sum(d_i))); W2 = rng.normal(size=(sum(d_i), d))
    W3 = rng.normal(size=(d, sum(d_i)))
    for act in ("gelu", "swiglu"):
        full = oracle.forward(X, W1, W2, act=act, W3=W3)
        sl = si.shard_slices(d_i)
        _, H_i = oracle.forward_sharded(X, [W1[:, a:b] for a, b in sl], [W2[a:b] for a, b in sl], act=act,
                                        W3_i=[W3[:, a:b] for a, b in sl] if act == "swiglu" else None)
        assert np.array_equal(np.concatenate(H_i, axis=1), full["H"])


@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("act", ["identity", "relu"])
def test_row_identity_exact_on_small_integers(t, act):
    """Sharded Y, dX, dW equal the unsharded ones exactly (integers below 2^53)."""
    inp = si.small_int_inputs(4, 8, [16 // t] * t, act)
    full_f = oracle.forward(inp.X, inp.W1, inp.W2, act=act)
    full_b = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, act=act)
    Y, _ = oracle.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act=act)
    b = oracle.backward_sharded(inp.X, inp.W1_i, inp.W2_i, inp.dY, act=act)
    assert np.array_equal(Y, full_f["Y"])
    assert np.array_equal(b["dX"], full_b["dX"])
    assert np.array_equal(np.concatenate(b["dW1_i"], 1), full_b["dW1"])
    assert np.array_equal(np.concatenate(b["dW2_i"], 0), full_b["dW2"])
    assert np.all(full_f["Y"] == np.round(full_f["Y"]))  # the integers stayed integers


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("d_i", [[16], [8, 8], [3, 5, 8], [4, 4, 4, 4], [1, 2, 3, 4, 6]])
def test_sharded_equals_unsharded_smooth_acts(act, d_i):
    rng = np.random.default_rng(5)
    T, d = 6, 7
    dff = sum(d_i)
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.3; W2 = rng.normal(size=(dff, d)) * 0.3
    W3 = rng.normal(size=(d, dff)) * 0.3 if act == "swiglu" else None
    dY = rng.normal(size=(T, d))
    sl = si.shard_slices(d_i)
    W1_i = [W1[:, a:b] for a, b in sl]; W2_i = [W2[a:b] for a, b in sl]
    W3_i = [W3[:, a:b] for a, b in sl] if W3 is not None else None
    full_f = oracle.forward(X, W1, W2, act=act, W3=W3)
    full_b = oracle.backward(X, W1, W2, dY, act=act, W3=W3)
    Y, _ = oracle.forward_sharded(X, W1_i, W2_i, act=act, W3_i=W3_i)
    b = oracle.backward_sharded(X, W1_i, W2_i, dY, act=act, W3_i=W3_i)
    np.testing.assert_allclose(Y, full_f["Y"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(b["dX"], full_b["dX"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(np.concatenate(b["dW1_i"], 1), full_b["dW1"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(np.concatenate(b["dW2_i"], 0), full_b["dW2"], rtol=1e-13, atol=1e-13)
    if act == "swiglu":
        np.testing.assert_allclose(np.concatenate(b["dW3_i"], 1), full_b["dW3"], rtol=1e-13, atol=1e-13)


def test_t1_is_the_plain_mlp():
    """t = 1: the sharded form is the textbook Linear-act-Linear block."""
    rng = np.random.default_rng(9)
    X = rng.normal(size=(5, 6)); W1 = rng.normal(size=(6, 10)); W2 = rng.normal(size=(10, 6))
    Y, _ = oracle.forward_sharded(X, [W1], [W2])
    assert np.array_equal(Y, oracle.forward(X, W1, W2)["Y"])


# ---------------------------------------------------------------- finite differences

def fd_check(o, act, seed=1, h=1e-6):
    """max over X, W1, W3, W2 of |analytic - central difference| / max|analytic|,
    for L = <dY, Y> at T=3, d=5, unequal shards d_i=[3,4]."""
    rng = np.random.default_rng(seed)
    T, d, dff = 3, 5, 7
    P = {"X": rng.normal(size=(T, d)), "W1": rng.normal(size=(d, dff)) * 0.5,
         "W2": rng.normal(size=(dff, d)) * 0.5}
    if act == "swiglu":
        P["W3"] = rng.normal(size=(d, dff)) * 0.5
    dY = rng.normal(size=(T, d))

    def loss(p):
        return float(np.sum(dY * o.forward(p["X"], p["W1"], p["W2"], act=act, W3=p.get("W3"))["Y"]))

    g = o.backward(P["X"], P["W1"], P["W2"], dY, act=act, W3=P.get("W3"))
    grads = {"X": g["dX"], "W1": g["dW1"], "W2": g["dW2"], "W3": g["dW3"]}
    worst = 0.0
    for name, val in P.items():
        num = np.zeros_like(val)
        for idx in np.ndindex(val.shape):
            p_plus = {k: v.copy() for k, v in P.items()}; p_plus[name][idx] += h
            p_minus = {k: v.copy() for k, v in P.items()}; p_minus[name][idx] -= h
            num[idx] = (loss(p_plus) - loss(p_minus)) / (2 * h)
        worst = max(worst, float(np.max(np.abs(num - grads[name])) / np.max(np.abs(grads[name]))))
    return worst


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_finite_differences(act):
    assert fd_check(oracle.default(), act) < 1e-7


def test_sharded_backward_finite_differences():
    """The f-sum (backward of the identity f) gives the true input gradient."""
    rng = np.random.default_rng(2)
    X = rng.normal(size=(3, 5)); W1 = rng.normal(size=(5, 7)) * 0.5; W2 = rng.normal(size=(7, 5)) * 0.5
    dY = rng.normal(size=(3, 5))
    sl = si.shard_slices([3, 4])
    W1_i = [W1[:, a:b] for a, b in sl]; W2_i = [W2[a:b] for a, b in sl]
    b = oracle.backward_sharded(X, W1_i, W2_i, dY)
    h = 1e-6
    num = np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        Xp = X.copy(); Xp[idx] += h
        Xm = X.copy(); Xm[idx] -= h
        yp, _ = oracle.forward_sharded(Xp, W1_i, W2_i)
        ym, _ = oracle.forward_sharded(Xm, W1_i, W2_i)
        num[idx] = np.sum(dY * (yp - ym)) / (2 * h)
    assert np.max(np.abs(num - b["dX"])) / np.max(np.abs(b["dX"])) < 1e-7


# ---------------------------------------------------------------- special inputs

def test_zero_inputs():
    rng = np.random.default_rng(4)
    T, d, dff = 4, 6, 8
    W1 = rng.normal(size=(d, dff)); W2 = rng.normal(size=(dff, d)); W3 = rng.normal(size=(d, dff))
    for act in ("gelu", "swiglu"):
        b = oracle.backward(np.zeros((T, d)), W1, W2, rng.normal(size=(T, d)), act=act, W3=W3)
        assert np.all(oracle.forward(np.zeros((T, d)), W1, W2, act=act, W3=W3)["Y"] == 0)
        assert np.all(b["dW2"] == 0) and np.all(b["dW1"] == 0)
        b0 = oracle.backward(rng.normal(size=(T, d)), W1, W2, np.zeros((T, d)), act=act, W3=W3)
        for k in ("dX", "dW1", "dW2"):
            assert np.all(b0[k] == 0)


def test_empty_token_batch():
    rng = np.random.default_rng(4)
    W1 = rng.normal(size=(6, 8)); W2 = rng.normal(size=(8, 6))
    b = oracle.backward(np.zeros((0, 6)), W1, W2, np.zeros((0, 6)))
    assert b["dX"].shape == (0, 6)
    assert np.all(b["dW1"] == 0) and np.all(b["dW2"] == 0)


def test_flop_count_matches_pages():
    """Forward MLP FLOPs with dff = 4h are 16 T h^2, the MLP part of the pages'
    24 h^2 per token (section 3.4 of the network primer); fwd+bwd is 3x."""
    h, T = 3072, 16384
    fwd = 2 * T * h * (4 * h) * 2  # two GEMMs of 2 T h dff
    assert fwd == 16 * T * h * h
    assert 3 * fwd == 12 * T * h * (4 * h)


# ---------------------------------------------------------------- independent cross-check

@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 9), (17, 12, 40), (33, 64, 96)])
def test_c_oracle_matches_numpy_oracle(act, shape):
    T, d, dff = shape
    rng = np.random.default_rng(T * 100 + d)
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.2; W2 = rng.normal(size=(dff, d)) * 0.2
    W3 = rng.normal(size=(d, dff)) * 0.2
    dY = rng.normal(size=(T, d))
    c_f = oracle.forward(X, W1, W2, act=act, W3=W3)
    c_b = oracle.backward(X, W1, W2, dY, act=act, W3=W3)
    n_f = np_oracle.forward(X, W1, W2, act=act, W3=W3)
    n_b = np_oracle.backward(X, W1, W2, dY, act=act, W3=W3)
    for a, b in ((c_f["Y"], n_f["Y"]), (c_f["H"], n_f["H"]), (c_b["dX"], n_b["dX"]), (c_b["dW1"], n_b["dW1"]),
                 (c_b["dW2"], n_b["dW2"]), (c_b["dA"], n_b["dA"])):
        assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))
    if act == "swiglu":
        assert np.max(np.abs(c_b["dW3"] - n_b["dW3"])) <= 1e-12 * max(1.0, np.max(np.abs(n_b["dW3"])))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_sampled_rows_and_units_match_full(act):
    rng = np.random.default_rng(8)
    T, d, dff = 37, 24, 40
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.2; W2 = rng.normal(size=(dff, d)) * 0.2
    W3 = rng.normal(size=(d, dff)) * 0.2 if act == "swiglu" else None
    dY = rng.normal(size=(T, d))
    full_f = np_oracle.forward(X, W1, W2, act=act, W3=W3)
    full_b = np_oracle.backward(X, W1, W2, dY, act=act, W3=W3)
    r = np.array([0, 5, 36, 17])
    Yr, dXr = oracle.rows(X, W1, W2, dY, r, act=act, W3=W3)
    np.testing.assert_allclose(Yr, full_f["Y"][r], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dXr, full_b["dX"][r], rtol=0, atol=1e-12)
    # the same rows with the per-token intermediates, against the independent
    # numpy oracle's full tensors
    Yr2, dXr2, inter = oracle.rows(X, W1, W2, dY, r, act=act, W3=W3, intermediates=True)
    assert np.array_equal(Yr2, Yr) and np.array_equal(dXr2, dXr)
    np.testing.assert_allclose(inter["A"], full_f["A"][r], rtol=0, atol=1e-12)
    np.testing.assert_allclose(inter["H"], full_f["H"][r], rtol=0, atol=1e-12)
    np.testing.assert_allclose(inter["dA"], full_b["dA"][r], rtol=0, atol=1e-12)
    if act == "swiglu":
        np.testing.assert_allclose(inter["U"], full_f["U"][r], rtol=0, atol=1e-12)
        np.testing.assert_allclose(inter["dU"], full_b["dU"][r], rtol=0, atol=1e-12)
    else:
        assert set(inter) == {"A", "H", "dA"}
    u = np.array([0, 39, 13])
    c1, c3, c2 = oracle.wgrad_units(X, W1, W2, dY, u, act=act, W3=W3)
    np.testing.assert_allclose(c1, full_b["dW1"][:, u].T, rtol=0, atol=1e-11)
    np.testing.assert_allclose(c2, full_b["dW2"][u, :], rtol=0, atol=1e-11)
    if act == "swiglu":
        np.testing.assert_allclose(c3, full_b["dW3"][:, u].T, rtol=0, atol=1e-11)


# ---------------------------------------------------------------- planted mistakes

_SRC = os.path.join(os.path.dirname(oracle.__file__), "tpmlp_oracle.c")

# (name, text to find, replacement, pin that must fail)
MUTANTS = [
    ("gelu_grad_drops_x_phi", "return norm_cdf(a) + a * norm_pdf(a);", "return norm_cdf(a);", "fd_gelu"),
    ("tanh_gelu", "static double gelu(double a) { return a * norm_cdf(a); }",
     "static double gelu(double a) { return 0.5 * a * (1.0 + tanh(0.7978845608028654 * (a + 0.044715 * a * a * a))); }",
     "table"),
    ("dW1_uses_dH", "matmul(d, dff, T, X, 1, d, dA, dff, 1, dW1, dff);",
     "matmul(d, dff, T, X, 1, d, dH, dff, 1, dW1, dff);", "fd_gelu"),
    ("dH_untransposed_W2", "matmul(T, dff, d, dY, d, 1, W2, 1, d, dH, dff);",
     "matmul(T, dff, d, dY, d, 1, W2, d, 1, dH, dff);", "fd_gelu"),
    ("swiglu_gate_up_swapped", "dU[i] = dH[i] * swish(A[i]);\n      dA[i] = dH[i] * U[i] * swish_grad(A[i]);",
     "dU[i] = dH[i] * swish(U[i]);\n      dA[i] = dH[i] * U[i] * swish_grad(A[i]);", "fd_swiglu"),
    ("g_sum_drops_partials", "Y[i] += Z[i]; /* g: sum of partial outputs */", "Y[i] = Z[i];", "row_identity"),
    ("f_sum_drops_partials", "dX[i] += dXs[i]; /* f: sum of partial dX */", "dX[i] = dXs[i];", "row_identity"),
    ("swish_grad_sign", "return s + g * s * (1.0 - s);", "return s - g * s * (1.0 - s);", "fd_swiglu"),
    ("rows_dU_uses_swish_grad", "dU_rows[q * dff + j] = dh[j] * swish(a[j]);",
     "dU_rows[q * dff + j] = dh[j] * swish_grad(a[j]);", "rows_intermediates"),
]


def _rows_intermediates_error(o):
    rng = np.random.default_rng(12)
    T, d, dff = 9, 8, 12
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.3; W3 = rng.normal(size=(d, dff)) * 0.3
    W2 = rng.normal(size=(dff, d)) * 0.3; dY = rng.normal(size=(T, d))
    r = np.array([1, 4, 8])
    _, _, inter = o.rows(X, W1, W2, dY, r, act="swiglu", W3=W3, intermediates=True)
    fb = np_oracle.backward(X, W1, W2, dY, act="swiglu", W3=W3)
    return float(np.max(np.abs(inter["dU"] - fb["dU"][r])))


def _row_identity_error(o):
    inp = si.small_int_inputs(4, 8, [4, 4, 8], "relu")
    Y, _ = o.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act="relu")
    b = o.backward_sharded(inp.X, inp.W1_i, inp.W2_i, inp.dY, act="relu")
    ff = o.forward(inp.X, inp.W1, inp.W2, act="relu")
    fb = o.backward(inp.X, inp.W1, inp.W2, inp.dY, act="relu")
    return max(np.max(np.abs(Y - ff["Y"])), np.max(np.abs(b["dX"] - fb["dX"])))


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(mutant, tmp_path):
    name, find, repl, pin = mutant
    src = open(_SRC).read()
    assert src.count(find) == 1, f"mutation site for {name} not found exactly once"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(find, repl))
    lib = oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant.so"))
    o = oracle.load_variant(lib)
    if pin == "fd_gelu":
        assert fd_check(o, "gelu") > 1e-4
    elif pin == "fd_swiglu":
        assert fd_check(o, "swiglu") > 1e-4
    elif pin == "table":
        assert check_normal_table(o) > 1e-6
    elif pin == "row_identity":
        assert _row_identity_error(o) >= 1.0
    elif pin == "rows_intermediates":
        assert _rows_intermediates_error(o) > 1e-3
    # and the unmodified oracle passes the same pin
    clean = oracle.default()
    if pin.startswith("fd"):
        assert fd_check(clean, pin[3:]) < 1e-7
    elif pin == "table":
        assert check_normal_table(clean) < 2e-15
    elif pin == "rows_intermediates":
        assert _rows_intermediates_error(clean) < 1e-12
    else:
        assert _row_identity_error(clean) == 0.0


# ---------------------------------------------------------------- biases (b1 before the activation, b2 after g)

def test_hand_worked_bias_example():
    f = _fixture("tiny_mlp_identity_t2_bias.txt")
    b1, b2 = f["b1"][0], f["b2"][0]
    fw = oracle.forward(f["X"], f["W1"], f["W2"], act="identity", b1=b1, b2=b2)
    bw = oracle.backward(f["X"], f["W1"], f["W2"], f["dY"], act="identity", b1=b1, b2=b2)
    assert np.array_equal(fw["Y"], f["Y"])
    for k in ("dX", "dW1", "dW2"):
        assert np.array_equal(bw[k], f[k]), k
    assert np.array_equal(bw["db1"], f["db1"][0]) and np.array_equal(bw["db2"], f["db2"][0])
    sl = si.shard_slices([2, 2])
    Y, _ = oracle.forward_sharded(f["X"], [f["W1"][:, a:b] for a, b in sl], [f["W2"][a:b] for a, b in sl],
                                  act="identity", b1_i=[b1[a:b] for a, b in sl], b2=b2)
    assert np.array_equal(Y, f["Y"])


def _bias_inputs(rng, d, dff, act, scale=1.0):
    b1 = rng.normal(size=dff) * scale
    b3 = rng.normal(size=dff) * scale if act == "swiglu" else None
    b2 = rng.normal(size=d) * scale
    return b1, b3, b2


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("act", ["identity", "relu"])
def test_bias_sharded_equals_unsharded_exact(t, act):
    """b2 added once after the g-sum: sharded == unsharded exactly on integers."""
    inp = si.small_int_inputs(4, 8, [16 // t] * t, act)
    g = np.random.default_rng(t)
    b1 = g.integers(-3, 4, 16).astype(np.float64)
    b2 = g.integers(-3, 4, 8).astype(np.float64)
    sl = si.shard_slices(inp.d_i)
    b1_i = [b1[a:b] for a, b in sl]
    ff = oracle.forward(inp.X, inp.W1, inp.W2, act=act, b1=b1, b2=b2)
    fb = oracle.backward(inp.X, inp.W1, inp.W2, inp.dY, act=act, b1=b1, b2=b2)
    Y, _ = oracle.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act=act, b1_i=b1_i, b2=b2)
    b = oracle.backward_sharded(inp.X, inp.W1_i, inp.W2_i, inp.dY, act=act, b1_i=b1_i)
    assert np.array_equal(Y, ff["Y"])
    assert np.array_equal(b["dX"], fb["dX"])
    assert np.array_equal(np.concatenate(b["db1_i"]), fb["db1"])
    assert np.array_equal(b["db2"], fb["db2"])


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bias_finite_differences(act):
    rng = np.random.default_rng(21)
    T, d, dff, h = 3, 5, 7, 1e-6
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.5; W2 = rng.normal(size=(dff, d)) * 0.5
    W3 = rng.normal(size=(d, dff)) * 0.5 if act == "swiglu" else None
    b1, b3, b2 = _bias_inputs(rng, d, dff, act, 0.5)
    dY = rng.normal(size=(T, d))
    P = {"b1": b1, "b2": b2}
    if b3 is not None:
        P["b3"] = b3

    def loss(p):
        return float(np.sum(dY * oracle.forward(X, W1, W2, act=act, W3=W3, b1=p["b1"], b3=p.get("b3"),
                                                 b2=p["b2"])["Y"]))

    g = oracle.backward(X, W1, W2, dY, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    for name, val in P.items():
        num = np.zeros_like(val)
        for i in range(val.size):
            pp = {k: v.copy() for k, v in P.items()}; pp[name][i] += h
            pm = {k: v.copy() for k, v in P.items()}; pm[name][i] -= h
            num[i] = (loss(pp) - loss(pm)) / (2 * h)
        ana = g["d" + name]
        assert np.max(np.abs(num - ana)) / np.max(np.abs(ana)) < 1e-7, name
    # the weight gradients still match finite differences with biases present
    num = np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        Xp = X.copy(); Xp[idx] += h
        Xm = X.copy(); Xm[idx] -= h
        yp = oracle.forward(Xp, W1, W2, act=act, W3=W3, b1=b1, b3=b3, b2=b2)["Y"]
        ym = oracle.forward(Xm, W1, W2, act=act, W3=W3, b1=b1, b3=b3, b2=b2)["Y"]
        num[idx] = np.sum(dY * (yp - ym)) / (2 * h)
    assert np.max(np.abs(num - g["dX"])) / np.max(np.abs(g["dX"])) < 1e-7


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bias_c_oracle_matches_numpy(act):
    rng = np.random.default_rng(31)
    T, d, dff = 17, 12, 40
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.2; W2 = rng.normal(size=(dff, d)) * 0.2
    W3 = rng.normal(size=(d, dff)) * 0.2
    b1, b3, b2 = _bias_inputs(rng, d, dff, act)
    dY = rng.normal(size=(T, d))
    c_f = oracle.forward(X, W1, W2, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    c_b = oracle.backward(X, W1, W2, dY, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    n_f = np_oracle.forward(X, W1, W2, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    n_b = np_oracle.backward(X, W1, W2, dY, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    pairs = [(c_f["Y"], n_f["Y"]), (c_b["dX"], n_b["dX"]), (c_b["dW1"], n_b["dW1"]), (c_b["dW2"], n_b["dW2"]),
             (c_b["db1"], n_b["db1"]), (c_b["db2"], n_b["db2"])]
    if act == "swiglu":
        pairs += [(c_b["db3"], n_b["db3"]), (c_b["dW3"], n_b["dW3"])]
    for a, b in pairs:
        assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.max(np.abs(b)))


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_bias_sampled_rows_and_units(act):
    rng = np.random.default_rng(41)
    T, d, dff = 29, 16, 24
    X = rng.normal(size=(T, d)); W1 = rng.normal(size=(d, dff)) * 0.2; W2 = rng.normal(size=(dff, d)) * 0.2
    W3 = rng.normal(size=(d, dff)) * 0.2 if act == "swiglu" else None
    b1, b3, b2 = _bias_inputs(rng, d, dff, act)
    dY = rng.normal(size=(T, d))
    f = np_oracle.forward(X, W1, W2, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    b = np_oracle.backward(X, W1, W2, dY, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    r = np.array([0, 3, 28])
    Yr, dXr = oracle.rows(X, W1, W2, dY, r, act=act, W3=W3, b1=b1, b3=b3, b2=b2)
    np.testing.assert_allclose(Yr, f["Y"][r], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dXr, b["dX"][r], rtol=0, atol=1e-12)
    u = np.array([0, 7, 23])
    c1, c3, c2, g1, g3 = oracle.wgrad_units(X, W1, W2, dY, u, act=act, W3=W3, b1=b1, b3=b3, with_bias_grads=True)
    np.testing.assert_allclose(c1, b["dW1"][:, u].T, rtol=0, atol=1e-11)
    np.testing.assert_allclose(c2, b["dW2"][u, :], rtol=0, atol=1e-11)
    np.testing.assert_allclose(g1, b["db1"][u], rtol=0, atol=1e-11)
    if act == "swiglu":
        np.testing.assert_allclose(g3, b["db3"][u], rtol=0, atol=1e-11)
    np.testing.assert_allclose(oracle.db2(dY), b["db2"], rtol=0, atol=1e-12)


def test_planted_bias_per_shard_is_caught(tmp_path):
    """Adding b2 inside every shard (before the g-sum) counts it t times; the
    exact sharded == unsharded pin must catch it."""
    src = open(_SRC).read()
    find = "    matmul(T, d, di, H, di, 1, W2_i[s], d, 1, Z, d);\n"
    assert src.count(find) == 1
    msrc = tmp_path / "mutant_bias.c"
    msrc.write_text(src.replace(find, find + "    add_row_bias(T, d, Z, b2);\n"))
    o = oracle.load_variant(oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant_bias.so")))
    inp = si.small_int_inputs(4, 8, [4, 4, 8], "relu")
    b2 = np.arange(8, dtype=np.float64) - 3
    Y, _ = o.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act="relu", b2=b2)
    ff = o.forward(inp.X, inp.W1, inp.W2, act="relu", b2=b2)
    assert np.max(np.abs(Y - ff["Y"])) >= 1.0
    Yc, _ = oracle.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act="relu", b2=b2)
    assert np.array_equal(Yc, oracle.forward(inp.X, inp.W1, inp.W2, act="relu", b2=b2)["Y"])


# ---------------------------------------------------------------- attention projections (QKV by heads, row-split WO)

def _attn_inputs(rng, T, d, dq, dkv, integer=False):
    draw = (lambda *s: rng.integers(-3, 4, s).astype(np.float64)) if integer else (lambda *s: rng.normal(size=s))
    return {"X": draw(T, d), "WQ": draw(d, dq), "WK": draw(d, dkv), "WV": draw(d, dkv), "O": draw(T, dq),
            "WO": draw(dq, d), "dZ": draw(T, d), "dQ": draw(T, dq), "dK": draw(T, dkv), "dV": draw(T, dkv)}


def _attn_args(P):
    return (P["X"], P["WQ"], P["WK"], P["WV"], P["O"], P["WO"], P["dZ"], P["dQ"], P["dK"], P["dV"])


@pytest.mark.parametrize("wq_i,wkv_i", [([16], [16]), ([8, 8], [8, 8]), ([4, 4, 4, 4], [4, 4, 4, 4]),
                                        ([4, 12], [4, 12]), ([8, 8], [4, 4]), ([12, 4, 8], [4, 4, 8])])
def test_attn_sharded_equals_unsharded_exact(wq_i, wkv_i):
    """g-sum of the row-split output projection and f-sum of the three QKV
    input gradients, with and without grouped-query widths: exact on small
    integers."""
    rng = np.random.default_rng(len(wq_i) + sum(wkv_i))
    P = _attn_inputs(rng, 5, 8, sum(wq_i), sum(wkv_i), integer=True)
    f = oracle.attn_forward(*_attn_args(P)[:6])
    b = oracle.attn_backward(*_attn_args(P))
    sq, skv = si.shard_slices(wq_i), si.shard_slices(wkv_i)
    cols = lambda M, sl: [M[:, a:c] for a, c in sl]
    rows = lambda M, sl: [M[a:c] for a, c in sl]
    s = oracle.attn_sharded(P["X"], cols(P["WQ"], sq), cols(P["WK"], skv), cols(P["WV"], skv), cols(P["O"], sq),
                            rows(P["WO"], sq), P["dZ"], cols(P["dQ"], sq), cols(P["dK"], skv), cols(P["dV"], skv))
    assert np.array_equal(s["Z"], f["Z"])
    assert np.array_equal(s["dX"], b["dX"])
    assert np.array_equal(np.concatenate(s["dWO_i"], 0), b["dWO"])
    assert np.array_equal(np.concatenate(s["dWQ_i"], 1), b["dWQ"])
    assert np.array_equal(np.concatenate(s["dWK_i"], 1), b["dWK"])
    assert np.array_equal(np.concatenate(s["dWV_i"], 1), b["dWV"])


def test_attn_finite_differences():
    """L = <dZ, Z> + <dQ, Q> + <dK, K> + <dV, V>: its gradients are the backward's outputs."""
    rng = np.random.default_rng(51)
    P = _attn_inputs(rng, 3, 5, 6, 2)
    h = 1e-6

    def loss(p):
        f = oracle.attn_forward(*_attn_args(p)[:6])
        return float(sum(np.sum(p[g] * f[k]) for g, k in (("dZ", "Z"), ("dQ", "Q"), ("dK", "K"), ("dV", "V"))))

    b = oracle.attn_backward(*_attn_args(P))
    for name, grad in (("X", "dX"), ("WQ", "dWQ"), ("WK", "dWK"), ("WV", "dWV"), ("O", "dO"), ("WO", "dWO")):
        num = np.zeros_like(P[name])
        for idx in np.ndindex(P[name].shape):
            pp = {k: v.copy() for k, v in P.items()}; pp[name][idx] += h
            pm = {k: v.copy() for k, v in P.items()}; pm[name][idx] -= h
            num[idx] = (loss(pp) - loss(pm)) / (2 * h)
        assert np.max(np.abs(num - b[grad])) / np.max(np.abs(b[grad])) < 1e-7, name


def test_attn_c_oracle_matches_numpy():
    rng = np.random.default_rng(61)
    P = _attn_inputs(rng, 19, 16, 24, 8)
    c_f, n_f = oracle.attn_forward(*_attn_args(P)[:6]), np_oracle.attn_forward(*_attn_args(P)[:6])
    c_b, n_b = oracle.attn_backward(*_attn_args(P)), np_oracle.attn_backward(*_attn_args(P))
    for k in ("Q", "K", "V", "Z"):
        assert np.max(np.abs(c_f[k] - n_f[k])) <= 1e-12 * max(1.0, np.max(np.abs(n_f[k])))
    for k in n_b:
        assert np.max(np.abs(c_b[k] - n_b[k])) <= 1e-12 * max(1.0, np.max(np.abs(n_b[k])))


def test_attn_row_and_column_subsets():
    """The projections are row-separable (Q, K, V, Z and dX, dO of a token
    depend on that token's rows only) and the weight gradients column-separable
    (a column of dWQ needs only that column of dQ): the property the sampled
    checks at full size rely on."""
    rng = np.random.default_rng(81)
    P = _attn_inputs(rng, 11, 8, 12, 4)
    f = oracle.attn_forward(*_attn_args(P)[:6])
    b = oracle.attn_backward(*_attn_args(P))
    rows = np.array([0, 4, 10])
    Pr = dict(P)
    for k in ("X", "O", "dZ", "dQ", "dK", "dV"):
        Pr[k] = P[k][rows]
    fr, br = oracle.attn_forward(*_attn_args(Pr)[:6]), oracle.attn_backward(*_attn_args(Pr))
    for k in ("Q", "K", "V", "Z"):
        assert np.allclose(fr[k], f[k][rows], rtol=1e-13, atol=1e-13)
    for k in ("dX", "dO"):
        assert np.allclose(br[k], b[k][rows], rtol=1e-13, atol=1e-13)
    cq, ckv = np.array([1, 7, 11]), np.array([0, 3])
    Pc = dict(P)
    Pc["WQ"], Pc["O"], Pc["WO"], Pc["dQ"] = P["WQ"][:, cq], P["O"][:, cq], P["WO"][cq], P["dQ"][:, cq]
    Pc["WK"], Pc["WV"], Pc["dK"], Pc["dV"] = P["WK"][:, ckv], P["WV"][:, ckv], P["dK"][:, ckv], P["dV"][:, ckv]
    bc = oracle.attn_backward(*_attn_args(Pc))
    assert np.allclose(bc["dWQ"], b["dWQ"][:, cq], rtol=1e-13, atol=1e-13)
    assert np.allclose(bc["dWK"], b["dWK"][:, ckv], rtol=1e-13, atol=1e-13)
    assert np.allclose(bc["dWV"], b["dWV"][:, ckv], rtol=1e-13, atol=1e-13)
    assert np.allclose(bc["dWO"], b["dWO"][cq], rtol=1e-13, atol=1e-13)


def test_planted_attn_f_sum_missing_term_is_caught(tmp_path):
    """Dropping the dV term of the f-sum must change dX (so the finite-difference pin catches it)."""
    src = open(_SRC).read()
    find = "  matmul(T, d, dkv, dV, dkv, 1, WV, 1, dkv, tmp, d);\n  for (int64_t i = 0; i < T * d; ++i) dX[i] += tmp[i];\n"
    assert src.count(find) == 1
    msrc = tmp_path / "mutant_attn.c"
    msrc.write_text(src.replace(find, ""))
    o = oracle.load_variant(oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant_attn.so")))
    rng = np.random.default_rng(71)
    P = _attn_inputs(rng, 3, 4, 4, 2)
    bad, good = o.attn_backward(*_attn_args(P)), oracle.attn_backward(*_attn_args(P))
    assert np.max(np.abs(bad["dX"] - good["dX"])) > 1e-3


def test_planted_attn_kv_operand_swap_is_caught(tmp_path):
    """Projecting K with WV (a swapped operand) must break the numpy cross-check."""
    src = open(_SRC).read()
    find = "  matmul(T, dkv, d, X, d, 1, WK, dkv, 1, K, dkv);\n"
    assert src.count(find) == 1
    msrc = tmp_path / "mutant_kv.c"
    msrc.write_text(src.replace(find, "  matmul(T, dkv, d, X, d, 1, WV, dkv, 1, K, dkv);\n"))
    o = oracle.load_variant(oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant_kv.so")))
    rng = np.random.default_rng(72)
    P = _attn_inputs(rng, 6, 8, 8, 4)
    bad = o.attn_forward(*_attn_args(P)[:6])
    good = np_oracle.attn_forward(*_attn_args(P)[:6])
    assert np.max(np.abs(bad["K"] - good["K"])) > 1e-3


# ---------------------------------------------------------------- sequence-parallel layout (stripes of tokens)

def _stripes(M, rows):
    out, r = [], 0
    for n in rows:
        out.append(M[r:r + n].copy())
        r += n
    return out


@pytest.mark.parametrize("act", ["identity", "relu", "swiglu"])
@pytest.mark.parametrize("rows", [[7], [3, 4], [1, 2, 4], [0, 7], [2, 0, 5]])
def test_sp_equals_gathered_sharded_block_exact(act, rows):
    """The SP layout (all-gather of X before the block, reduce-scatter of the
    partial outputs after it, and the mirror in backward) is the sharded block
    with its rows cut into stripes: exact on small integers."""
    inp = si.small_int_inputs(7, 6, (4, 2), "swiglu" if act == "swiglu" else "gelu", seed=len(rows) + 3)
    W3_i = inp.W3_i if act == "swiglu" else None
    Y, H_i = oracle.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act=act, W3_i=W3_i)
    b = oracle.backward_sharded(inp.X, inp.W1_i, inp.W2_i, inp.dY, act=act, W3_i=W3_i)
    Y_j, H_sp = oracle.forward_sp(_stripes(inp.X.numpy(), rows), inp.W1_i, inp.W2_i, act=act, W3_i=W3_i)
    bs = oracle.backward_sp(_stripes(inp.X.numpy(), rows), inp.W1_i, inp.W2_i, _stripes(inp.dY.numpy(), rows),
                            act=act, W3_i=W3_i)
    assert [y.shape[0] for y in Y_j] == rows
    assert np.array_equal(np.concatenate(Y_j, 0), Y)
    assert np.array_equal(np.concatenate(bs["dX_j"], 0), b["dX"])
    for k in ("dW1_i", "dW2_i") + (("dW3_i",) if act == "swiglu" else ()):
        for x, y in zip(bs[k], b[k]):
            assert np.array_equal(x, y)
    for x, y in zip(H_sp, H_i):
        assert np.array_equal(x, y)
    assert np.array_equal(bs["db2"], b["db2"])


def test_sp_bias_added_once_per_token():
    """b2 is added to every stripe row once, after the reduce-scatter sum."""
    inp = si.small_int_inputs(6, 4, (2, 2), "gelu", seed=9)
    b2 = np.arange(4, dtype=np.float64)
    Y, _ = oracle.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act="identity", b2=b2)
    Y_j, _ = oracle.forward_sp(_stripes(inp.X.numpy(), [2, 4]), inp.W1_i, inp.W2_i, act="identity", b2=b2)
    assert np.array_equal(np.concatenate(Y_j, 0), Y)


def test_planted_sp_reduce_scatter_without_sum_is_caught(tmp_path):
    """A reduce-scatter that keeps only shard 0's partial output must fail the exact pin."""
    src = open(_SRC).read()
    find = "for (int32_t s = 0; s < t; ++s) v += Z["
    assert src.count(find) == 1
    msrc = tmp_path / "mutant_sp.c"
    msrc.write_text(src.replace(find, "for (int32_t s = 0; s < 1; ++s) v += Z["))
    o = oracle.load_variant(oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant_sp.so")))
    inp = si.small_int_inputs(5, 4, (2, 2), "gelu", seed=11)
    Y, _ = oracle.forward_sharded(inp.X, inp.W1_i, inp.W2_i, act="identity")
    Y_j, _ = o.forward_sp(_stripes(inp.X.numpy(), [2, 3]), inp.W1_i, inp.W2_i, act="identity")
    assert not np.array_equal(np.concatenate(Y_j, 0), Y)
