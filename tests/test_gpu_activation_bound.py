"""The epilogues' activation forms against the fp64 oracle within a derived
error bound, element by element on a dense fp32 grid.

The bf16 tensor-core epilogues do not call erff: Phi(-|a|) comes from the
rational approximation of erfc given as formula 7.1.26 in Abramowitz & Stegun
(absolute error at most 1.5e-7), with the fast exponential and reciprocal;
the sigmoid uses the same fast exponential and reciprocal.  The fp32 path
calls erff / expf.  tpmlp_eval_activation runs those exact instruction
sequences on device arrays; each output is compared with the oracle's
act_value / act_grad (fp64) on every point of [-12, 12] in steps of 2^-10,
plus signed zeros, tiny and huge magnitudes up to the largest float.

Bounds (u = 2^-24, the fp32 unit roundoff; q = Phi(-|a|) = erfc(|a|/sqrt 2)/2):
  * the exponentials are ex2.approx (relative error about 2^-22, 4u) of an
    argument that carries the log2(e) scale (a^2 times -log2(e)/2; -g log2(e)
    for the sigmoid), whose three roundings add a relative error of at most
    1.5 a^2 u, resp. 2 |g| u, to the result; the fast reciprocal is within
    2 ulp; an ulp of a result r is at most 2u |r|;
  * q: the approximation is within 7.5e-8 (half of A&S's 1.5e-7, since
    q = erfc / 2); its fp32 evaluation (reciprocal, a Horner chain whose
    condition number is at most 4.5 on t in (0, 1], the exponential of
    -a^2/2 and the final product, about (30 + 1.5 a^2) u in all) adds at most
    C_q(a) q with C_q(a) = (64 + 2 a^2) u;
  * GeLU(a) = max(a, 0) - |a| q, one fma:  |a| (7.5e-8 + C_q q) + u |GeLU|;
  * GeLU'(a) = 1/2 + sign(a)(1/2 - q) + a phi(a):
        7.5e-8 + C_q q + 2u + |a| phi(a) (8 + 2 a^2) u + 2u |GeLU'|,
    and dA = dH GeLU' adds u |dA|;
  * sigmoid s = 1 / (1 + e^-g): relative error
        d_s = (9 + (4 + 2.35 |g|)(1 - s)) u,
    H = U Swish(g) and dU = dH Swish(g): (d_s + 2u) |result|;
    dG = dH U (s + g s (1 - s)): |dH U| (s d_s (1 + 2|g|) + 2u (|Swish'| + |g| s (1 - s))) + 2u |dG|;
  * the fp32 path (erff, expf within 2 ulp): GeLU |a| 8u + |a|^2 phi(a) u + u |GeLU|;
    GeLU' 8u + |a| phi(a) (8 + a^2) u + 2u |GeLU'|; the Swish forms as above
    with 2.35 |g| replaced by 4 (expf's bound does not grow with |g|).
Every bound also has an absolute floor of 1e-34 (flushed subnormals, and the
fast reciprocal returns 0 for divisors above 2^126); a reference beyond the
fp32 range must give an infinity of its sign.  At
+-inf the forms give NaN or the limit, never a finite wrong value (the
epilogues' inputs are finite fp32 accumulators).
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
FLT_MAX = float(np.finfo(np.float32).max)


def _grid():
    g = np.arange(-12 * 1024, 12 * 1024 + 1, dtype=np.float64) / 1024.0
    extra = [0.0, -0.0, 1e-30, -1e-30, 1e-6, -1e-6, 20.0, -20.0, 40.0, -40.0, 87.0, -87.0, 100.0, -100.0, 1e4,
             -1e4, 1e20, -1e20, 1e30, -1e30, FLT_MAX, -FLT_MAX]
    return np.concatenate([g, np.array(extra)]).astype(np.float32)


def _ref(fn, xs):
    return np.array([fn(float(v)) for v in xs], dtype=np.float64)


def _phi(a):
    return np.exp(-0.5 * a * a) / math.sqrt(2 * math.pi)


def _q(a):
    from scipy.special import erfc
    return 0.5 * erfc(np.abs(a) / math.sqrt(2.0))


def _run(tp, form, x, y=None, dh=None, nout=1):
    dev = lambda v: None if v is None else torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
    xd, yd, dd = dev(x), dev(y), dev(dh)
    outs = [torch.full_like(xd, float("nan")) for _ in range(nout)] + [None] * (3 - nout)
    tp.tpmlp_eval_activation(form, xd, yd, dd, *outs)
    torch.cuda.synchronize()
    return [o.double().cpu().numpy() for o in outs[:nout]]


def _check(name, got, ref, bound):
    # a reference beyond the fp32 range must come out as an infinity of its sign
    over = np.isfinite(ref) & (np.abs(ref) > FLT_MAX)
    assert np.all(np.isinf(got[over]) & (np.sign(got[over]) == np.sign(ref[over]))), f"{name}: overflow"
    finite = np.isfinite(ref) & ~over
    err = np.abs(got[finite] - ref[finite])
    b = bound[finite] + 1e-34
    ratio = err / b
    worst = int(np.argmax(ratio))
    assert np.all(np.isfinite(got[finite])), f"{name}: non-finite output for a finite reference"
    assert ratio[worst] <= 1.0, (f"{name}: error {err[worst]:.3e} above bound {b[worst]:.3e} "
                                 f"(ratio {ratio[worst]:.2f})")
    return float(ratio.max())


def _gelu_refs(x):
    a = x.astype(np.float64)
    return _ref(lambda v: oracle.act_value("gelu", v), a), _ref(lambda v: oracle.act_grad("gelu", v), a)


def _gelu_bounds(a, G, Gp, dh):
    q = _q(a)
    cq = (64.0 + 2.0 * a * a) * U
    with np.errstate(over="ignore", invalid="ignore"):
        b_g = np.abs(a) * (7.5e-8 + cq * q) + U * np.abs(G)
        b_gp = 7.5e-8 + cq * q + 2 * U + np.abs(a) * _phi(a) * (8 + 2 * a * a) * U + 2 * U * np.abs(Gp)
    b_da = np.abs(dh) * b_gp + U * np.abs(dh * Gp)
    return np.nan_to_num(b_g, nan=np.inf), np.nan_to_num(b_da, nan=np.inf)


def test_gelu_forms_within_bound(gpu_lib):
    tp = gpu_lib
    x = _grid()
    rng = np.random.default_rng(5)
    dh = rng.uniform(-3, 3, size=x.shape).astype(np.float32)
    a = x.astype(np.float64)
    G, Gp = _gelu_refs(x)
    b_g, b_da = _gelu_bounds(a, G, Gp, dh.astype(np.float64))
    ref_da = dh.astype(np.float64) * Gp
    (h,) = _run(tp, "gelu", x, nout=1)
    (da,) = _run(tp, "gelu_bwd", x, dh=dh, nout=1)
    da2, h2 = _run(tp, "gelu_bwd_h", x, dh=dh, nout=2)
    _check("GeLU", h, G, b_g)
    _check("dA", da, ref_da, b_da)
    assert np.array_equal(da2, da), "dA differs with and without the recomputed H"
    assert np.array_equal(h2, h), "the recomputed H differs from the forward epilogue's"
    # GeLU(0) = 0 and GeLU'(0) = 1/2 exactly; the limits at large magnitudes
    z = np.where(x == 0)[0]
    assert np.all(h[z] == 0.0) and np.all(da[z] == dh[z].astype(np.float64) * 0.5)
    big = np.abs(a) >= 20
    assert np.all(h[big & (a > 0)] == a[big & (a > 0)]) and np.all(h[big & (a < 0)] == 0.0)


def test_swiglu_forms_within_bound(gpu_lib):
    tp = gpu_lib
    g = _grid()
    rng = np.random.default_rng(6)
    u = rng.uniform(-3, 3, size=g.shape).astype(np.float32)
    dh = rng.uniform(-3, 3, size=g.shape).astype(np.float32)
    gd, ud, dd = g.astype(np.float64), u.astype(np.float64), dh.astype(np.float64)
    S = _ref(lambda v: oracle.act_value("swiglu", v), gd)   # Swish(g)
    Sp = _ref(lambda v: oracle.act_grad("swiglu", v), gd)   # Swish'(g)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-gd))
    ds = (9 + (4 + 2.35 * np.abs(gd)) * (1 - s)) * U
    ref_h, ref_du, ref_dg = ud * S, dd * S, dd * ud * Sp
    b_h = (ds + 2 * U) * np.abs(ref_h)
    b_du = (ds + 2 * U) * np.abs(ref_du)
    b_dg = np.abs(dd * ud) * (s * ds * (1 + 2 * np.abs(gd)) + 2 * U * (np.abs(Sp) + np.abs(gd) * s * (1 - s))) \
        + 2 * U * np.abs(ref_dg)
    (h,) = _run(tp, "swiglu", g, y=u, nout=1)
    dg, du = _run(tp, "swiglu_bwd", g, y=u, dh=dh, nout=2)
    dg2, du2, h2 = _run(tp, "swiglu_bwd_h", g, y=u, dh=dh, nout=3)
    _check("H", h, ref_h, b_h)
    _check("dU", du, ref_du, b_du)
    _check("dG", dg, ref_dg, b_dg)
    assert np.array_equal(dg2, dg) and np.array_equal(du2, du)
    assert np.array_equal(h2, h), "the recomputed H differs from the forward epilogue's"


def test_fp32_path_forms_within_bound(gpu_lib):
    tp = gpu_lib
    x = _grid()
    rng = np.random.default_rng(7)
    y = rng.uniform(-3, 3, size=x.shape).astype(np.float32)
    dh = rng.uniform(-3, 3, size=x.shape).astype(np.float32)
    a, yd, dd = x.astype(np.float64), y.astype(np.float64), dh.astype(np.float64)
    G, Gp = _gelu_refs(x)
    with np.errstate(over="ignore", invalid="ignore"):
        b_g = np.abs(a) * 8 * U + a * a * _phi(a) * U + U * np.abs(G)
        b_gp = 8 * U + np.abs(a) * _phi(a) * (8 + a * a) * U + 2 * U * np.abs(Gp)
    b_da = np.abs(dd) * np.nan_to_num(b_gp, nan=np.inf) + U * np.abs(dd * Gp)
    h, da = _run(tp, "fp32_gelu", x, dh=dh, nout=2)
    _check("fp32 GeLU", h, G, np.nan_to_num(b_g, nan=np.inf))
    _check("fp32 dA", da, dd * Gp, b_da)
    S = _ref(lambda v: oracle.act_value("swiglu", v), a)
    Sp = _ref(lambda v: oracle.act_grad("swiglu", v), a)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-a))
    ds = (9 + 4 * (1 - s)) * U
    hs, dg, du = _run(tp, "fp32_swiglu", x, y=y, dh=dh, nout=3)
    _check("fp32 H", hs, yd * S, (ds + 2 * U) * np.abs(yd * S))
    _check("fp32 dU", du, dd * S, (ds + 2 * U) * np.abs(dd * S))
    _check("fp32 dG", dg, dd * yd * Sp, np.abs(dd * yd) * (s * ds * (1 + 2 * np.abs(a)) + 2 * U * (
        np.abs(Sp) + np.abs(a) * s * (1 - s))) + 2 * U * np.abs(dd * yd * Sp))


@pytest.mark.parametrize("form,nout,needs", [("gelu", 1, ""), ("gelu_bwd_h", 2, "d"), ("swiglu", 1, "y"),
                                             ("swiglu_bwd_h", 3, "yd"), ("fp32_gelu", 2, "d"),
                                             ("fp32_swiglu", 3, "yd")])
def test_infinities_give_nan_or_the_limit(gpu_lib, form, nout, needs):
    """+-inf lies outside the epilogues' domain (their inputs are finite fp32
    accumulators); the forms must not turn it into a finite wrong value."""
    tp = gpu_lib
    x = np.array([np.inf, -np.inf] * 16, dtype=np.float32)
    one = np.ones_like(x)
    outs = _run(tp, form, x, y=one if "y" in needs else None, dh=one if "d" in needs else None, nout=nout)
    lim_g = np.where(x > 0, np.inf, 0.0)       # GeLU(+inf) = inf, GeLU(-inf) -> 0
    lim_gp = np.where(x > 0, 1.0, 0.0)         # GeLU' -> 1, 0
    lim_s = np.where(x > 0, np.inf, 0.0)       # Swish -> inf, 0
    lim_sp = np.where(x > 0, 1.0, 0.0)         # Swish' -> 1, 0
    lims = {"gelu": [lim_g], "gelu_bwd_h": [lim_gp, lim_g], "swiglu": [lim_s], "swiglu_bwd_h": [lim_sp, lim_s, lim_s],
            "fp32_gelu": [lim_g, lim_gp], "fp32_swiglu": [lim_s, lim_sp, lim_s]}[form]
    for o, lim in zip(outs, lims):
        ok = np.isnan(o) | (o == lim)
        assert ok.all(), f"{form}: finite wrong value at an infinite input: {o[~ok]}"
