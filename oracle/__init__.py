"""fp64 CPU oracle for the t-sharded Megatron MLP block.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA path (``megatron_tensor_transformer_column_gb300``)
and neither side imports the other.

Two independent implementations live here:

* ``tpmlp_oracle.c`` (loaded through ctypes, OpenMP over output rows): the
  unsharded block, the pages' sharded formulation, and per-row / per-unit
  sampled outputs for problems too large to compute in full; also the
  attention block's QKV and output projections, unsharded and split by heads;
  and the sequence-parallel layout (token stripes gathered before the block,
  the partial outputs reduce-scattered into stripes after it);
* ``np_oracle.py``: the same block written with numpy float64 matrix products,
  used to cross-check the C oracle on small shapes.

Sources (page title, section): "Parallelism" tag page of Jiang Yi's homepage,
post "megatron-lm", Method / FFN (column split of W1, row split of W2, f/g
table, SwiGLU split); "AI Training Network Primer", ch. 3, section 3.4
"Megatron's matrix split" (Fig. 3.4, 3.6); "Tensor parallelism"
(brunomaga.github.io), "Megatron-LM tensor parallelism" (Megatron_f,
Megatron_g, Megatron_FeedForward).

Every function has a pin in ``tests/test_oracle_pins.py`` (closed forms,
exact small-integer identities, finite differences, the numpy cross-check and
planted-mistake checks); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

ACT_GELU = 0
ACT_SWIGLU = 1
ACT_IDENTITY = 2  # test hook: keeps integer inputs integral
ACT_RELU = 3  # test hook

ACTS = {"gelu": ACT_GELU, "swiglu": ACT_SWIGLU, "identity": ACT_IDENTITY, "relu": ACT_RELU}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tpmlp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtpmlp_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP) into oracle/_build/ (or ``out``)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-D_GNU_SOURCE",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    i64, i32, ci, dp = ctypes.c_int64, ctypes.c_int32, ctypes.c_int, ctypes.c_void_p
    pp = ctypes.POINTER(ctypes.c_void_p)
    lib.oracle_forward.argtypes = [i64, i64, i64, ci, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_forward.restype = ci
    lib.oracle_backward.argtypes = [i64, i64, i64, ci, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                    dp]
    lib.oracle_backward.restype = ci
    lib.oracle_forward_sharded.argtypes = [i64, i64, i32, dp, ci, dp, pp, pp, pp, pp, pp, dp, dp, pp]
    lib.oracle_forward_sharded.restype = ci
    lib.oracle_backward_sharded.argtypes = [i64, i64, i32, dp, ci, dp, pp, pp, pp, pp, pp, dp, dp, pp, pp, pp, pp,
                                            pp, dp]
    lib.oracle_backward_sharded.restype = ci
    lib.oracle_forward_sp.argtypes = [i64, i64, i32, dp, ci, i32, dp, pp, pp, pp, pp, pp, pp, dp, pp, pp]
    lib.oracle_forward_sp.restype = ci
    lib.oracle_backward_sp.argtypes = [i64, i64, i32, dp, ci, i32, dp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp,
                                       pp, dp]
    lib.oracle_backward_sp.restype = ci
    lib.oracle_rows.argtypes = [i64, i64, i64, ci, dp, dp, dp, dp, dp, dp, dp, dp, i64, dp, dp, dp] + [dp] * 5
    lib.oracle_rows.restype = ci
    lib.oracle_wgrad_units.argtypes = [i64, i64, i64, ci, dp, dp, dp, dp, dp, dp, dp, i64, dp, dp, dp, dp, dp, dp]
    lib.oracle_wgrad_units.restype = ci
    lib.oracle_attn_forward.argtypes = [i64, i64, i64, i64] + [dp] * 10
    lib.oracle_attn_forward.restype = ci
    lib.oracle_attn_backward.argtypes = [i64, i64, i64, i64] + [dp] * 16
    lib.oracle_attn_backward.restype = ci
    lib.oracle_attn_sharded.argtypes = [i64, i64, i32, dp, dp, dp, pp, pp, pp, pp, pp, dp, pp, pp, pp, dp, dp, pp, pp,
                                        pp, pp]
    lib.oracle_attn_sharded.restype = ci
    lib.oracle_db2.argtypes = [i64, i64, dp, dp]
    lib.oracle_db2.restype = ci
    lib.oracle_act_value.argtypes = [ci, ctypes.c_double]
    lib.oracle_act_value.restype = ctypes.c_double
    lib.oracle_act_grad.argtypes = [ci, ctypes.c_double]
    lib.oracle_act_grad.restype = ctypes.c_double
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ci
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def load_variant(path: str) -> "COracle":
    """Load another build of the C oracle (used by the planted-mistake tests)."""
    return COracle(_bind(ctypes.CDLL(path)))


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> numpy (float64, contiguous)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _act(act):
    return ACTS[act] if isinstance(act, str) else int(act)


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed with code {rc}")


class COracle:
    """Bound C oracle; the module-level functions use the default build."""

    def __init__(self, lib):
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def act_value(self, act, a: float) -> float:
        return float(self.lib.oracle_act_value(_act(act), float(a)))

    def act_grad(self, act, a: float) -> float:
        return float(self.lib.oracle_act_grad(_act(act), float(a)))

    def forward(self, X, W1, W2, act="gelu", W3=None, b1=None, b3=None, b2=None):
        """Unsharded forward.  Returns dict with A (SwiGLU: G), U, H, Y (fp64)."""
        lib = self.lib
        a = _act(act)
        X, W1, W2, W3 = _f64(X), _f64(W1), _f64(W2), _f64(W3)
        b1, b3, b2 = _f64(b1), _f64(b3), _f64(b2)
        T, d = X.shape
        dff = W1.shape[1]
        A = np.empty((T, dff)); H = np.empty((T, dff)); Y = np.empty((T, d))
        U = np.empty((T, dff)) if a == ACT_SWIGLU else None
        _check(lib.oracle_forward(T, d, dff, a, _ptr(X), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(b1), _ptr(b3), _ptr(b2),
                                  _ptr(A), _ptr(U), _ptr(H), _ptr(Y)), "oracle_forward")
        return {"A": A, "U": U, "H": H, "Y": Y}

    def backward(self, X, W1, W2, dY, act="gelu", W3=None, b1=None, b3=None, b2=None):
        """Unsharded backward.  Returns dict with dX, dW1, dW3, dW2, db1, db3, db2, dA (SwiGLU: dG), dU."""
        lib = self.lib
        a = _act(act)
        X, W1, W2, W3, dY = _f64(X), _f64(W1), _f64(W2), _f64(W3), _f64(dY)
        b1, b3, b2 = _f64(b1), _f64(b3), _f64(b2)
        T, d = X.shape
        dff = W1.shape[1]
        dX = np.empty((T, d)); dW1 = np.empty((d, dff)); dW2 = np.empty((dff, d))
        dA = np.empty((T, dff))
        sw = a == ACT_SWIGLU
        dW3 = np.empty((d, dff)) if sw else None
        dU = np.empty((T, dff)) if sw else None
        db1, db2 = np.empty(dff), np.empty(d)
        db3 = np.empty(dff) if sw else None
        _check(lib.oracle_backward(T, d, dff, a, _ptr(X), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(b1), _ptr(b3), _ptr(b2),
                                   _ptr(dY), _ptr(dX), _ptr(dW1), _ptr(dW3), _ptr(dW2), _ptr(db1), _ptr(db3), _ptr(db2),
                                   _ptr(dA), _ptr(dU)), "oracle_backward")
        return {"dX": dX, "dW1": dW1, "dW3": dW3, "dW2": dW2, "db1": db1, "db3": db3, "db2": db2, "dA": dA, "dU": dU}

    def forward_sharded(self, X, W1_i, W2_i, act="gelu", W3_i=None, b1_i=None, b3_i=None, b2=None):
        """The pages' per-shard forward with the g-sum (b2 added once after it).  Returns (Y, [H_i])."""
        lib = self.lib
        a = _act(act)
        X = _f64(X)
        W1_i = [_f64(w) for w in W1_i]; W2_i = [_f64(w) for w in W2_i]
        W3_i = [_f64(w) for w in W3_i] if W3_i is not None else None
        b1_i = [_f64(b) for b in b1_i] if b1_i is not None else None
        b3_i = [_f64(b) for b in b3_i] if b3_i is not None else None
        b2 = _f64(b2)
        T, d = X.shape
        t = len(W1_i)
        d_i = np.array([w.shape[1] for w in W1_i], dtype=np.int64)
        Y = np.empty((T, d))
        H_i = [np.empty((T, int(di))) for di in d_i]
        _check(lib.oracle_forward_sharded(T, d, t, d_i.ctypes.data_as(ctypes.c_void_p), a, _ptr(X), _ptrs(W1_i),
                                          _ptrs(W3_i) if W3_i else None, _ptrs(W2_i), _ptrs(b1_i) if b1_i else None,
                                          _ptrs(b3_i) if b3_i else None, _ptr(b2), _ptr(Y), _ptrs(H_i)),
               "oracle_forward_sharded")
        return Y, H_i

    def backward_sharded(self, X, W1_i, W2_i, dY, act="gelu", W3_i=None, b1_i=None, b3_i=None):
        """The pages' per-shard backward with the f-sum.  Returns dict dX, dW1_i, dW3_i, dW2_i, db1_i, db3_i, db2."""
        lib = self.lib
        a = _act(act)
        X, dY = _f64(X), _f64(dY)
        W1_i = [_f64(w) for w in W1_i]; W2_i = [_f64(w) for w in W2_i]
        W3_i = [_f64(w) for w in W3_i] if W3_i is not None else None
        b1_i = [_f64(b) for b in b1_i] if b1_i is not None else None
        b3_i = [_f64(b) for b in b3_i] if b3_i is not None else None
        T, d = X.shape
        t = len(W1_i)
        d_i = np.array([w.shape[1] for w in W1_i], dtype=np.int64)
        dX = np.empty((T, d))
        dW1_i = [np.empty((d, int(di))) for di in d_i]
        dW2_i = [np.empty((int(di), d)) for di in d_i]
        dW3_i = [np.empty((d, int(di))) for di in d_i] if W3_i else None
        db1_i = [np.empty(int(di)) for di in d_i]
        db3_i = [np.empty(int(di)) for di in d_i] if W3_i else None
        db2 = np.empty(d)
        _check(lib.oracle_backward_sharded(T, d, t, d_i.ctypes.data_as(ctypes.c_void_p), a, _ptr(X), _ptrs(W1_i),
                                           _ptrs(W3_i) if W3_i else None, _ptrs(W2_i), _ptrs(b1_i) if b1_i else None,
                                           _ptrs(b3_i) if b3_i else None, _ptr(dY), _ptr(dX), _ptrs(dW1_i),
                                           _ptrs(dW3_i) if dW3_i else None, _ptrs(dW2_i), _ptrs(db1_i),
                                           _ptrs(db3_i) if db3_i else None, _ptr(db2)),
               "oracle_backward_sharded")
        return {"dX": dX, "dW1_i": dW1_i, "dW3_i": dW3_i, "dW2_i": dW2_i, "db1_i": db1_i, "db3_i": db3_i, "db2": db2}

    def forward_sp(self, X_j, W1_i, W2_i, act="gelu", W3_i=None, b1_i=None, b3_i=None, b2=None):
        """Sequence-parallel layout: X given as token stripes X_j; returns (Y_j stripes, [H_i])."""
        lib = self.lib
        a = _act(act)
        X_j = [_f64(x) for x in X_j]
        W1_i = [_f64(w) for w in W1_i]; W2_i = [_f64(w) for w in W2_i]
        W3_i = [_f64(w) for w in W3_i] if W3_i is not None else None
        b1_i = [_f64(b) for b in b1_i] if b1_i is not None else None
        b3_i = [_f64(b) for b in b3_i] if b3_i is not None else None
        b2 = _f64(b2)
        rows = np.array([x.shape[0] for x in X_j], dtype=np.int64)
        T, d = int(rows.sum()), W2_i[0].shape[1]
        d_i = np.array([w.shape[1] for w in W1_i], dtype=np.int64)
        Y_j = [np.empty((int(r), d)) for r in rows]
        H_i = [np.empty((T, int(di))) for di in d_i]
        _check(lib.oracle_forward_sp(T, d, len(W1_i), d_i.ctypes.data_as(ctypes.c_void_p), a, len(X_j),
                                     rows.ctypes.data_as(ctypes.c_void_p), _ptrs(X_j), _ptrs(W1_i),
                                     _ptrs(W3_i) if W3_i else None, _ptrs(W2_i), _ptrs(b1_i) if b1_i else None,
                                     _ptrs(b3_i) if b3_i else None, _ptr(b2), _ptrs(Y_j), _ptrs(H_i)),
               "oracle_forward_sp")
        return Y_j, H_i

    def backward_sp(self, X_j, W1_i, W2_i, dY_j, act="gelu", W3_i=None, b1_i=None, b3_i=None):
        """Sequence-parallel layout: X, dY as token stripes; returns dict dX_j, dW1_i, dW3_i, dW2_i, db1_i, db3_i, db2."""
        lib = self.lib
        a = _act(act)
        X_j = [_f64(x) for x in X_j]; dY_j = [_f64(x) for x in dY_j]
        W1_i = [_f64(w) for w in W1_i]; W2_i = [_f64(w) for w in W2_i]
        W3_i = [_f64(w) for w in W3_i] if W3_i is not None else None
        b1_i = [_f64(b) for b in b1_i] if b1_i is not None else None
        b3_i = [_f64(b) for b in b3_i] if b3_i is not None else None
        rows = np.array([x.shape[0] for x in X_j], dtype=np.int64)
        T, d = int(rows.sum()), W2_i[0].shape[1]
        d_i = np.array([w.shape[1] for w in W1_i], dtype=np.int64)
        dX_j = [np.empty((int(r), d)) for r in rows]
        dW1_i = [np.empty((d, int(di))) for di in d_i]
        dW2_i = [np.empty((int(di), d)) for di in d_i]
        dW3_i = [np.empty((d, int(di))) for di in d_i] if W3_i else None
        db1_i = [np.empty(int(di)) for di in d_i]
        db3_i = [np.empty(int(di)) for di in d_i] if W3_i else None
        db2 = np.empty(d)
        _check(lib.oracle_backward_sp(T, d, len(W1_i), d_i.ctypes.data_as(ctypes.c_void_p), a, len(X_j),
                                      rows.ctypes.data_as(ctypes.c_void_p), _ptrs(X_j), _ptrs(W1_i),
                                      _ptrs(W3_i) if W3_i else None, _ptrs(W2_i), _ptrs(b1_i) if b1_i else None,
                                      _ptrs(b3_i) if b3_i else None, _ptrs(dY_j), _ptrs(dX_j), _ptrs(dW1_i),
                                      _ptrs(dW3_i) if dW3_i else None, _ptrs(dW2_i), _ptrs(db1_i),
                                      _ptrs(db3_i) if db3_i else None, _ptr(db2)),
               "oracle_backward_sp")
        return {"dX_j": dX_j, "dW1_i": dW1_i, "dW3_i": dW3_i, "dW2_i": dW2_i, "db1_i": db1_i, "db3_i": db3_i, "db2": db2}

    def rows(self, X, W1, W2, dY, rows_idx, act="gelu", W3=None, b1=None, b3=None, b2=None,
             intermediates=False):
        """Y[r, :] and dX[r, :] for the listed token rows.  Returns (Y_rows, dX_rows);
        with intermediates=True (Y_rows, dX_rows, inter), inter holding the same
        rows of A (SwiGLU: G), H and dA (SwiGLU: dG), and for SwiGLU U and dU,
        each [len(rows) x dff]."""
        lib = self.lib
        a = _act(act)
        X, W1, W2, W3, dY = _f64(X), _f64(W1), _f64(W2), _f64(W3), _f64(dY)
        b1, b3, b2 = _f64(b1), _f64(b3), _f64(b2)
        T, d = X.shape
        dff = W1.shape[1]
        r = np.ascontiguousarray(rows_idx, dtype=np.int64)
        Yr = np.empty((len(r), d)); dXr = np.empty((len(r), d))
        sw = act == "swiglu"
        inter = {}
        if intermediates:
            names = ("A", "U", "H", "dA", "dU") if sw else ("A", "H", "dA")
            inter = {k: np.empty((len(r), dff)) for k in names}
        _check(lib.oracle_rows(T, d, dff, a, _ptr(X), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(b1), _ptr(b3), _ptr(b2),
                               _ptr(dY), len(r), _ptr(r), _ptr(Yr), _ptr(dXr), _ptr(inter.get("A")),
                               _ptr(inter.get("U")), _ptr(inter.get("H")), _ptr(inter.get("dA")),
                               _ptr(inter.get("dU"))), "oracle_rows")
        if intermediates:
            return Yr, dXr, inter
        return Yr, dXr

    def attn_forward(self, X, WQ, WK, WV, O, WO):
        """Attention projections: Q, K, V = X WQ, X WK, X WV and Z = O WO (fp64).
        WQ [d x dq], WK and WV [d x dkv], O [T x dq], WO [dq x d]."""
        X, WQ, WK, WV, O, WO = (_f64(m) for m in (X, WQ, WK, WV, O, WO))
        T, d = X.shape
        dq, dkv = WQ.shape[1], WK.shape[1]
        Q, K, V, Z = np.empty((T, dq)), np.empty((T, dkv)), np.empty((T, dkv)), np.empty((T, d))
        _check(self.lib.oracle_attn_forward(T, d, dq, dkv, _ptr(X), _ptr(WQ), _ptr(WK), _ptr(WV), _ptr(O), _ptr(WO),
                                            _ptr(Q), _ptr(K), _ptr(V), _ptr(Z)), "oracle_attn_forward")
        return {"Q": Q, "K": K, "V": V, "Z": Z}

    def attn_backward(self, X, WQ, WK, WV, O, WO, dZ, dQ, dK, dV):
        """Gradients of the attention projections given dZ and the core's dQ, dK, dV."""
        X, WQ, WK, WV, O, WO, dZ, dQ, dK, dV = (_f64(m) for m in (X, WQ, WK, WV, O, WO, dZ, dQ, dK, dV))
        T, d = X.shape
        dq, dkv = WQ.shape[1], WK.shape[1]
        out = {"dO": np.empty((T, dq)), "dWO": np.empty((dq, d)), "dX": np.empty((T, d)), "dWQ": np.empty((d, dq)),
               "dWK": np.empty((d, dkv)), "dWV": np.empty((d, dkv))}
        _check(self.lib.oracle_attn_backward(T, d, dq, dkv, _ptr(X), _ptr(WQ), _ptr(WK), _ptr(WV), _ptr(O),
                                             _ptr(WO), _ptr(dZ), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(out["dO"]),
                                             _ptr(out["dWO"]), _ptr(out["dX"]), _ptr(out["dWQ"]), _ptr(out["dWK"]),
                                             _ptr(out["dWV"])), "oracle_attn_backward")
        return out

    def attn_sharded(self, X, WQ_i, WK_i, WV_i, O_i, WO_i, dZ, dQ_i, dK_i, dV_i):
        """Per-shard projections with the g-sum (Z) and the f-sum (dX), and the
        per-shard weight gradients dWO_i, dWQ_i, dWK_i, dWV_i."""
        X, dZ = _f64(X), _f64(dZ)
        L = lambda xs: [_f64(x) for x in xs]
        WQ_i, WK_i, WV_i, O_i, WO_i, dQ_i, dK_i, dV_i = map(L, (WQ_i, WK_i, WV_i, O_i, WO_i, dQ_i, dK_i, dV_i))
        T, d = X.shape
        wq = np.array([m.shape[1] for m in WQ_i], dtype=np.int64)
        wkv = np.array([m.shape[1] for m in WK_i], dtype=np.int64)
        Z, dX = np.empty((T, d)), np.empty((T, d))
        dWO_i = [np.empty((int(x), d)) for x in wq]
        dWQ_i = [np.empty((d, int(x))) for x in wq]
        dWK_i = [np.empty((d, int(x))) for x in wkv]
        dWV_i = [np.empty((d, int(x))) for x in wkv]
        _check(self.lib.oracle_attn_sharded(T, d, len(wq), wq.ctypes.data_as(ctypes.c_void_p),
                                            wkv.ctypes.data_as(ctypes.c_void_p), _ptr(X), _ptrs(WQ_i), _ptrs(WK_i),
                                            _ptrs(WV_i), _ptrs(O_i), _ptrs(WO_i), _ptr(dZ), _ptrs(dQ_i), _ptrs(dK_i),
                                            _ptrs(dV_i), _ptr(Z), _ptr(dX), _ptrs(dWO_i), _ptrs(dWQ_i), _ptrs(dWK_i),
                                            _ptrs(dWV_i)), "oracle_attn_sharded")
        return {"Z": Z, "dX": dX, "dWO_i": dWO_i, "dWQ_i": dWQ_i, "dWK_i": dWK_i, "dWV_i": dWV_i}

    def db2(self, dY):
        """Column sums of dY over tokens (gradient of the bias added after the g-sum)."""
        dY = _f64(dY)
        out = np.empty(dY.shape[1])
        _check(self.lib.oracle_db2(dY.shape[0], dY.shape[1], _ptr(dY), _ptr(out)), "oracle_db2")
        return out

    def wgrad_units(self, X, W1, W2, dY, units, act="gelu", W3=None, b1=None, b3=None, with_bias_grads=False):
        """dW1[:, j], dW3[:, j], dW2[j, :] for the listed hidden units j.

        Returns (dW1_cols, dW3_cols or None, dW2_rows), each [len(units) x d], and with
        with_bias_grads also (db1_units, db3_units or None), each [len(units)]."""
        lib = self.lib
        a = _act(act)
        X, W1, W2, W3, dY = _f64(X), _f64(W1), _f64(W2), _f64(W3), _f64(dY)
        b1, b3 = _f64(b1), _f64(b3)
        T, d = X.shape
        dff = W1.shape[1]
        u = np.ascontiguousarray(units, dtype=np.int64)
        c1 = np.empty((len(u), d)); c2 = np.empty((len(u), d))
        c3 = np.empty((len(u), d)) if a == ACT_SWIGLU else None
        g1 = np.empty(len(u))
        g3 = np.empty(len(u)) if a == ACT_SWIGLU else None
        _check(lib.oracle_wgrad_units(T, d, dff, a, _ptr(X), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(b1), _ptr(b3), _ptr(dY),
                                      len(u), _ptr(u), _ptr(c1), _ptr(c3), _ptr(c2), _ptr(g1), _ptr(g3)),
               "oracle_wgrad_units")
        if with_bias_grads:
            return c1, c3, c2, g1, g3
        return c1, c3, c2


_default = None


def default() -> COracle:
    global _default
    if _default is None:
        _default = COracle(_load())
    return _default


def num_threads(*args, **kwargs):
    return default().num_threads(*args, **kwargs)


def act_value(*args, **kwargs):
    return default().act_value(*args, **kwargs)


def act_grad(*args, **kwargs):
    return default().act_grad(*args, **kwargs)


def forward(*args, **kwargs):
    return default().forward(*args, **kwargs)


def backward(*args, **kwargs):
    return default().backward(*args, **kwargs)


def forward_sharded(*args, **kwargs):
    return default().forward_sharded(*args, **kwargs)


def backward_sharded(*args, **kwargs):
    return default().backward_sharded(*args, **kwargs)


def rows(*args, **kwargs):
    return default().rows(*args, **kwargs)


def forward_sp(*args, **kwargs):
    return default().forward_sp(*args, **kwargs)


def backward_sp(*args, **kwargs):
    return default().backward_sp(*args, **kwargs)


def wgrad_units(*args, **kwargs):
    return default().wgrad_units(*args, **kwargs)


def db2(*args, **kwargs):
    return default().db2(*args, **kwargs)


def attn_forward(*args, **kwargs):
    return default().attn_forward(*args, **kwargs)


def attn_backward(*args, **kwargs):
    return default().attn_backward(*args, **kwargs)


def attn_sharded(*args, **kwargs):
    return default().attn_sharded(*args, **kwargs)


num_threads.__doc__ = "OpenMP threads the C oracle uses."
