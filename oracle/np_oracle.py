"""Second, independent fp64 oracle written with numpy matrix products.

TEST INFRASTRUCTURE ONLY (same rule as the package docstring): it exists so
that the C oracle can be cross-checked on small shapes by code that shares
nothing with it -- numpy's own matmul instead of the C loops, and the
standard normal CDF from scipy.special.ndtr (Cephes) instead of libm's erf.

Block definition: "Parallelism" tag page of Jiang Yi's homepage, post
"megatron-lm", Method / FFN (Y = GeLU(X W1) W2 and the SwiGLU form
Y = (X W3 . Swish(X W1)) W2); GeLU is the erf form used by F.gelu in
Megatron_FeedForward ("Tensor parallelism", brunomaga.github.io).
"""
from __future__ import annotations

import numpy as np
from scipy.special import ndtr


def _phi(a):
    return np.exp(-0.5 * a * a) / np.sqrt(2.0 * np.pi)


def _sig(g):
    return 1.0 / (1.0 + np.exp(-g))


def _vec(b, n):
    return np.zeros(n) if b is None else np.asarray(b, dtype=np.float64)


def forward(X, W1, W2, act="gelu", W3=None, b1=None, b3=None, b2=None):
    X, W1, W2 = (np.asarray(m, dtype=np.float64) for m in (X, W1, W2))
    A = X @ W1 + _vec(b1, W1.shape[1])
    if act == "swiglu":
        U = X @ np.asarray(W3, dtype=np.float64) + _vec(b3, W1.shape[1])
        H = U * (A * _sig(A))
    else:
        U = None
        H = A * ndtr(A)
    return {"A": A, "U": U, "H": H, "Y": H @ W2 + _vec(b2, W2.shape[1])}


def backward(X, W1, W2, dY, act="gelu", W3=None, b1=None, b3=None, b2=None):
    X, W1, W2, dY = (np.asarray(m, dtype=np.float64) for m in (X, W1, W2, dY))
    f = forward(X, W1, W2, act, W3, b1, b3, b2)
    A, U, H = f["A"], f["U"], f["H"]
    dH = dY @ W2.T
    out = {"dW2": H.T @ dY, "db2": dY.sum(axis=0)}
    if act == "swiglu":
        W3 = np.asarray(W3, dtype=np.float64)
        s = _sig(A)
        dU = dH * (A * s)
        dG = dH * U * (s * (1.0 + A * (1.0 - s)))
        out.update(dW1=X.T @ dG, dW3=X.T @ dU, dX=dG @ W1.T + dU @ W3.T, dA=dG, dU=dU, db1=dG.sum(axis=0),
                   db3=dU.sum(axis=0))
    else:
        dA = dH * (ndtr(A) + A * _phi(A))
        out.update(dW1=X.T @ dA, dW3=None, dX=dA @ W1.T, dA=dA, dU=None, db1=dA.sum(axis=0), db3=None)
    return out


def attn_forward(X, WQ, WK, WV, O, WO):
    X, WQ, WK, WV, O, WO = (np.asarray(m, dtype=np.float64) for m in (X, WQ, WK, WV, O, WO))
    return {"Q": X @ WQ, "K": X @ WK, "V": X @ WV, "Z": O @ WO}


def attn_backward(X, WQ, WK, WV, O, WO, dZ, dQ, dK, dV):
    X, WQ, WK, WV, O, WO, dZ, dQ, dK, dV = (np.asarray(m, dtype=np.float64)
                                            for m in (X, WQ, WK, WV, O, WO, dZ, dQ, dK, dV))
    return {"dO": dZ @ WO.T, "dWO": O.T @ dZ, "dX": dQ @ WQ.T + dK @ WK.T + dV @ WV.T, "dWQ": X.T @ dQ,
            "dWK": X.T @ dK, "dWV": X.T @ dV}
