"""Python binding of libtpmlp: the t-sharded Megatron tensor-parallel MLP block
on one GB300.

The functions named ``tpmlp_*`` mirror the C ABI of ``include/tpmlp.h`` one to
one: they only marshal arguments (torch CUDA tensors or raw device pointers,
lists of per-shard tensors) and raise :class:`TpmlpError` on a non-OK status.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback, and :func:`load` raises if the library is missing.

``ShardedMLP`` is a small convenience layer that allocates the outputs with
PyTorch (device memory and streams are all PyTorch provides here) and
``TPMLPFunction`` wraps forward/backward as a ``torch.autograd.Function``.
``ShardedAttentionProj`` does the same for the attention block's QKV and
output projections (``tpmlp_attn_*``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional, Sequence

from . import _build

__all__ = [
    "TpmlpError", "load", "Plan", "tpmlp_plan_create", "tpmlp_plan_destroy", "tpmlp_workspace_size",
    "tpmlp_plan_set_timeout", "tpmlp_plan_set_stall_injection", "tpmlp_plan_set_stream_k",
    "STREAM_K_OFF", "STREAM_K_AUTO", "STREAM_K_ALWAYS", "STREAM_K_BALANCE",
    "tpmlp_forward", "tpmlp_backward", "tpmlp_backward_recompute", "tpmlp_forward_column", "tpmlp_forward_row", "tpmlp_forward_row_noalloc", "tpmlp_backward_dgrad",
    "tpmlp_backward_fsum", "tpmlp_check", "tpmlp_status_string", "tpmlp_last_cuda_error", "tpmlp_version",
    "tpmlp_last_launch_count", "tpmlp_last_error", "ShardedMLP", "TPMLPFunction", "EXPORTED_SYMBOLS",
    "AttnPlan", "tpmlp_attn_plan_create", "tpmlp_attn_qkv_forward", "tpmlp_attn_out_forward",
    "tpmlp_attn_out_backward", "tpmlp_attn_qkv_backward", "ShardedAttentionProj",
    "tpmlp_plan_set_sequence_stripes", "tpmlp_forward_sp", "tpmlp_backward_sp", "tpmlp_last_split_tiles",
    "LAUNCH_FWD_COLUMN", "LAUNCH_FWD_ROW", "LAUNCH_BWD_DGRAD", "LAUNCH_BWD_FSUM", "tpmlp_eval_activation",
    "ACT_EVAL",
]

ACT = {"gelu": 0, "swiglu": 1}
DTYPE = {"bf16": 0, "fp32": 1}
STATUS = {0: "TPMLP_OK", 1: "TPMLP_ERR_INVALID_ARG", 2: "TPMLP_ERR_SHAPE", 3: "TPMLP_ERR_ALIGNMENT",
          4: "TPMLP_ERR_UNSUPPORTED", 5: "TPMLP_ERR_CUDA", 6: "TPMLP_ERR_DEVICE_TIMEOUT",
          7: "TPMLP_ERR_NOT_IMPLEMENTED"}
MAX_SHARDS = 16

EXPORTED_SYMBOLS = (
    "tpmlp_plan_create", "tpmlp_plan_destroy", "tpmlp_workspace_size", "tpmlp_forward", "tpmlp_backward",
    "tpmlp_forward_column", "tpmlp_forward_row", "tpmlp_forward_row_noalloc", "tpmlp_backward_dgrad",
    "tpmlp_backward_fsum", "tpmlp_check", "tpmlp_status_string", "tpmlp_last_cuda_error", "tpmlp_version",
    "tpmlp_last_launch_count", "tpmlp_last_error", "tpmlp_plan_set_timeout", "tpmlp_plan_set_stall_injection",
    "tpmlp_backward_recompute", "tpmlp_attn_plan_create", "tpmlp_attn_qkv_forward", "tpmlp_attn_out_forward",
    "tpmlp_attn_out_backward", "tpmlp_attn_qkv_backward", "tpmlp_plan_set_sequence_stripes", "tpmlp_forward_sp",
    "tpmlp_backward_sp", "tpmlp_plan_set_stream_k", "tpmlp_last_split_tiles", "tpmlp_eval_activation",
)

# forms of tpmlp_eval_activation
ACT_EVAL = {"gelu": 0, "gelu_bwd": 1, "gelu_bwd_h": 2, "swiglu": 3, "swiglu_bwd": 4, "swiglu_bwd_h": 5,
            "fp32_gelu": 6, "fp32_swiglu": 7}

# launch kinds of tpmlp_last_split_tiles
LAUNCH_FWD_COLUMN, LAUNCH_FWD_ROW, LAUNCH_BWD_DGRAD, LAUNCH_BWD_FSUM = 0, 1, 2, 3


class TpmlpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        name = STATUS.get(self.status, f"status {status}")
        extra = ""
        if _lib is not None:
            msg = _lib.tpmlp_last_error()
            if msg:
                extra = f": {msg.decode(errors='replace')}"
        super().__init__(f"{where}: {name}{extra}")


class _Desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("t", ctypes.c_int32),
                ("d_i", ctypes.POINTER(ctypes.c_int64)), ("act", ctypes.c_int), ("dtype", ctypes.c_int)]


class _AttnDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("t", ctypes.c_int32),
                ("dq_i", ctypes.POINTER(ctypes.c_int64)), ("dkv_i", ctypes.POINTER(ctypes.c_int64)),
                ("dtype", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load():
    """Load libtpmlp.so (built by ``__graft_entry__.build()`` / ``_build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        vp, pp, i32, st = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int
        lib.tpmlp_plan_create.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(vp)]
        lib.tpmlp_plan_create.restype = st
        lib.tpmlp_plan_destroy.argtypes = [vp]
        lib.tpmlp_plan_destroy.restype = None
        lib.tpmlp_plan_set_timeout.argtypes = [vp, ctypes.c_uint32]
        lib.tpmlp_plan_set_timeout.restype = st
        lib.tpmlp_plan_set_stall_injection.argtypes = [vp, ctypes.c_int]
        lib.tpmlp_plan_set_stall_injection.restype = st
        lib.tpmlp_plan_set_stream_k.argtypes = [vp, ctypes.c_int]
        lib.tpmlp_plan_set_stream_k.restype = st
        lib.tpmlp_workspace_size.argtypes = [vp]
        lib.tpmlp_workspace_size.restype = ctypes.c_size_t
        lib.tpmlp_forward.argtypes = [vp, vp, pp, pp, pp, pp, pp, vp, vp, pp, pp, vp, vp]
        lib.tpmlp_forward.restype = st
        lib.tpmlp_backward.argtypes = [vp, vp, pp, pp, pp, pp, pp, vp, pp, vp, pp, pp, pp, pp, pp, vp, vp, vp]
        lib.tpmlp_backward.restype = st
        lib.tpmlp_backward_recompute.argtypes = [vp, vp, pp, pp, pp, pp, pp, vp, pp, vp, pp, pp, pp, pp, pp, vp, vp,
                                                 vp]
        lib.tpmlp_backward_recompute.restype = st
        lib.tpmlp_forward_column.argtypes = [vp, vp, pp, pp, pp, pp, pp, pp, vp, vp]
        lib.tpmlp_forward_column.restype = st
        lib.tpmlp_forward_row.argtypes = [vp, pp, vp, pp, vp, vp, vp]
        lib.tpmlp_forward_row.restype = st
        lib.tpmlp_forward_row_noalloc.argtypes = [vp, pp, pp, vp, vp]
        lib.tpmlp_forward_row_noalloc.restype = st
        lib.tpmlp_backward_dgrad.argtypes = [vp, pp, pp, pp, vp, pp, pp, vp, vp, vp]
        lib.tpmlp_backward_dgrad.restype = st
        lib.tpmlp_backward_fsum.argtypes = [vp, vp, pp, pp, pp, vp, pp, pp, pp, pp, vp, vp]
        lib.tpmlp_backward_fsum.restype = st
        lib.tpmlp_attn_plan_create.argtypes = [ctypes.POINTER(_AttnDesc), ctypes.POINTER(vp)]
        lib.tpmlp_attn_plan_create.restype = st
        lib.tpmlp_attn_qkv_forward.argtypes = [vp, vp, pp, pp, vp, vp]
        lib.tpmlp_attn_qkv_forward.restype = st
        lib.tpmlp_attn_out_forward.argtypes = [vp, pp, pp, vp, vp, vp]
        lib.tpmlp_attn_out_forward.restype = st
        lib.tpmlp_attn_out_backward.argtypes = [vp, pp, pp, vp, pp, pp, vp, vp]
        lib.tpmlp_attn_out_backward.restype = st
        lib.tpmlp_attn_qkv_backward.argtypes = [vp, vp, pp, pp, vp, pp, vp, vp]
        lib.tpmlp_attn_qkv_backward.restype = st
        lib.tpmlp_plan_set_sequence_stripes.argtypes = [vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64)]
        lib.tpmlp_plan_set_sequence_stripes.restype = st
        lib.tpmlp_forward_sp.argtypes = [vp, pp, pp, pp, pp, pp, pp, vp, pp, pp, pp, vp, vp]
        lib.tpmlp_forward_sp.restype = st
        lib.tpmlp_backward_sp.argtypes = [vp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, pp, vp, vp, vp]
        lib.tpmlp_backward_sp.restype = st
        lib.tpmlp_check.argtypes = [vp, vp, vp]
        lib.tpmlp_check.restype = st
        lib.tpmlp_status_string.argtypes = [i32]
        lib.tpmlp_status_string.restype = ctypes.c_char_p
        lib.tpmlp_last_error.argtypes = []
        lib.tpmlp_last_error.restype = ctypes.c_char_p
        lib.tpmlp_last_cuda_error.argtypes = []
        lib.tpmlp_last_cuda_error.restype = i32
        lib.tpmlp_version.argtypes = []
        lib.tpmlp_version.restype = i32
        lib.tpmlp_last_launch_count.argtypes = []
        lib.tpmlp_last_launch_count.restype = i32
        lib.tpmlp_last_split_tiles.argtypes = [i32, ctypes.POINTER(ctypes.c_int64), i32]
        lib.tpmlp_last_split_tiles.restype = i32
        lib.tpmlp_eval_activation.argtypes = [i32, vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp]
        lib.tpmlp_eval_activation.restype = st
        _lib = lib
        return lib


# ---------------------------------------------------------------- marshalling

def _addr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if x.numel() and not x.is_cuda:
            raise ValueError("tensor must live on a CUDA device")
        if x.numel() and not x.is_contiguous():
            raise ValueError("tensor must be contiguous (row-major)")
        return x.data_ptr() or None
    raise TypeError(f"expected a tensor or an int device pointer, got {type(x)}")


def _arr(xs) -> Optional[ctypes.Array]:
    if xs is None:
        return None
    return (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream or None
        except Exception:  # no torch CUDA: legacy default stream
            return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _ok(status: int, where: str):
    if status != 0:
        raise TpmlpError(status, where)


class Plan:
    """Owns a ``tpmlp_plan*`` (host memory only)."""

    def __init__(self, T: int, d: int, d_i: Sequence[int], act: str = "gelu", dtype: str = "bf16"):
        lib = load()
        self.T, self.d, self.d_i = int(T), int(d), tuple(int(v) for v in d_i)
        self.t = len(self.d_i)
        self.act, self.dtype = act, dtype
        self._d_i = (ctypes.c_int64 * max(1, self.t))(*self.d_i)
        desc = _Desc(self.T, self.d, self.t, ctypes.cast(self._d_i, ctypes.POINTER(ctypes.c_int64)),
                     ACT[act] if isinstance(act, str) else int(act),
                     DTYPE[dtype] if isinstance(dtype, str) else int(dtype))
        h = ctypes.c_void_p()
        _ok(lib.tpmlp_plan_create(ctypes.byref(desc), ctypes.byref(h)), "tpmlp_plan_create")
        self.handle = h
        self.stripe_rows = ()  # sequence-parallel token stripes (tpmlp_plan_set_sequence_stripes)

    @property
    def dff(self) -> int:
        return sum(self.d_i)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.tpmlp_plan_destroy(h)
            self.handle = None


def tpmlp_plan_create(T, d, d_i, act="gelu", dtype="bf16") -> Plan:
    return Plan(T, d, d_i, act, dtype)


def tpmlp_plan_destroy(plan: Plan):
    if plan.handle is not None and plan.handle.value:
        load().tpmlp_plan_destroy(plan.handle)
        plan.handle = None


class AttnPlan(Plan):
    """Owns an attention ``tpmlp_plan*``: per-shard query widths dq_i and
    key/value widths dkv_i (fused QKV width n_i = dq_i + 2 dkv_i)."""

    def __init__(self, T: int, d: int, dq_i: Sequence[int], dkv_i: Sequence[int], dtype: str = "bf16"):
        lib = load()
        self.T, self.d = int(T), int(d)
        self.dq_i, self.dkv_i = tuple(int(v) for v in dq_i), tuple(int(v) for v in dkv_i)
        if len(self.dq_i) != len(self.dkv_i):
            raise ValueError("dq_i and dkv_i must have one entry per shard")
        self.t = len(self.dq_i)
        self.d_i = tuple(q + 2 * kv for q, kv in zip(self.dq_i, self.dkv_i))
        self.act, self.dtype = None, dtype
        self._dq = (ctypes.c_int64 * max(1, self.t))(*self.dq_i)
        self._dkv = (ctypes.c_int64 * max(1, self.t))(*self.dkv_i)
        desc = _AttnDesc(self.T, self.d, self.t, ctypes.cast(self._dq, ctypes.POINTER(ctypes.c_int64)),
                         ctypes.cast(self._dkv, ctypes.POINTER(ctypes.c_int64)),
                         DTYPE[dtype] if isinstance(dtype, str) else int(dtype))
        h = ctypes.c_void_p()
        _ok(lib.tpmlp_attn_plan_create(ctypes.byref(desc), ctypes.byref(h)), "tpmlp_attn_plan_create")
        self.handle = h


def tpmlp_attn_plan_create(T, d, dq_i, dkv_i, dtype="bf16") -> AttnPlan:
    return AttnPlan(T, d, dq_i, dkv_i, dtype)


def tpmlp_attn_qkv_forward(plan, X, Wqkv, QKV, workspace, stream=None):
    _ok(load().tpmlp_attn_qkv_forward(plan.handle, _addr(X), _arr(Wqkv), _arr(QKV), _addr(workspace),
                                      _stream(stream)), "tpmlp_attn_qkv_forward")


def tpmlp_attn_out_forward(plan, WO, O, Z, workspace, stream=None):
    _ok(load().tpmlp_attn_out_forward(plan.handle, _arr(WO), _arr(O), _addr(Z), _addr(workspace), _stream(stream)),
        "tpmlp_attn_out_forward")


def tpmlp_attn_out_backward(plan, WO, O, dZ, dO, dWO, workspace, stream=None):
    _ok(load().tpmlp_attn_out_backward(plan.handle, _arr(WO), _arr(O), _addr(dZ), _arr(dO), _arr(dWO),
                                       _addr(workspace), _stream(stream)), "tpmlp_attn_out_backward")


def tpmlp_attn_qkv_backward(plan, X, Wqkv, dQKV, dX, dWqkv, workspace, stream=None):
    _ok(load().tpmlp_attn_qkv_backward(plan.handle, _addr(X), _arr(Wqkv), _arr(dQKV), _addr(dX), _arr(dWqkv),
                                       _addr(workspace), _stream(stream)), "tpmlp_attn_qkv_backward")


def tpmlp_plan_set_sequence_stripes(plan: Plan, stripe_rows: Sequence[int]):
    rows = (ctypes.c_int64 * max(1, len(stripe_rows)))(*[int(r) for r in stripe_rows])
    _ok(load().tpmlp_plan_set_sequence_stripes(plan.handle, len(stripe_rows), rows),
        "tpmlp_plan_set_sequence_stripes")
    plan.stripe_rows = tuple(int(r) for r in stripe_rows)


def tpmlp_forward_sp(plan, X_stripes, W1, W3, W2, b1, b3, b2, Y_stripes, saved, H, workspace, stream=None):
    _ok(load().tpmlp_forward_sp(plan.handle, _arr(X_stripes), _arr(W1), _arr(W3), _arr(W2), _arr(b1), _arr(b3),
                                _addr(b2), _arr(Y_stripes), _arr(saved), _arr(H), _addr(workspace), _stream(stream)),
        "tpmlp_forward_sp")


def tpmlp_backward_sp(plan, X_stripes, W1, W3, W2, saved, H, dY_stripes, dact, dX_stripes, dW1, dW3, dW2, db1, db3,
                      db2, workspace, stream=None):
    _ok(load().tpmlp_backward_sp(plan.handle, _arr(X_stripes), _arr(W1), _arr(W3), _arr(W2), _arr(saved), _arr(H),
                                 _arr(dY_stripes), _arr(dact), _arr(dX_stripes), _arr(dW1), _arr(dW3), _arr(dW2),
                                 _arr(db1), _arr(db3), _addr(db2), _addr(workspace), _stream(stream)),
        "tpmlp_backward_sp")


def tpmlp_plan_set_timeout(plan: Plan, timeout_ms: int):
    _ok(load().tpmlp_plan_set_timeout(plan.handle, int(timeout_ms)), "tpmlp_plan_set_timeout")


def tpmlp_plan_set_stall_injection(plan: Plan, enable):
    """False / True (1): producers load nothing; 2: stream-K parts are never published."""
    mode = 2 if enable == 2 else (1 if enable else 0)
    _ok(load().tpmlp_plan_set_stall_injection(plan.handle, mode), "tpmlp_plan_set_stall_injection")


STREAM_K_OFF, STREAM_K_AUTO, STREAM_K_ALWAYS, STREAM_K_BALANCE = 0, 1, 2, 3


def tpmlp_plan_set_stream_k(plan: Plan, mode: int):
    """Stream-K tail of the bf16 launches: STREAM_K_AUTO (default), _ALWAYS or _OFF."""
    _ok(load().tpmlp_plan_set_stream_k(plan.handle, int(mode)), "tpmlp_plan_set_stream_k")


def tpmlp_workspace_size(plan: Plan) -> int:
    return int(load().tpmlp_workspace_size(plan.handle))


def tpmlp_forward(plan, X, W1, W3, W2, b1, b3, b2, Y, saved, H, workspace, stream=None):
    _ok(load().tpmlp_forward(plan.handle, _addr(X), _arr(W1), _arr(W3), _arr(W2), _arr(b1), _arr(b3), _addr(b2),
                             _addr(Y), _arr(saved), _arr(H), _addr(workspace), _stream(stream)), "tpmlp_forward")


def tpmlp_backward(plan, X, W1, W3, W2, saved, H, dY, dact, dX, dW1, dW3, dW2, db1, db3, db2, workspace,
                   stream=None):
    _ok(load().tpmlp_backward(plan.handle, _addr(X), _arr(W1), _arr(W3), _arr(W2), _arr(saved), _arr(H),
                              _addr(dY), _arr(dact), _addr(dX), _arr(dW1), _arr(dW3), _arr(dW2), _arr(db1),
                              _arr(db3), _addr(db2), _addr(workspace), _stream(stream)), "tpmlp_backward")


def tpmlp_backward_recompute(plan, X, W1, W3, W2, saved, H, dY, dact, dX, dW1, dW3, dW2, db1, db3, db2, workspace,
                             stream=None):
    _ok(load().tpmlp_backward_recompute(plan.handle, _addr(X), _arr(W1), _arr(W3), _arr(W2), _arr(saved), _arr(H),
                                        _addr(dY), _arr(dact), _addr(dX), _arr(dW1), _arr(dW3), _arr(dW2), _arr(db1),
                                        _arr(db3), _addr(db2), _addr(workspace), _stream(stream)),
        "tpmlp_backward_recompute")


def tpmlp_forward_column(plan, X, W1, W3, b1, b3, saved, H, workspace, stream=None):
    _ok(load().tpmlp_forward_column(plan.handle, _addr(X), _arr(W1), _arr(W3), _arr(b1), _arr(b3), _arr(saved),
                                    _arr(H), _addr(workspace), _stream(stream)), "tpmlp_forward_column")


def tpmlp_forward_row(plan, W2, b2, H, Y, workspace, stream=None):
    _ok(load().tpmlp_forward_row(plan.handle, _arr(W2), _addr(b2), _arr(H), _addr(Y), _addr(workspace),
                                 _stream(stream)), "tpmlp_forward_row")


def tpmlp_forward_row_noalloc(plan, W2, H, Y, stream=None):
    """Row-parallel GEMM (g-sum) without a workspace: the scratch status word
    is a library-owned static device array, for callers that cannot allocate
    device memory.  Blocks until its kernel has finished."""
    _ok(load().tpmlp_forward_row_noalloc(plan.handle, _arr(W2), _arr(H), _addr(Y), _stream(stream)),
        "tpmlp_forward_row_noalloc")


def tpmlp_backward_dgrad(plan, W2, saved, H, dY, dact, dW2, db2, workspace, stream=None):
    _ok(load().tpmlp_backward_dgrad(plan.handle, _arr(W2), _arr(saved), _arr(H), _addr(dY), _arr(dact), _arr(dW2),
                                    _addr(db2), _addr(workspace), _stream(stream)), "tpmlp_backward_dgrad")


def tpmlp_backward_fsum(plan, X, W1, W3, dact, dX, dW1, dW3, db1, db3, workspace, stream=None):
    _ok(load().tpmlp_backward_fsum(plan.handle, _addr(X), _arr(W1), _arr(W3), _arr(dact), _addr(dX), _arr(dW1),
                                   _arr(dW3), _arr(db1), _arr(db3), _addr(workspace), _stream(stream)),
        "tpmlp_backward_fsum")


def tpmlp_check(plan, workspace, stream=None):
    _ok(load().tpmlp_check(plan.handle, _addr(workspace), _stream(stream)), "tpmlp_check")


def tpmlp_status_string(status: int) -> str:
    return load().tpmlp_status_string(int(status)).decode()


def tpmlp_last_cuda_error() -> int:
    return int(load().tpmlp_last_cuda_error())


def tpmlp_last_error() -> str:
    return load().tpmlp_last_error().decode(errors="replace")


def tpmlp_version() -> int:
    return int(load().tpmlp_version())


def tpmlp_last_launch_count() -> int:
    return int(load().tpmlp_last_launch_count())


def tpmlp_eval_activation(form: str, x, y=None, dh=None, out0=None, out1=None, out2=None, stream=None):
    """The epilogues' activation forms on fp32 device tensors of n elements
    (form: a key of ACT_EVAL); outputs are caller tensors like x."""
    n = x.numel()
    _ok(load().tpmlp_eval_activation(ACT_EVAL[form], _addr(x), _addr(y), _addr(dh), _addr(out0), _addr(out1),
                                     _addr(out2), n, _stream(stream)), "tpmlp_eval_activation")


def tpmlp_last_split_tiles(launch_kind: int) -> List[tuple]:
    """(problem, first row, first column, address of the problem's first output)
    of every tile the stream-K schedule split in the last launch of this kind on
    the calling thread."""
    lib = load()
    n = int(lib.tpmlp_last_split_tiles(int(launch_kind), None, 0))
    if n < 0:
        raise ValueError(f"unknown launch kind {launch_kind}")
    buf = (ctypes.c_int64 * max(1, 4 * n))()
    lib.tpmlp_last_split_tiles(int(launch_kind), buf, n)
    return [tuple(int(buf[4 * i + k]) for k in range(4)) for i in range(n)]


# ---------------------------------------------------------------- convenience layer

class ShardedMLP:
    """Plan + workspace + output allocation for one problem shape.

    Tensors follow the C ABI: X [T, d]; W1_i, W3_i [d, d_i]; W2_i [d_i, d];
    every tensor contiguous on the current CUDA device, in the plan's dtype.
    """

    def __init__(self, T: int, d: int, d_i: Sequence[int], act: str = "gelu", dtype: str = "bf16", device=None):
        import torch
        self.plan = Plan(T, d, d_i, act, dtype)
        self.device = torch.device(device or "cuda")
        self.tdtype = {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]
        self.workspace = torch.zeros(tpmlp_workspace_size(self.plan), dtype=torch.uint8, device=self.device)

    @property
    def swiglu(self) -> bool:
        return self.plan.act == "swiglu"

    def _empty(self, *shape):
        import torch
        return torch.empty(*shape, dtype=self.tdtype, device=self.device)

    def check_inputs(self, X, W1_i, W2_i, W3_i=None):
        p = self.plan
        assert tuple(X.shape) == (p.T, p.d), f"X shape {tuple(X.shape)} != {(p.T, p.d)}"
        assert len(W1_i) == p.t and len(W2_i) == p.t
        for i, w in enumerate(p.d_i):
            assert tuple(W1_i[i].shape) == (p.d, w) and tuple(W2_i[i].shape) == (w, p.d)
            if self.swiglu:
                assert tuple(W3_i[i].shape) == (p.d, w)
        for x in [X, *W1_i, *W2_i, *(W3_i or [])]:
            assert x.dtype == self.tdtype and x.is_cuda

    def alloc_forward(self):
        p = self.plan
        Y = self._empty(p.T, p.d)
        H = [self._empty(p.T, w) for w in p.d_i]
        saved = [self._empty(p.T, w) for w in p.d_i * (2 if self.swiglu else 1)]
        return Y, saved, H

    def alloc_backward(self):
        p = self.plan
        dX = self._empty(p.T, p.d)
        dact = [self._empty(p.T, w) for w in p.d_i * (2 if self.swiglu else 1)]
        dW1 = [self._empty(p.d, w) for w in p.d_i]
        dW3 = [self._empty(p.d, w) for w in p.d_i] if self.swiglu else None
        dW2 = [self._empty(w, p.d) for w in p.d_i]
        return dact, dX, dW1, dW3, dW2

    def forward(self, X, W1_i, W2_i, W3_i=None, out=None, stream=None, b1_i=None, b3_i=None, b2=None):
        """Y = sum_i act(X W1_i + b1_i) W2_i + b2 (biases optional).  Returns (Y, saved, H)."""
        self.check_inputs(X, W1_i, W2_i, W3_i)
        Y, saved, H = out if out is not None else self.alloc_forward()
        tpmlp_forward(self.plan, X, W1_i, W3_i, W2_i, b1_i, b3_i, b2, Y, saved, H, self.workspace, stream)
        return Y, saved, H

    def alloc_bias_grads(self):
        p = self.plan
        db1 = [self._empty(w) for w in p.d_i]
        db3 = [self._empty(w) for w in p.d_i] if self.swiglu else None
        return db1, db3, self._empty(p.d)

    def backward(self, X, W1_i, W2_i, saved, H, dY, W3_i=None, out=None, stream=None, bias_grads=False,
                 recompute=False):
        """Gradients of X, the weights and, with bias_grads, the biases.  With
        recompute, H is scratch (its contents are not read) and is rewritten."""
        dact, dX, dW1, dW3, dW2 = out if out is not None else self.alloc_backward()
        db1, db3, db2 = self.alloc_bias_grads() if bias_grads else (None, None, None)
        fn = tpmlp_backward_recompute if recompute else tpmlp_backward
        fn(self.plan, X, W1_i, W3_i, W2_i, saved, H, dY, dact, dX, dW1, dW3, dW2, db1, db3, db2, self.workspace,
           stream)
        return {"dX": dX, "dW1": dW1, "dW3": dW3, "dW2": dW2, "dact": dact, "db1": db1, "db3": db3, "db2": db2}

    def check(self, stream=None):
        tpmlp_check(self.plan, self.workspace, stream)

    # ---- sequence-parallel layout: X, dY in and Y, dX out as token stripes
    def set_sequence_stripes(self, stripe_rows: Sequence[int]):
        tpmlp_plan_set_sequence_stripes(self.plan, stripe_rows)

    def alloc_stripes(self):
        return [self._empty(r, self.plan.d) for r in self.plan.stripe_rows]

    def forward_sp(self, X_stripes, W1_i, W2_i, W3_i=None, stream=None, b1_i=None, b3_i=None, b2=None):
        """Y stripes = reduce-scatter of sum_i act(X W1_i + b1_i) W2_i (+ b2), X gathered from its stripes.
        Returns (Y_stripes, saved, H)."""
        Y_j = self.alloc_stripes()
        _, saved, H = self.alloc_forward()
        tpmlp_forward_sp(self.plan, X_stripes, W1_i, W3_i, W2_i, b1_i, b3_i, b2, Y_j, saved, H, self.workspace,
                         stream)
        return Y_j, saved, H

    def backward_sp(self, X_stripes, W1_i, W2_i, saved, H, dY_stripes, W3_i=None, stream=None, bias_grads=False):
        dact, _, dW1, dW3, dW2 = self.alloc_backward()
        dX_j = self.alloc_stripes()
        db1, db3, db2 = self.alloc_bias_grads() if bias_grads else (None, None, None)
        tpmlp_backward_sp(self.plan, X_stripes, W1_i, W3_i, W2_i, saved, H, dY_stripes, dact, dX_j, dW1, dW3, dW2,
                          db1, db3, db2, self.workspace, stream)
        return {"dX_stripes": dX_j, "dW1": dW1, "dW3": dW3, "dW2": dW2, "dact": dact, "db1": db1, "db3": db3,
                "db2": db2}


class ShardedAttentionProj:
    """Attention plan + workspace + output allocation for one shape.

    Tensors follow the C ABI: X [T, d]; Wqkv_i [d, n_i] = [WQ_i | WK_i | WV_i];
    QKV_i [T, n_i]; O_i [T, dq_i]; WO_i [dq_i, d]; Z [T, d].
    """

    def __init__(self, T: int, d: int, dq_i: Sequence[int], dkv_i: Sequence[int], dtype: str = "bf16",
                 device=None):
        import torch
        self.plan = AttnPlan(T, d, dq_i, dkv_i, dtype)
        self.device = torch.device(device or "cuda")
        self.tdtype = {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]
        self.workspace = torch.zeros(tpmlp_workspace_size(self.plan), dtype=torch.uint8, device=self.device)

    def _empty(self, *shape):
        import torch
        return torch.empty(*shape, dtype=self.tdtype, device=self.device)

    def qkv_forward(self, X, Wqkv_i, out=None, stream=None):
        p = self.plan
        QKV = out if out is not None else [self._empty(p.T, n) for n in p.d_i]
        tpmlp_attn_qkv_forward(p, X, Wqkv_i, QKV, self.workspace, stream)
        return QKV

    def out_forward(self, WO_i, O_i, out=None, stream=None):
        Z = out if out is not None else self._empty(self.plan.T, self.plan.d)
        tpmlp_attn_out_forward(self.plan, WO_i, O_i, Z, self.workspace, stream)
        return Z

    def out_backward(self, WO_i, O_i, dZ, out=None, stream=None):
        p = self.plan
        dO, dWO = out if out is not None else ([self._empty(p.T, q) for q in p.dq_i],
                                               [self._empty(q, p.d) for q in p.dq_i])
        tpmlp_attn_out_backward(p, WO_i, O_i, dZ, dO, dWO, self.workspace, stream)
        return dO, dWO

    def qkv_backward(self, X, Wqkv_i, dQKV_i, out=None, stream=None):
        p = self.plan
        dX, dWqkv = out if out is not None else (self._empty(p.T, p.d), [self._empty(p.d, n) for n in p.d_i])
        tpmlp_attn_qkv_backward(p, X, Wqkv_i, dQKV_i, dX, dWqkv, self.workspace, stream)
        return dX, dWqkv

    def check(self, stream=None):
        tpmlp_check(self.plan, self.workspace, stream)


def _make_function():
    import torch

    class TPMLPFunction(torch.autograd.Function):
        """Y = TPMLPFunction.apply(mlp, X, *W1_i, *W2_i[, *W3_i]) with the library's backward."""

        @staticmethod
        def forward(ctx, mlp: ShardedMLP, X, *weights):
            t = mlp.plan.t
            W1_i, W2_i = list(weights[:t]), list(weights[t:2 * t])
            W3_i = list(weights[2 * t:3 * t]) if mlp.swiglu else None
            Y, saved, H = mlp.forward(X.contiguous(), W1_i, W2_i, W3_i)
            ctx.mlp = mlp
            ctx.save_for_backward(X, *weights, *saved, *H)
            return Y

        @staticmethod
        def backward(ctx, dY):
            mlp = ctx.mlp
            t = mlp.plan.t
            ns = 2 * t if mlp.swiglu else t
            tensors = ctx.saved_tensors
            X = tensors[0]
            nw = 3 * t if mlp.swiglu else 2 * t
            weights = list(tensors[1:1 + nw])
            saved = list(tensors[1 + nw:1 + nw + ns])
            H = list(tensors[1 + nw + ns:])
            W1_i, W2_i = weights[:t], weights[t:2 * t]
            W3_i = weights[2 * t:] if mlp.swiglu else None
            g = mlp.backward(X, W1_i, W2_i, saved, H, dY.contiguous(), W3_i)
            grads = g["dW1"] + g["dW2"] + (g["dW3"] if mlp.swiglu else [])
            return (None, g["dX"], *grads)

    return TPMLPFunction


class _LazyFunction:
    _fn = None

    def __getattr__(self, name):
        if _LazyFunction._fn is None:
            _LazyFunction._fn = _make_function()
        return getattr(_LazyFunction._fn, name)


TPMLPFunction = _LazyFunction()
