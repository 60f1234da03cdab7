"""CPU-only checks of the C ABI: the library loads, exports every function the
header declares, validates plans, and refuses to compute without a GPU (no
CPU fallback).  No kernel is launched here."""
import ctypes
import os
import re

import pytest
import torch

import megatron_tensor_transformer_column_gb300 as tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")
SK_WORKSPACE = 16384 + 160 * 256 * 256 * 4  # status block, stream-K ticket counters, 2 partial slots per range


@pytest.fixture(scope="module")
def lib():
    from megatron_tensor_transformer_column_gb300 import _build
    _build.build()
    return tp.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"TPMLP_API\s+[\w\s\*]*?\b(tpmlp_\w+)\s*\(", src)))


def test_header_declares_the_binding_names():
    names = declared_functions()
    assert len(names) >= 14
    assert set(names) == set(tp.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", tp.library_path()], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    ours = {s for s in syms if s.startswith("tpmlp")}
    assert ours == set(declared_functions())


def test_version_and_status_strings(lib):
    assert tp.tpmlp_version() == 105
    for code, name in tp.STATUS.items():
        assert tp.tpmlp_status_string(code) == name
    assert tp.tpmlp_status_string(99) == "TPMLP_ERR_UNKNOWN"


@pytest.mark.parametrize("args,status", [
    ((16, 64, [64], "gelu", "bf16"), 0),
    ((0, 64, [64, 128], "swiglu", "bf16"), 0),
    ((16, 64, [60], "gelu", "fp32"), 0),
    ((-1, 64, [64], "gelu", "bf16"), 2),
    ((16, 0, [64], "gelu", "bf16"), 2),
    ((16, 64, [], "gelu", "bf16"), 2),
    ((16, 64, [64, 0], "gelu", "bf16"), 2),
    ((16, 64, [8] * 17, "gelu", "bf16"), 2),
    ((16, 60, [64], "gelu", "bf16"), 3),
    ((16, 64, [60], "gelu", "bf16"), 3),
    ((16, 64, [62], "gelu", "fp32"), 3),
    ((16, 64, [64], 7, "bf16"), 1),
    ((16, 64, [64], "gelu", 9), 1),
    ((2 ** 31, 64, [64], "gelu", "bf16"), 4),
])
def test_plan_validation(lib, args, status):
    if status == 0:
        p = tp.Plan(*args)
        assert tp.tpmlp_workspace_size(p) == (SK_WORKSPACE if args[4] == "bf16" else 256)
    else:
        with pytest.raises(tp.TpmlpError) as e:
            tp.Plan(*args)
        assert e.value.status == status


def test_null_arguments_rejected(lib):
    h = ctypes.c_void_p()
    assert lib.tpmlp_plan_create(None, ctypes.byref(h)) == 1
    assert lib.tpmlp_workspace_size(None) == 0
    assert lib.tpmlp_forward(None, None, None, None, None, None, None, None, None, None, None, None, None) == 1
    lib.tpmlp_plan_destroy(None)  # no-op


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_no_cpu_fallback_without_gpu(lib):
    """Without a device the compute entry points fail loudly instead of computing on the CPU."""
    p = tp.Plan(16, 64, [64], "gelu", "bf16")
    fake = 1 << 20  # never dereferenced: the device query fails first
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(p, fake, [fake], None, [fake], None, None, None, fake, [fake], [fake], fake, stream=0)
    assert e.value.status in (4, 5)


@pytest.mark.parametrize("args,status", [
    ((16, 64, [64], [64], "bf16"), 0),
    ((0, 64, [128, 64], [16, 8], "bf16"), 0),
    ((16, 64, [12], [4], "fp32"), 0),
    ((-1, 64, [64], [64], "bf16"), 2),
    ((16, 0, [64], [64], "bf16"), 2),
    ((16, 64, [], [], "bf16"), 2),
    ((16, 64, [64, 0], [8, 8], "bf16"), 2),
    ((16, 64, [64], [0], "bf16"), 2),
    ((16, 64, [8] * 17, [8] * 17, "bf16"), 2),
    ((16, 60, [64], [64], "bf16"), 3),
    ((16, 64, [64], [12], "bf16"), 3),
    ((16, 64, [60], [64], "bf16"), 3),
    ((16, 64, [64], [64], 9), 1),
    ((2 ** 31, 64, [64], [64], "bf16"), 4),
])
def test_attn_plan_validation(lib, args, status):
    if status == 0:
        p = tp.AttnPlan(*args)
        assert tp.tpmlp_workspace_size(p) == (SK_WORKSPACE if args[4] == "bf16" else 256)
        assert p.d_i == tuple(q + 2 * kv for q, kv in zip(args[2], args[3]))
    else:
        with pytest.raises(tp.TpmlpError) as e:
            tp.AttnPlan(*args)
        assert e.value.status == status


def test_plan_kinds_are_not_interchangeable(lib):
    """An attention plan is refused by the MLP entry points and the reverse,
    before any device query."""
    ap = tp.AttnPlan(16, 64, [64], [64])
    mp = tp.Plan(16, 64, [64], "gelu", "bf16")
    fake = 1 << 20  # never dereferenced: the plan kind is checked first
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward(ap, fake, [fake], None, [fake], None, None, None, fake, [fake], [fake], fake, stream=0)
    assert e.value.status == 1 and "attention plan" in str(e.value)
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward_row_noalloc(ap, [fake], [fake], fake, stream=0)
    assert e.value.status == 1
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_attn_qkv_forward(mp, fake, [fake], [fake], fake, stream=0)
    assert e.value.status == 1 and "MLP plan" in str(e.value)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_attn_no_cpu_fallback_without_gpu(lib):
    p = tp.AttnPlan(16, 64, [64], [64])
    fake = 1 << 20
    for call in (lambda: tp.tpmlp_attn_qkv_forward(p, fake, [fake], [fake], fake, stream=0),
                 lambda: tp.tpmlp_attn_out_forward(p, [fake], [fake], fake, fake, stream=0),
                 lambda: tp.tpmlp_attn_out_backward(p, [fake], [fake], fake, [fake], [fake], fake, stream=0),
                 lambda: tp.tpmlp_attn_qkv_backward(p, fake, [fake], [fake], fake, [fake], fake, stream=0)):
        with pytest.raises(tp.TpmlpError) as e:
            call()
        assert e.value.status in (4, 5)


@pytest.mark.parametrize("T,rows,status", [
    (1000, [1000], 0),
    (1000, [256, 744], 0),
    (1000, [128, 0, 384, 488], 0),
    (0, [0, 0], 0),
    (1000, [500, 500], 3),     # the second stripe starts at 500, not a multiple of 128
    (1000, [256, 700], 2),     # rows do not add up to T
    (1000, [256, -1, 745], 2),
    (1000, [], 2),
    (1000, [64] * 17, 2),
])
def test_sequence_stripe_validation(lib, T, rows, status):
    p = tp.Plan(T, 64, [64], "gelu", "bf16")
    if status == 0:
        tp.tpmlp_plan_set_sequence_stripes(p, rows)
        assert p.stripe_rows == tuple(rows)
    else:
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_plan_set_sequence_stripes(p, rows)
        assert e.value.status == status


def test_sequence_stripes_refused_on_attention_plans(lib):
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_plan_set_sequence_stripes(tp.AttnPlan(256, 64, [64], [64]), [256])
    assert e.value.status == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_sp_no_cpu_fallback_without_gpu(lib):
    p = tp.Plan(256, 64, [64], "gelu", "bf16")
    tp.tpmlp_plan_set_sequence_stripes(p, [128, 128])
    fake = 1 << 20
    with pytest.raises(tp.TpmlpError) as e:
        tp.tpmlp_forward_sp(p, [fake, fake], [fake], None, [fake], None, None, None, [fake, fake], [fake], [fake],
                            fake, stream=0)
    assert e.value.status in (4, 5)


def test_stream_k_mode_validation(lib):
    p = tp.Plan(512, 64, [64], "gelu", "bf16")
    for mode in (tp.STREAM_K_OFF, tp.STREAM_K_ALWAYS, tp.STREAM_K_AUTO, tp.STREAM_K_BALANCE):
        tp.tpmlp_plan_set_stream_k(p, mode)
    for bad in (-1, 4, 100):
        with pytest.raises(tp.TpmlpError) as e:
            tp.tpmlp_plan_set_stream_k(p, bad)
        assert e.value.status == 1
    assert lib.tpmlp_plan_set_stream_k(None, 1) == 1
    a = tp.AttnPlan(512, 64, [64], [64], "bf16")
    tp.tpmlp_plan_set_stream_k(a, tp.STREAM_K_OFF)
