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
    assert tp.tpmlp_version() == 101
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
        assert tp.tpmlp_workspace_size(p) == 256
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
