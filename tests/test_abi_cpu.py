"""The C-ABI library builds, loads without a GPU, and exports what include/q4lin.h
declares; host-side validation runs before any device work.  No compute calls."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4lin.h")


@pytest.fixture(scope="module")
def lib():
    from bit_weight_quantized_int4_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"Q4LIN_API\s+[\w\s\*]+?\b(q4lin_\w+)\s*\(", text)


def declared_enums():
    text = open(HEADER).read()
    return {name: int(val) for name, val in re.findall(r"\b(Q4LIN_[A-Z0-9_]+)\s*=\s*(\d+)", text)}


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"q4lin_create", "q4lin_run", "q4lin_destroy", "q4lin_plan", "q4lin_set_option",
            "q4lin_get_option", "q4lin_check_device_status", "q4lin_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in q4lin.h but not exported"


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and "q4lin" in l}
    assert exported == set(declared_functions())


def test_python_constants_match_header():
    from bit_weight_quantized_int4_gb300 import q4lin
    for name, val in declared_enums().items():
        assert getattr(q4lin, name) == val, name


def test_status_strings(lib):
    from bit_weight_quantized_int4_gb300 import q4lin
    for code in range(7):
        s = q4lin.q4lin_status_string(code)
        assert s and s != "unknown status"
    assert q4lin.q4lin_status_string(99) == "unknown status"


def test_validation_rejects_before_device_work():
    """A NULL handle and bad sizes are rejected on the host; nothing touches a GPU."""
    from bit_weight_quantized_int4_gb300 import q4lin as q
    assert q.q4lin_run(None, 16, 16, 16, None, 4096, 1, 1, 32, 32, 0, None) == q.Q4LIN_ERR_INVALID_ARG
    st, _ = q.q4lin_plan(None, 16, 16, 16, None, 4096, 1, 1, 32, 32, 0)
    assert st == q.Q4LIN_ERR_INVALID_ARG
    assert q.q4lin_set_option(None, q.Q4LIN_OPT_PDL, 1) == q.Q4LIN_ERR_INVALID_ARG
    assert q.q4lin_destroy(None) == q.Q4LIN_OK
    assert (q.q4lin_run_backward_dx(None, 16, 16, 16, 4096, 1, 1, 32, 32, 0, None)
            == q.Q4LIN_ERR_INVALID_ARG)
    assert q.q4lin_run_requant(None, 16, 16, 4096, 1, 32, 32, 0, None) == q.Q4LIN_ERR_INVALID_ARG


def test_create_without_gpu_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from bit_weight_quantized_int4_gb300 import q4lin as q
    with pytest.raises(q.Q4LinError) as e:
        q.q4lin_create(0)
    assert e.value.status == q.Q4LIN_ERR_NO_DEVICE
