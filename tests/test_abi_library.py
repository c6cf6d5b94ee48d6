"""The C-ABI library loads (no GPU needed) and exports every declared entry point."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT, library


def _declared():
    text = open(os.path.join(ROOT, "include", "fsdp_unit.h")).read()
    return sorted(set(re.findall(r"FSDP_API\s+[\w\s\*]+?\b(fsdp_\w+)\s*\(", text)))


def test_header_declares_the_cycle():
    names = _declared()
    for n in ("fsdp_unit_create", "fsdp_allgather", "fsdp_reduce_scatter", "fsdp_adamw_step", "fsdp_step"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = library()
    for name in _declared():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else():
    from fully_sharded_unit_gb300.build import LIB
    library()
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("fsdp_")})
    assert exported == _declared()


def test_binding_covers_every_declared_symbol():
    from fully_sharded_unit_gb300 import binding
    for name in _declared():
        assert callable(getattr(binding, name)), name


def test_strerror_and_codes():
    from fully_sharded_unit_gb300 import binding as B
    library()
    assert B.fsdp_strerror(B.FSDP_OK) == "ok"
    assert B.fsdp_strerror(B.FSDP_E_ALIGN) == "misaligned buffer"
    assert B.fsdp_strerror(12345) == "unknown error"


def test_oracle_is_not_imported_by_the_package():
    pkg = os.path.join(ROOT, "fully_sharded_unit_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".hpp", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "from oracle" not in src and "import oracle" not in src, f


def test_status_and_selftest_reject_bad_arguments_without_a_device():
    """Argument checks come before any CUDA call, so they hold on a host
    without a GPU."""
    library()
    from fully_sharded_unit_gb300 import binding as B
    for limit in (0.0, 1e-4, 20.0, float("nan")):
        with pytest.raises(B.FsdpError) as e:
            B.fsdp_selftest_bounded_wait(limit, stream=0)
        assert e.value.code == B.FSDP_E_INVALID_ARG
    f = ctypes.c_int32()
    assert B.lib().fsdp_kernel_status(None, ctypes.byref(f), None) == B.FSDP_E_INVALID_ARG
