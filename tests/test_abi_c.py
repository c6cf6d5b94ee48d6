"""The header is valid C99 and the library links and works from a plain C
caller (host-only entry points; no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT, library


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_caller(tmp_path):
    library()
    from fully_sharded_unit_gb300.build import LIB, LIBDIR
    exe = tmp_path / "c_abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", str(exe), LIB, f"-Wl,-rpath,{LIBDIR}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines()
    assert out[0] == "P=3136 segments=4"
    # floor boundaries: 3136 / 4 = 784 each; arena slot congruent to the global index mod 32
    for k, line in enumerate(out[1:5]):
        f = dict(x.split("=") for x in line.split())
        assert (int(f["rank"]), int(f["global"]), int(f["len"])) == (k, 784 * k, 784)
        assert int(f["arena"]) % 32 == int(f["global"]) % 32
    assert out[5] == "N=0 -> invalid argument"
