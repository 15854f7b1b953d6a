"""The boundary is a plain C ABI: a C11 program that includes only
``include/clef.h`` compiles with warnings as errors, links the built
``libclef.so`` and gets the documented host-side answers (version, status
names, argument errors before any launch).  Needs no GPU."""
import os
import shutil
import subprocess

import pytest

import w8a8_quantized_projections_gb300 as clef

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_caller(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    lib = clef.library_path()
    clef.library()                         # builds the library if it is missing
    exe = str(tmp_path / "c_abi_check")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           "-o", exe, lib, "-Wl,-rpath," + os.path.dirname(lib)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert p.returncode == 0 and p.stdout.strip() == "ok", p.stderr
