"""The C ABI from plain C: include/bf16_linear.h compiles as C99 with warnings as
errors, a C program links against the library, and the host-only entry points
answer as documented (tests/c_abi_check.c; no GPU is touched)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_header_and_library_from_c(lib, tmp_path):
    lib.load()  # builds the library if needed
    libdir = os.path.dirname(lib.LIB_PATH)
    name = os.path.basename(lib.LIB_PATH)[3:-3]  # libNAME.so -> NAME
    exe = tmp_path / "c_abi_check"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           "-L", libdir, f"-l{name}", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "FAIL" not in run.stdout
    assert run.stdout.count("ok ") >= 14
