"""The C ABI from C: include/rx.h compiles as C99 (and as C++), and a C program linked against
librx.so runs the host-side calls (accounting, radix cache, checks, plans) without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "c_abi_host.c")


def test_c99_program_runs_the_host_calls(librx, tmp_path):
    from prefix_shared_kv_gb300 import build
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(build.LIB)
    exe = str(tmp_path / "c_abi_host")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, SRC,
                        "-L", libdir, "-lrx", "-Wl,-rpath," + libdir, "-lm", "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_header_compiles_as_cplusplus(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "h.cpp"
    src.write_text('#include "rx.h"\nint main() { return rx_saved_tokens(16, 16) == 16 ? 0 : 1; }\n')
    r = subprocess.run([gxx, "-std=c++11", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                        INCLUDE, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
