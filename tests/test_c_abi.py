"""The boundary from plain C: tests/c/abi_check.c includes include/moe.h as C99 (with -Wall
-Wextra -pedantic -Werror), links the built library and runs its host-side checks (no GPU)."""
import os
import shutil
import subprocess

import pytest

import mixture_experts_layer_09_gb300 as moe
from mixture_experts_layer_09_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_as_c_and_links(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    moe.build()
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(_build.LIB)
    libname = os.path.basename(_build.LIB)
    assert libname.startswith("lib") and libname.endswith(".so")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_check.c"),
                    "-L", libdir, "-l:" + libname, "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
