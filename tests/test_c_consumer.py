"""The C ABI from plain C (no GPU needed): include/mbw.h compiles as C99 and
as C++ with strict warnings, and a C program linked against libmbw.so gets
the documented status from every call whose argument checks run before any
CUDA work (tests/c/abi_consumer.c)."""
import os
import shutil
import subprocess

import pytest

from memory_bound_weight_gb300 import _binding as B
from memory_bound_weight_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(ROOT, "tests", "c", "abi_consumer.c")


def need(tool):
    if shutil.which(tool) is None:
        pytest.skip(f"{tool} not found")


def test_header_compiles_as_c_and_cpp(tmp_path):
    need("gcc")
    need("g++")
    stub = tmp_path / "h.c"
    stub.write_text('#include "mbw.h"\nint main(void) { return MBW_OK; }\n')
    for cc, std, lang in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "c++")):
        r = subprocess.run([cc, std, "-x", lang, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                            "-I", INCLUDE, str(stub)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_program_links_and_gets_documented_statuses(tmp_path):
    need("gcc")
    mbuild.build()
    lib_dir = os.path.dirname(B.LIB_PATH)
    exe = tmp_path / "abi_consumer"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, SRC,
                        "-o", str(exe), f"-L{lib_dir}", "-l:libmbw.so", f"-Wl,-rpath,{lib_dir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
