"""The C ABI from plain C and from C++: tests/c_abi/abi_check.c includes
include/fmha.h (gcc -std=c99, and g++ -std=c++17 with the file read as C++;
warnings as errors), links against the library and runs the calls that need
no GPU (version, build flags, split layout, planner, argument errors,
workspace size)."""
import os
import shutil
import subprocess

import pytest

from head_attention_forward_fmha_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c99"), ("g++", "-std=c++17")])
def test_plain_c_client(tmp_path, compiler, std):
    if shutil.which(compiler) is None:
        pytest.skip(compiler + " not found")
    lib = build.build()
    exe = str(tmp_path / "abi_check")
    src = os.path.join(ROOT, "tests", "c_abi", "abi_check.c")
    # the C source read as C++ by g++; "-x none" so that the library is not
    lang, reset = (["-x", "c++"], ["-x", "none"]) if compiler == "g++" else ([], [])
    cmd = [compiler, std, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include")] + lang + [src] + \
          reset + ["-o", exe, lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
