"""The C ABI from plain C: tests/c_abi/abi_check.c includes include/fmha.h as C
(gcc, -std=c99, warnings as errors), links against the library and runs the
calls that need no GPU (version, build flags, split layout, planner, argument
errors, workspace size)."""
import os
import shutil
import subprocess

import pytest

from head_attention_forward_fmha_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_plain_c_client(tmp_path):
    lib = build.build()
    exe = str(tmp_path / "abi_check")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-o", exe, lib,
           "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
