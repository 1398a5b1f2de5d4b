"""The checked build (``libfmha_gb300_checked.so``, compiled with -DFMHA_CHECKED).

Its kernels test every computed shared-memory offset, tensor-memory column,
global-memory index and TMA coordinate before the access and report a failed
check through the device status word.  This stands in for a memory checker
(none runs on these GPUs): the GPU parity suites are re-run in a child
process against the checked build, and ``tests/conftest.py`` reads the status
word after each test there, so every kernel path those suites reach is also
run with its index checks on.  A failing check is only ever planted through
the self-test entry point, which runs a false check with no access behind it.
"""
import os
import subprocess
import sys

import pytest

from head_attention_forward_fmha_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _checked_env():
    env = dict(os.environ)
    env["FMHA_GB300_LIB"] = build.build(checked=True)
    return env


def test_checked_library_exports_the_same_entry_points():
    normal = binding.load(build.build())
    checked = binding.load(build.build(checked=True))
    for name in binding.SIGNATURES:
        assert hasattr(checked, name), "checked build lacks " + name
    assert normal.fmha_build_flags() == 0
    assert checked.fmha_build_flags() == binding.FMHA_BUILD_CHECKED
    # host-side argument checks are the same code in both
    for lib in (normal, checked):
        assert lib.fmha_fwd(16, 16, 16, 16, 16, 1, 2, 1, 1, 8, 80, 0.125, 0, 0, None) == -3
        assert lib.fmha_fwd(16, 16, 16, 16, 16, 1, 3, 2, 1, 8, 64, 0.125, 0, 0, None) == -4


@pytest.mark.gpu
def test_selftest_check_is_compiled_out_of_the_normal_build():
    binding.load()
    binding.fmha_check_device_status()
    binding.fmha_selftest_bounds_check()
    binding.fmha_check_device_status()  # nothing recorded


_SELFTEST = r"""
import sys
sys.path.insert(0, %r)
import torch
from head_attention_forward_fmha_gb300 import binding
assert binding.fmha_build_flags() == binding.FMHA_BUILD_CHECKED
binding.fmha_check_device_status()
binding.fmha_selftest_bounds_check()
try:
    binding.fmha_check_device_status()
    raise SystemExit("the failed self-test check was not reported")
except binding.FmhaError as e:
    assert e.code == -10, e
    assert "0x601" in str(e) and "self-test" in str(e), e
binding.fmha_check_device_status()  # reading cleared it
q = torch.randn(1, 4, 1, 64, device="cuda").to(torch.bfloat16)
k = torch.randn(1, 1, 300, 64, device="cuda").to(torch.bfloat16)
o, lse = binding.fmha_fwd(q, k, k.clone(), scale=0.125)
binding.fmha_check_device_status()
print("checked self-test ok")
""" % ROOT


@pytest.mark.gpu
def test_checked_build_reports_a_failed_check():
    r = subprocess.run([sys.executable, "-c", _SELFTEST], env=_checked_env(), cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "checked self-test ok" in r.stdout


SUITES = ["tests/test_parity.py", "tests/test_kernel_paths.py", "tests/test_sink.py", "tests/test_host_entry.py",
          "tests/test_segments.py", "tests/test_nvfp4.py", "tests/test_pair_kernel.py",
          "tests/test_zz_no_alloc.py"]


@pytest.mark.gpu
def test_gpu_parity_suites_pass_with_index_checks():
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider"],
                       env=_checked_env(), cwd=ROOT, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
