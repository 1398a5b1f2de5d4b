"""Failure detection without a GPU fault.

Every wait inside the kernels is bounded; when one gives up, the kernel sets a
device status word and returns.  The self-test kernel waits on a barrier that
nothing completes; the host must then read FMHA_ERR_DEVICE_TIMEOUT once, find
the word cleared afterwards, and the context must still compute correctly.
"""
import pytest
import torch

from check_utils import compare, device_inputs, oracle_full
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    binding.fmha_check_device_status()                 # start clean
    binding.fmha_selftest_wait_timeout(20000)          # 20 ms
    with pytest.raises(binding.FmhaError) as ei:
        binding.fmha_check_device_status()
    assert ei.value.code == -8
    binding.fmha_check_device_status()                 # cleared after one report
    w = inputs.Workload("after_timeout", 1, 8, 2, 1, 300, 128, window=100)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=31)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, "after timeout")


def test_selftest_argument_range():
    with pytest.raises(binding.FmhaError):
        binding.fmha_selftest_wait_timeout(0)
