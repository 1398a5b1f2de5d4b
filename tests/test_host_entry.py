"""fmha_fwd_host: the forward from host memory (C ABI with host buffers).

CPU: argument errors return their codes before any CUDA call.  GPU: the host
entry returns bit for bit what fmha_fwd returns on the same inputs, for every
kernel family, with page-locked and pageable host memory, and with calls
alternating between two streams (each stream keeps its own device copies).
"""
import pytest
import torch

from head_attention_forward_fmha_gb300 import binding, build, inputs


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_host_entry_argument_errors(lib):
    f = lib.fmha_fwd_host
    # q, k, v, o, lse, batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, stream
    assert f(None, 8, 8, 8, 8, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -1         # q NULL
    assert f(8, 8, 8, None, 8, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -1         # o NULL
    assert f(8, 8, 8, 8, None, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -1         # lse NULL
    assert f(8, 8, 8, 8, 8, 1, 2, 1, 1, 8, 80, 0.125, 0, 0, None) == -3           # head dim
    assert f(8, 8, 8, 8, 8, 1, 3, 2, 1, 8, 64, 0.125, 0, 0, None) == -4           # heads
    assert f(8, 8, 8, 8, 8, 1, 2, 1, 9, 8, 64, 0.125, 0, 1, None) == -5           # causal T > s_k
    assert f(8, 8, 8, 8, 8, 0, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == 0            # empty: nothing to do
    assert f(8, 8, 8, None, 8, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -1
    assert "non-NULL" in binding.fmha_get_last_error()


CASES = [
    inputs.Workload("host_gqa_split", 2, 8, 2, 1, 700, 128, window=300),   # decode kernel + merge
    inputs.Workload("host_tc_causal", 1, 4, 4, 96, 200, 64, causal=True),  # 128-row tensor-core kernel
    inputs.Workload("host_wide", 2, 64, 1, 1, 300, 512),                   # hd-512 kernel, fp16 partials + merge
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry_matches_device_entry(w, pinned):
    q, k, v = inputs.make_inputs(w, seed=3)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    stream = torch.cuda.Stream()
    o_h, lse_h = binding.fmha_fwd_host(q, k, v, scale=w.scale, window=w.window, causal=w.causal, stream=stream)
    stream.synchronize()
    o_d, lse_d = binding.fmha_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    assert torch.equal(o_h.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse_d.cpu())


@pytest.mark.gpu
def test_host_entry_two_streams_alternating():
    w = CASES[0]
    sets = [inputs.make_inputs(w, seed=10 + i) for i in range(6)]
    sets = [tuple(t.pin_memory() for t in s) for s in sets]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i, (q, k, v) in enumerate(sets):
        o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((w.batch, w.n_h, w.T), dtype=torch.float32).pin_memory()
        binding.fmha_fwd_host(q, k, v, o, lse, scale=w.scale, window=w.window, stream=streams[i % 2])
        outs.append((o, lse))
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    for (q, k, v), (o, lse) in zip(sets, outs):
        o_d, lse_d = binding.fmha_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, window=w.window)
        assert torch.equal(o.view(torch.int16), o_d.cpu().view(torch.int16))
        assert torch.equal(lse, lse_d.cpu())
