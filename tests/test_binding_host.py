"""The Python binding's own argument checks (no GPU, no kernel launch): tensors
of the wrong dtype, device, layout or shape are refused before any call into
the library, and the host entry takes CPU tensors only."""
import pytest
import torch

from head_attention_forward_fmha_gb300 import binding, build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load()


def cpu_qkv(b=1, n_h=2, n_kv_h=1, T=1, s_k=8, hd=64, dtype=torch.bfloat16):
    return (torch.zeros(b, n_h, T, hd, dtype=dtype), torch.zeros(b, n_kv_h, s_k, hd, dtype=dtype),
            torch.zeros(b, n_kv_h, s_k, hd, dtype=dtype))


def test_device_entry_refuses_host_tensors():
    q, k, v = cpu_qkv()
    with pytest.raises(TypeError):
        binding.fmha_fwd(q, k, v, o=torch.empty(0), lse=torch.empty(0))


def test_shape_checks():
    q, k, v = cpu_qkv()
    with pytest.raises(ValueError):
        binding.fmha_fwd(q[0], k, v)                       # q not 4-D
    with pytest.raises(ValueError):
        binding.fmha_fwd(q, k, v[:, :, :4].contiguous())   # k and v differ
    with pytest.raises(ValueError):
        binding.fmha_fwd(q, k[..., :32].contiguous(), v[..., :32].contiguous())  # head dims differ


def test_host_entry_checks():
    q, k, v = cpu_qkv(dtype=torch.float32)
    with pytest.raises(TypeError):
        binding.fmha_fwd_host(q, k, v, o=torch.empty(1, 2, 1, 64, dtype=torch.bfloat16),
                              lse=torch.empty(1, 2, 1))    # fp32 inputs
    q, k, v = cpu_qkv()
    with pytest.raises(TypeError):
        strided_q = torch.zeros(1, 2, 1, 128, dtype=torch.bfloat16)[..., ::2]  # right shape, not contiguous
        binding.fmha_fwd_host(strided_q, k, v, o=torch.empty(1, 2, 1, 64, dtype=torch.bfloat16),
                              lse=torch.empty(1, 2, 1))
    with pytest.raises(ValueError):
        binding.fmha_fwd_host(q, k, v, o=torch.empty(1, 2, 2, 64, dtype=torch.bfloat16),
                              lse=torch.empty(1, 2, 1))    # o of the wrong shape


def test_noalloc_refuses_undersized_outputs():
    """fmha_fwd_noalloc and fmha_fwd take caller buffers for O and LSE; one
    smaller than the output is refused before any launch (the kernels would
    write past its end)."""
    q, k, v = cpu_qkv(b=2, n_h=4, n_kv_h=2, T=3)
    good_o, good_lse = torch.empty_like(q), torch.empty(2, 4, 3)
    binding._check_outputs(q, good_o, good_lse)
    with pytest.raises(ValueError):
        binding._check_outputs(q, torch.empty(2, 4, 2, 64, dtype=torch.bfloat16), good_lse)   # o one row short
    with pytest.raises(ValueError):
        binding._check_outputs(q, good_o, torch.empty(2, 4, 2))                               # lse one row short
    with pytest.raises(ValueError):
        binding._check_outputs(q, good_o.reshape(-1), good_lse)                               # o flattened
    with pytest.raises(ValueError):
        binding._check_outputs(q, good_o, torch.empty(2, 4, 3, device="meta"))               # another device
    # Both entry points run the check before calling into the library; with
    # host tensors the dtype/device check (TypeError) comes first, so the order
    # is checked by source: _check_outputs precedes the library call.
    import inspect
    for fn, call in ((binding.fmha_fwd_noalloc, "fmha_fwd_noalloc("), (binding.fmha_fwd, "fmha_fwd(")):
        src = inspect.getsource(fn)
        assert "_check_outputs(q, o, lse)" in src
        assert src.index("_check_outputs(q, o, lse)") < src.index("load()." + call)


def test_workspace_bytes_alias():
    assert binding.fmha_workspace_bytes(2, 8, 1, 128, 4) == binding.fmha_splitkv_workspace_bytes(2, 8, 1, 128, 4)
    assert binding.fmha_workspace_bytes(3, 5, 7, 512, 2) == 2 * 3 * 5 * 7 * (512 + 1) * 4


def test_merge_checks():
    with pytest.raises(ValueError):
        binding.fmha_merge(torch.empty(2, 1, 2, 1), torch.empty(2, 1, 2, 1))  # o_parts not 5-D


def test_error_codes_are_named():
    for code in range(-1, -11, -1):
        assert binding.ERRORS[code].startswith("FMHA_ERR_")
