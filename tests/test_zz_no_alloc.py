"""fmha_fwd_noalloc: the entry point for callers that cannot allocate device
memory (a runtime that reserves all of its memory up front, a strict memory
budget, a hot loop that must not risk allocator synchronisation).  It must
return what fmha_fwd returns, through the C ABI, on consecutive calls that
share its fixed split-KV scratch, and must refuse shapes whose partials do
not fit that scratch.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import pytest
import torch

from check_utils import LSE_ATOL, O_ATOL
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

# Shapes that fmha_fwd splits, so the scratch array is really used: a GQA
# sliding-window decode with few KV heads (decode kernel) and an MQA decode
# with many cached keys (tensor-core kernel).
SPLIT_SHAPES = [
    W("gqa_swa_decode_b4", 4, 64, 8, 1, 8192, 128, window=4096),
    W("mqa_G128_hd128_long", 2, 128, 1, 1, 4096, 128),
]


def _plan(w):
    return binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window, w.causal)


@pytest.mark.parametrize("w", SPLIT_SHAPES, ids=[w.name for w in SPLIT_SHAPES])
def test_noalloc_matches_fmha_fwd_on_two_calls(w):
    binding.fmha_set_kernel_path(0)
    n_splits, _ = _plan(w)
    assert n_splits > 1, "shape must exercise the split-KV scratch"
    need = binding.fmha_splitkv_workspace_bytes(w.batch, w.n_h, w.T, w.hd, n_splits)
    assert need <= binding.NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((21, 22)):       # two calls in a row, different inputs
        q, k, v = inputs.make_inputs(w, seed=seed, device="cuda")
        o_ref, lse_ref = binding.fmha_fwd(q, k, v, scale=w.scale, window=w.window, causal=w.causal)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.batch, w.n_h, w.T), float("nan"), dtype=torch.float32, device="cuda")
        binding.fmha_fwd_noalloc(q, k, v, o, lse, scale=w.scale, window=w.window, causal=w.causal)
        torch.cuda.synchronize()
        binding.fmha_check_device_status()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), "call %d left outputs unwritten" % call
        assert (o.float() - o_ref.float()).abs().max().item() <= O_ATOL, "call %d: O differs" % call
        assert (lse - lse_ref).abs().max().item() <= LSE_ATOL, "call %d: LSE differs" % call


def test_noalloc_unsplit_shape_needs_no_scratch():
    w = inputs.WORKLOADS["causal_prefill"].with_(batch=2)
    q, k, v = inputs.make_inputs(w, seed=23, device="cuda")
    o_ref, lse_ref = binding.fmha_fwd(q, k, v, scale=w.scale, causal=True)
    o = torch.empty_like(q)
    lse = torch.empty((w.batch, w.n_h, w.T), dtype=torch.float32, device="cuda")
    binding.fmha_fwd_noalloc(q, k, v, o, lse, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    assert (o.float() - o_ref.float()).abs().max().item() <= O_ATOL
    assert (lse - lse_ref).abs().max().item() <= LSE_ATOL


def test_noalloc_rejects_partials_larger_than_the_scratch():
    # MHA prefill at hd 512, 100 heads, 4096 cached keys: the plan splits the
    # keys in two, and the fp32 partials of 12,800 query rows need ~52 MB, more
    # than the scratch.  The call is refused before anything runs, so the
    # inputs need no values.
    w = W("oversize", 1, 100, 100, 128, 4096, 512)
    n_splits, _ = _plan(w)
    need = binding.fmha_splitkv_workspace_bytes(w.batch, w.n_h, w.T, w.hd, n_splits)
    if need <= binding.NOALLOC_SCRATCH_BYTES:
        pytest.skip("this GPU's plan for the shape fits the scratch (%d bytes)" % need)
    q = torch.empty((w.batch, w.n_h, w.T, w.hd), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((w.batch, w.n_kv_h, w.s_k, w.hd), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    o = torch.zeros_like(q)
    lse = torch.zeros((w.batch, w.n_h, w.T), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.FmhaError) as ei:
        binding.fmha_fwd_noalloc(q, k, v, o, lse, scale=w.scale)
    assert ei.value.code == -6
    assert "scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert (o == 0).all() and (lse == 0).all()   # nothing was launched
