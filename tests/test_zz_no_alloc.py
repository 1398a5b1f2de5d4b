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

from check_utils import LSE_ATOL, O_ATOL, compare, cosine_per_head
import oracle
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

# Shapes that fmha_fwd splits, so the scratch array is really used: a GQA
# sliding-window decode with few KV heads (decode kernel, fp32 partials), an
# MQA decode with many cached keys (tensor-core kernel, fp32 partials), the
# MQA decode at hd 512 (hd-512 tensor-core kernel, fp16 partials with range
# factors) and two GQA prefills (two-row-tile kernel, fp32 partials, hd 128
# and 64); the hd-512 and hd-64 ones are also checked against the fp64 oracle.
SPLIT_SHAPES = [
    W("gqa_swa_decode_b4", 4, 64, 8, 1, 8192, 128, window=4096),
    W("mqa_G128_hd128_long", 2, 128, 1, 1, 4096, 128),
    W("mqa_decode_hd512", 16, 128, 1, 1, 512, 512),
    W("gqa_prefill_pair_hd128", 1, 64, 8, 128, 4096, 128, causal=True),
    W("gqa_pair_hd64_long", 1, 32, 2, 64, 8192, 64),
]
ORACLE_CHECKED = {"mqa_decode_hd512", "gqa_pair_hd64_long"}


def _plan(w):
    return binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window, w.causal, with_kernel=True)


def _scratch_need(w, n_splits, kernel):
    """Bytes of partials fmha_fwd_noalloc keeps in its scratch: fp16 O plus fp32
    LSE and two fp32 range factors per row on the hd-512 tensor-core kernel,
    fp32 O and LSE elsewhere."""
    rows = w.batch * w.n_h * w.T
    if w.hd == 512 and kernel == "fwd_tc_wide":
        return n_splits * rows * (w.hd * 2 + 12)
    return binding.fmha_splitkv_workspace_bytes(w.batch, w.n_h, w.T, w.hd, n_splits)


@pytest.mark.parametrize("w", SPLIT_SHAPES, ids=[w.name for w in SPLIT_SHAPES])
def test_noalloc_matches_fmha_fwd_on_two_calls(w):
    binding.fmha_set_kernel_path(0)
    n_splits, _, kernel = _plan(w)
    assert n_splits > 1, "shape must exercise the split-KV scratch"
    assert _scratch_need(w, n_splits, kernel) <= binding.NOALLOC_SCRATCH_BYTES
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
        # same plan, kernels and partial format: the same bits
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), "call %d: not fmha_fwd's bits" % call
        if w.name in ORACLE_CHECKED:
            bits = [inputs.bf16_bits(t.cpu()) for t in (q, k, v)]
            o_or, lse_or = oracle.attention(*bits, w.scale, w.window, w.causal)
            compare(o, lse, o_or, lse_or, "%s call %d vs oracle" % (w.name, call))
            cosine_per_head(o, o_or, "%s call %d vs oracle" % (w.name, call))


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


# MQA prefills at hd 256 with 100 query heads over long caches: 12,800 query
# rows (25,600 for batch 2) whose fp32 partials take ~13 MB per KV chunk, and
# the plan splits them into 2-4 chunks (~50 MB).  The first one this GPU's
# plan splits beyond the scratch is used.
OVERSIZE = [W("oversize_b1_sk16k", 1, 100, 1, 128, 16384, 256),
            W("oversize_b2_sk8k", 2, 100, 1, 128, 8192, 256),
            W("oversize_b1_sk32k", 1, 100, 1, 128, 32768, 256)]


def test_noalloc_rejects_partials_larger_than_the_scratch():
    # The call is refused before anything runs, so the inputs need no values.
    for w in OVERSIZE:
        n_splits, _, kernel = _plan(w)
        need = _scratch_need(w, n_splits, kernel)
        if n_splits > 1 and need > binding.NOALLOC_SCRATCH_BYTES:
            break
    else:
        pytest.skip("this GPU's plans for the oversize shapes fit the scratch")
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
