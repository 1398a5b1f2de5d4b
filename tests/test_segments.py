"""Multi-segment decode through the public split-KV calls.

A KV cache held in separate buffers (say a shared prefix and the new tokens)
is attended by running fmha_fwd_splitkv on each segment into consecutive
slices of one partial buffer and merging all slices with fmha_merge: the LSE
merge is exact, so the result is attention over the concatenated keys.
Checked against the fp64 oracle on the concatenated cache (no mask: key
positions inside a segment do not matter).
"""
import pytest
import torch

from check_utils import compare, cosine_per_head, oracle_full
from head_attention_forward_fmha_gb300 import binding, inputs

CASES = [
    # name, batch, n_h, n_kv_h, T, hd, segment lengths, kv_chunk
    ("gqa_two_segments", 2, 8, 2, 1, 128, (300, 200), 128),
    ("mqa_three_segments", 2, 64, 1, 1, 64, (128, 1, 383), 96),
    ("mha_short_query", 1, 4, 4, 4, 256, (64, 448), 256),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,b,n_h,n_kv_h,T,hd,segs,chunk", CASES, ids=[c[0] for c in CASES])
def test_segmented_cache_matches_concatenated(name, b, n_h, n_kv_h, T, hd, segs, chunk):
    w = inputs.Workload(name, b, n_h, n_kv_h, T, sum(segs), hd)
    q, k, v = inputs.make_inputs(w, seed=5)
    dev = torch.device("cuda")
    qd = q.to(dev)
    counts = [binding.fmha_split_layout(T, n, 0, chunk)[1] for n in segs]
    o_parts = torch.empty((sum(counts), b, n_h, T, hd), dtype=torch.float32, device=dev)
    lse_parts = torch.empty((sum(counts), b, n_h, T), dtype=torch.float32, device=dev)
    start, off = 0, 0
    for n, c in zip(segs, counts):
        ks = k[:, :, start:start + n].contiguous().to(dev)   # each segment in its own buffer
        vs = v[:, :, start:start + n].contiguous().to(dev)
        binding.fmha_fwd_splitkv(qd, ks, vs, chunk, o_parts=o_parts[off:off + c], lse_parts=lse_parts[off:off + c],
                                 scale=w.scale)
        start, off = start + n, off + c
    o, lse = binding.fmha_merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, name)
    cosine_per_head(o, o_ref, name)
