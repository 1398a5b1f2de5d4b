"""GPU parity of the attention sink (fmha_fwd_sink, fmha_merge with a sink)
against the fp64 oracle.

The pages leave the sink undefined ("D5c sink", a TODO); the reading the oracle
states and the library implements: a per-query-head logit that joins the
softmax denominator only.  Every kernel family is run (forced paths and the
automatic plan, split and unsplit), with sinks below, around and far above
the scores, and with -inf (no sink) for some heads.
"""
import numpy as np
import pytest
import torch

import oracle
from check_utils import compare, cosine_per_head, device_inputs, to_np_bits
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

SHAPES = [
    W("sink_gqa_decode", 2, 16, 2, 1, 300, 128),
    W("sink_T4_causal_hd64", 2, 8, 8, 4, 70, 64, causal=True),
    W("sink_hd64_R40_causal_long", 1, 8, 2, 10, 16500, 64, causal=True),
    W("sink_window_hd256", 1, 32, 1, 2, 900, 256, window=300),
    W("sink_prefill_hd256", 2, 4, 4, 128, 256, 256, causal=True),
    W("sink_mqa_hd512_split", 2, 128, 1, 1, 512, 512),
    W("sink_hd512_R200", 1, 200, 1, 1, 129, 512),
    W("sink_hd512_T32_q32", 4, 16, 16, 32, 512, 512, causal=True),
]


def make_sink(n_h, seed):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(n_h, generator=g, dtype=torch.float64) * 2.0
    s[0::5] = 30.0           # dominates every score: O -> 0, lse -> sigma
    s[1::5] = -float("inf")  # no sink for these heads
    s[2::5] = 0.0
    return s.float().double()  # the fp32 values the GPU reads


def oracle_sink(w, q, k, v, sink):
    return oracle.attention(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, w.window, w.causal,
                            sink=sink.numpy())


@pytest.fixture
def path():
    yield binding.fmha_set_kernel_path
    binding.fmha_set_kernel_path(0)


@pytest.mark.parametrize("which", [0, 1, 2], ids=["auto", "decode_kernel", "tensor_core_kernel"])
@pytest.mark.parametrize("w", SHAPES, ids=[w.name for w in SHAPES])
def test_fwd_sink_matches_oracle(w, which, path):
    path(which)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=31)
    sink = make_sink(w.n_h, 5)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal,
                              sink=sink.float().cuda())
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_sink(w, q, k, v, sink)
    label = "%s/path%d" % (w.name, which)
    compare(o, lse, o_ref, lse_ref, label)
    # heads whose sink dominates have O ~ 0: the cosine is not informative there
    keep = np.ones(w.n_h, dtype=bool)
    keep[0::5] = False
    cosine_per_head(o[:, keep], o_ref[:, keep], label)


def test_sink_of_minus_inf_is_fmha_fwd():
    w = SHAPES[0]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=32)
    o0, l0 = binding.fmha_fwd(qd, kd, vd, scale=w.scale)
    o1, l1 = binding.fmha_fwd(qd, kd, vd, scale=w.scale,
                              sink=torch.full((w.n_h,), -float("inf"), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.parametrize("chunk", [64, 128])
def test_merge_with_sink_matches_oracle(chunk):
    w = W("sink_split_api", 2, 8, 2, 3, 400, 128, window=250, causal=True)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=33)
    sink = make_sink(w.n_h, 6)
    op, lp = binding.fmha_fwd_splitkv(qd, kd, vd, chunk, scale=w.scale, window=w.window, causal=w.causal)
    o, lse = binding.fmha_merge(op, lp, sink=sink.float().cuda())
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_sink(w, q, k, v, sink)
    compare(o, lse, o_ref, lse_ref, "merge+sink chunk %d" % chunk)
