"""GPU parity of each kernel family on shapes the automatic choice would send
to the other one: the decode kernel (mma.sync, 8/16 query rows per block) and
the 128-row tensor-core kernels (tcgen05 + TMEM), all against the fp64 oracle.
Path 2 forces the tensor-core kernels, with two row tiles per block where that
kernel applies (hd 64/128, more than 128 rows per KV head); path 4 forces one
row tile per block.  The row-tile kernel's P V product runs in the TS form by
default (P written over S in tensor memory, read from there as the MMA's A
operand); path 3 forces the SS form (P through shared memory), and both are
checked.
"""
import numpy as np
import pytest
import torch

import oracle
from check_utils import compare, cosine_per_head, device_inputs, oracle_full, to_np_bits
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

SHAPES = [
    W("k1_decode_gqa8", 2, 16, 2, 1, 300, 128),
    W("k2_T1_hd64", 3, 4, 4, 1, 1000, 64),
    W("k3_T128_causal_hd64", 1, 2, 2, 128, 300, 64, causal=True),
    W("k4_T128_causal_hd128", 2, 2, 1, 128, 520, 128, causal=True),
    W("k5_T128_causal_hd256", 1, 4, 4, 128, 512, 256, causal=True),
    W("k6_T100_window_causal", 1, 2, 2, 100, 333, 128, window=77, causal=True),
    W("k7_mqa_G128_hd128", 2, 128, 1, 1, 700, 128),
    W("k8_mqa_G128_hd256", 1, 128, 1, 1, 257, 256),
    W("k9_gqa_prefill_G4_T40", 1, 8, 2, 40, 200, 128, causal=True),
    W("k10_R200_two_tiles", 1, 200, 1, 1, 129, 64),
    W("k11_T64_no_mask_sk1", 1, 2, 2, 64, 1, 128),
    W("k12_sk0", 1, 2, 2, 70, 0, 64),
    W("k13_T_gt_sk", 1, 2, 2, 90, 40, 256),
    W("k14_window_only_T128", 1, 2, 1, 128, 1000, 64, window=200),
    W("k15_long_sk_T64", 1, 1, 1, 64, 4097, 128, causal=True),
    W("k16_mqa_G128_hd512", 2, 128, 1, 1, 300, 512),
    W("k17_T128_causal_hd512", 1, 2, 2, 128, 260, 512, causal=True),
    W("k18_hd512_G64_T2_window", 1, 64, 1, 2, 700, 512, window=300),
    W("k19_hd512_R200", 1, 200, 1, 1, 129, 512),
    # hd 512, at most 32 or 64 query rows per KV head and blocks of two or
    # more KV tiles: the compact resident Q (32 or 64 rows per chunk)
    W("k20_hd512_T32_causal_q32", 1, 2, 2, 32, 600, 512, causal=True),
    W("k21_hd512_G4_T8_window_q32", 1, 8, 2, 8, 1000, 512, window=700),
    W("k22_hd512_T17_causal_q32", 1, 2, 2, 17, 300, 512, causal=True),
    W("k23_hd512_T1_q32", 2, 4, 4, 1, 700, 512),
    W("k24_hd512_T64_causal_q64", 1, 2, 2, 64, 600, 512, causal=True),
    W("k25_hd512_G3_T15_window_q64", 1, 6, 2, 15, 900, 512, window=500),
]


@pytest.fixture
def path():
    yield binding.fmha_set_kernel_path
    binding.fmha_set_kernel_path(0)


@pytest.mark.parametrize("which", [1, 2, 3, 4],
                         ids=["decode_kernel", "tensor_core_kernels", "tensor_core_kernel_ss", "tensor_core_kernel_ts"])
@pytest.mark.parametrize("w", SHAPES, ids=[w.name for w in SHAPES])
def test_kernel_family_matches_oracle(w, which, path):
    path(which)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=4)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, "%s/path%d" % (w.name, which))
    cosine_per_head(o, o_ref, "%s/path%d" % (w.name, which))


TS_SHAPES = [
    # the TS-form PV at every row-tile head dim, with causal, window and both
    W("ts_hd64_causal", 2, 4, 2, 128, 700, 64, causal=True),
    W("ts_hd64_window", 1, 8, 4, 64, 900, 64, window=333),
    W("ts_hd128_causal", 1, 4, 4, 128, 1000, 128, causal=True),
    W("ts_hd128_window_causal", 2, 8, 2, 32, 777, 128, window=129, causal=True),
    W("ts_hd256_causal", 1, 4, 4, 128, 512, 256, causal=True),
    W("ts_hd256_window", 1, 64, 1, 1, 1500, 256, window=1000),
    W("ts_hd256_window_causal", 1, 2, 2, 100, 640, 256, window=64, causal=True),
]


@pytest.mark.parametrize("which", [4, 3], ids=["ts", "ss"])
@pytest.mark.parametrize("w", TS_SHAPES, ids=[w.name for w in TS_SHAPES])
def test_pv_forms_match_oracle(w, which, path):
    """Row-tile kernel forced, in the TS form (path 4) and the SS form (path 3),
    against the oracle."""
    path(which)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=12)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, "%s/path%d" % (w.name, which))
    cosine_per_head(o, o_ref, "%s/path%d" % (w.name, which))


@pytest.mark.parametrize("hd,chunk", [(128, 64), (128, 100), (128, 256), (512, 128), (512, 200)])
def test_tensor_core_kernel_partials(hd, chunk, path):
    path(2)
    w = W("tc_split", 1, 4, 2, 64, 500, hd, window=300, causal=True)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=6)
    op, lp = binding.fmha_fwd_splitkv(qd, kd, vd, chunk, scale=w.scale, window=w.window, causal=w.causal)
    o, lse = binding.fmha_merge(op, lp)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    op_ref, lp_ref = oracle.partials(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, chunk, w.window,
                                     w.causal)
    compare(op, lp, op_ref, lp_ref, "tc partials hd %d chunk %d" % (hd, chunk))
    o_ref, lse_ref = oracle.merge(op_ref, lp_ref)
    compare(o, lse, o_ref, lse_ref, "tc merged hd %d chunk %d" % (hd, chunk))


def test_causal_prefill_both_families_agree(path):
    w = inputs.WORKLOADS["causal_prefill"]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=8)
    outs = []
    for which in (1, 2):
        path(which)
        o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, causal=True)
        torch.cuda.synchronize()
        outs.append((o.float(), lse))
    binding.fmha_check_device_status()
    assert (outs[0][0] - outs[1][0]).abs().max().item() <= 1.5e-2
    assert (outs[0][1] - outs[1][1]).abs().max().item() <= 1e-3
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(outs[1][0], outs[1][1], o_ref, lse_ref, "causal_prefill tc")


@pytest.mark.parametrize("v_scale_log2", [0, 17, -20, 100])
def test_hd512_fp16_workspace_keeps_range(v_scale_log2):
    """fmha_fwd holds hd-512 split partials in fp16 with a power-of-two factor
    per row half; V scaled by 2^17 (beyond fp16's 65504) or 2^-20 (below its
    normal range) must come out as the same result scaled exactly."""
    w = W("hd512_split_range", 2, 128, 1, 1, 512, 512)
    n, _, kern = binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, with_kernel=True)
    assert kern == "fwd_tc_wide" and n > 1, (n, kern)
    (q, k, v), (qd, kd, _) = device_inputs(w, seed=12)
    s = 2.0 ** v_scale_log2
    vd = (v.double() * s).to(torch.bfloat16).cuda()  # exact: a power-of-two multiple
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    o_back = o.double() / s
    label = "V x 2^%d" % v_scale_log2
    compare(o_back, lse, o_ref, lse_ref, label)
    cosine_per_head(o_back, o_ref, label)


@pytest.mark.parametrize("chunk", [128, 200])
def test_f16_partial_format_matches_oracle_and_fmha_fwd(chunk):
    """FMHA_PARTS_F16: the stored fp16 values times their range factors are the
    oracle's partials, the merge of them is the oracle's merge, and with
    fmha_fwd's own chunking the pair reproduces fmha_fwd bit for bit."""
    w = W("hd512_f16_parts", 2, 128, 1, 1, 700, 512, window=500)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=14)
    op, lp, rp = binding.fmha_fwd_splitkv_f16(qd, kd, vd, chunk, scale=w.scale, window=w.window)
    o, lse = binding.fmha_merge_f16(op, lp, rp)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    n, b, n_h, T, hd = op.shape
    deq = op.double() * rp.double().repeat_interleave(hd // 2, dim=-1)
    op_ref, lp_ref = oracle.partials(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, chunk, w.window, False)
    compare(deq, lp, op_ref, lp_ref, "f16 partials chunk %d" % chunk)
    o_ref, lse_ref = oracle.merge(op_ref, lp_ref)
    compare(o, lse, o_ref, lse_ref, "f16 merged chunk %d" % chunk)
    n_plan, chunk_plan = binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window, w.causal)
    op2, lp2, rp2 = binding.fmha_fwd_splitkv_f16(qd, kd, vd, chunk_plan, scale=w.scale, window=w.window)
    o2, lse2 = binding.fmha_merge_f16(op2, lp2, rp2)
    o3, lse3 = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window)
    torch.cuda.synchronize()
    assert op2.shape[0] == n_plan
    assert torch.equal(o2, o3) and torch.equal(lse2, lse3)
    _check_f16_ranges(op, "chunk %d" % chunk)
    _check_f16_ranges(op2, "plan chunk")


def _check_f16_ranges(op, label):
    """The range factor of each (split, row, half): the half row's largest stored
    |O_i 2^-k| lies in [2^14, 2^15) before rounding, so in [2^14, 2^15] in fp16 (whose
    spacing there is 16), unless the half row is all zero."""
    n, b, n_h, T, hd = op.shape
    mh = op.float().abs().reshape(n, b, n_h, T, 2, hd // 2).amax(-1)
    assert bool((mh <= 2.0 ** 15).all()), label + ": a stored fp16 partial exceeds 2^15"
    nz = mh > 0
    assert bool((mh[nz] >= 2.0 ** 14).all()), "%s: smallest half-row maximum %.3e < 2^14" % (label, mh[nz].min().item())


@pytest.mark.parametrize("chunk", [128, 0])
def test_f16_partials_beside_a_large_v_row_of_negligible_weight(chunk):
    """One key's V row is 2^60 times the rest while its K row is zero and Q is
    scaled by 30, so every row gives that key a weight below e^-40: |V| over the
    tile is no bound worth scaling the fp16 partials by (the other values would
    flush to zero), and the range factors must follow |O| itself.  chunk 0 = the
    plan's."""
    w = W("hd512_v_outlier", 2, 128, 1, 1, 700, 512, window=500)
    q, k, v = inputs.make_inputs(w, seed=15)
    q = (q.double() * 30).to(torch.bfloat16)
    key = 330
    k[:, :, key, :] = 0
    v[:, :, key, :] = (v[:, :, key, :].double() * 2.0 ** 60).to(torch.bfloat16)
    if chunk == 0:
        _, chunk = binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window, w.causal)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    op, lp, rp = binding.fmha_fwd_splitkv_f16(qd, kd, vd, chunk, scale=w.scale, window=w.window)
    o, lse = binding.fmha_merge_f16(op, lp, rp)
    o3, lse3 = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    n, b, n_h, T, hd = op.shape
    deq = op.double() * rp.double().repeat_interleave(hd // 2, dim=-1)
    qb, kb, vb = to_np_bits(q), to_np_bits(k), to_np_bits(v)
    op_ref, lp_ref = oracle.partials(qb, kb, vb, w.scale, chunk, w.window, False)
    label = "V outlier, chunk %d" % chunk
    compare(deq, lp, op_ref, lp_ref, label + " partials")
    o_ref, lse_ref = oracle.merge(op_ref, lp_ref)
    compare(o, lse, o_ref, lse_ref, label + " merged")
    cosine_per_head(o, o_ref, label)
    o_full, lse_full = oracle.attention(qb, kb, vb, w.scale, w.window, w.causal)
    compare(o3, lse3, o_full, lse_full, label + " fmha_fwd")
    _check_f16_ranges(op, label)


BACK_TO_BACK_SHAPES = [
    W("cnt_mqa", 2, 128, 1, 1, 512, 512),
    W("cnt_R200_two_row_tiles", 1, 200, 1, 1, 600, 512),
    W("cnt_T32_q32", 1, 4, 4, 32, 700, 512),
    W("cnt_G32_R32", 3, 64, 2, 1, 900, 512),
    W("cnt_mqa_8_chunks", 2, 128, 1, 1, 2000, 512),
]


def test_hd512_split_calls_back_to_back_and_graph_replays():
    """fmha_fwd at hd 512 with split KV (fp16 partials in the stream's workspace,
    then the merge as a programmatic dependent): calls of different shapes back
    to back on one stream, so that each reuses the workspace and its merge
    overlaps the next call's split kernel set-up, then one shape captured in a
    CUDA graph and replayed with fresh inputs, must each match the oracle."""
    stream = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(stream):
        for rep in range(2):
            for i, w in enumerate(BACK_TO_BACK_SHAPES):
                n, _, kern = binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, with_kernel=True)
                assert n > 1 and kern == "fwd_tc_wide", (w.name, n, kern)
                (q, k, v), (qd, kd, vd) = device_inputs(w, seed=40 + 7 * rep + i)
                o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, stream=stream)
                outs.append((w, q, k, v, o, lse))
    stream.synchronize()
    binding.fmha_check_device_status()
    for w, q, k, v, o, lse in outs:
        o_ref, lse_ref = oracle_full(w, q, k, v)
        compare(o, lse, o_ref, lse_ref, w.name)
        cosine_per_head(o, o_ref, w.name)

    w = BACK_TO_BACK_SHAPES[0]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=60)
    o = torch.empty_like(qd)
    lse = torch.empty(qd.shape[:3], dtype=torch.float32, device=qd.device)
    with torch.cuda.stream(stream):
        binding.fmha_fwd(qd, kd, vd, o, lse, scale=w.scale, stream=stream)  # workspaces exist before capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        binding.fmha_fwd(qd, kd, vd, o, lse, scale=w.scale, stream=stream)
    for rep in range(3):
        (q, k, v), _ = device_inputs(w, seed=61 + rep)
        qd.copy_(q.cuda())
        kd.copy_(k.cuda())
        vd.copy_(v.cuda())
        g.replay()
        torch.cuda.synchronize()
        binding.fmha_check_device_status()
        o_ref, lse_ref = oracle_full(w, q, k, v)
        compare(o, lse, o_ref, lse_ref, "graph replay %d" % rep)
