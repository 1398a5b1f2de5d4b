"""GPU parity of the two-row-tile tensor-core kernel (two 128-row query tiles
per thread block sharing every K/V tile, one softmax warpgroup per tile, P V
computed transposed for both tiles at once; hd 64 and 128) against the fp64
oracle.

Path 2 forces it wherever it applies (hd 64 or 128, more than 128 query rows per
KV head); the shapes cover GQA prefill, causal and window masks, row counts that
leave the last block with one row tile or a partial second tile, no key at
all, T > s_k, long KV ranges, split-KV partials and the attention sink.  The
NVFP4 output of such a shape runs the one-row-tile kernel (checked here too).
Path 4 (one row tile per block) must agree with it.
"""
import numpy as np
import pytest
import torch

import oracle
from check_utils import LSE_ATOL, compare, cosine_per_head, device_inputs, oracle_full, to_np_bits
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

PAIR_SHAPES = [
    W("p1_gqa8_T128_causal_hd128", 2, 16, 2, 128, 700, 128, causal=True),        # 1024 rows: 4 blocks
    W("p2_gqa4_T64_window_causal", 1, 8, 2, 64, 900, 128, window=333, causal=True),  # 256 rows
    W("p3_R384_last_block_one_tile", 1, 3, 1, 128, 500, 128, causal=True),       # 384 rows
    W("p4_R300_ragged", 1, 3, 1, 100, 333, 128),                                 # 300 rows
    W("p5_R200_partial_tile_b", 1, 2, 1, 100, 129, 128, window=50),              # 200 rows
    W("p6_no_key", 1, 4, 1, 70, 0, 128),                                         # O = 0, LSE = -inf
    W("p7_T_gt_sk", 1, 4, 2, 90, 40, 128),
    W("p8_mqa_G256_decode_hd128", 1, 256, 1, 1, 1000, 128),
    W("p9_long_sk", 1, 8, 1, 32, 5000, 128, causal=True),                        # 40 KV tiles
    W("p10_sharp_softmax", 1, 16, 2, 128, 2048, 128, k_mult=3.0),               # many rescales
    W("p11_window_only_hd128", 1, 4, 1, 128, 3000, 128, window=700),
    # hd 64: O^T is an M = 64 accumulator (the first 16 lanes of each TMEM quarter)
    W("p12_gqa8_T128_causal_hd64", 2, 16, 2, 128, 700, 64, causal=True),
    W("p13_R300_ragged_hd64", 1, 3, 1, 100, 333, 64),
    W("p14_window_causal_hd64", 1, 8, 2, 64, 900, 64, window=333, causal=True),
    W("p15_sharp_softmax_hd64", 1, 16, 2, 128, 2048, 64, k_mult=3.0),
    W("p16_no_key_hd64", 1, 4, 1, 70, 0, 64),
]


@pytest.fixture
def path():
    yield binding.fmha_set_kernel_path
    binding.fmha_set_kernel_path(0)


def _plan_kernel(w):
    return binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window, w.causal,
                                 with_kernel=True)[2]


@pytest.mark.parametrize("w", PAIR_SHAPES, ids=[w.name for w in PAIR_SHAPES])
def test_pair_kernel_matches_oracle(w, path):
    path(2)
    assert _plan_kernel(w) == "fwd_tc_pair"
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=21)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, w.name)
    if w.s_k > 0:
        cosine_per_head(o, o_ref, w.name)


@pytest.mark.parametrize("hd,chunk", [(128, 256), (128, 384), (128, 1000), (64, 256), (64, 640)])
def test_pair_kernel_partials(hd, chunk, path):
    """Split-KV partials of the pair kernel (fp32) and their merge."""
    path(2)
    w = W("pair_split", 1, 8, 2, 64, 1500, hd, window=1100, causal=True)
    assert _plan_kernel(w) == "fwd_tc_pair"
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=22)
    op, lp = binding.fmha_fwd_splitkv(qd, kd, vd, chunk, scale=w.scale, window=w.window, causal=w.causal)
    o, lse = binding.fmha_merge(op, lp)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    op_ref, lp_ref = oracle.partials(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, chunk, w.window,
                                     w.causal)
    compare(op, lp, op_ref, lp_ref, "pair partials hd %d chunk %d" % (hd, chunk))
    o_ref, lse_ref = oracle.merge(op_ref, lp_ref)
    compare(o, lse, o_ref, lse_ref, "pair merged hd %d chunk %d" % (hd, chunk))
    cosine_per_head(o, o_ref, "pair merged hd %d chunk %d" % (hd, chunk))


@pytest.mark.parametrize("hd", [64, 128])
def test_pair_kernel_sink(hd, path):
    path(2)
    w = W("pair_sink", 2, 16, 2, 32, 600, hd, causal=True)
    assert _plan_kernel(w) == "fwd_tc_pair"
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=23)
    g = torch.Generator().manual_seed(7)
    sink = torch.randn(w.n_h, generator=g, dtype=torch.float64) * 2.0
    sink[1::5] = -float("inf")
    sink = sink.float().double()
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, causal=True, sink=sink.float().cuda())
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle.attention(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, 0, True,
                                      sink=sink.numpy())
    compare(o, lse, o_ref, lse_ref, "pair sink")
    cosine_per_head(o, o_ref, "pair sink")


def _decode_scales(s):
    c = s.astype(np.int64)
    return np.where(c >> 3 == 0, (c & 7) / 8.0 * 2.0 ** -6, (1 + (c & 7) / 8.0) * np.exp2((c >> 3) - 7.0))


@pytest.mark.parametrize("g", [1.0, 0.25])
def test_pair_kernel_nvfp4(g, path):
    """NVFP4 output of a shape planned for the pair kernel (it runs the
    one-row-tile kernel, same chunks): dequantised values within the
    quantisation step of the oracle's O (as in test_nvfp4.py), block scales
    the oracle's code of the block amax or a neighbour, LSE within tolerance."""
    path(2)
    w = W("pair_fp4", 1, 16, 2, 64, 900, 128, causal=True)
    assert _plan_kernel(w) == "fwd_tc_pair"
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=24)
    codes, scales, lse = binding.fmha_fwd_nvfp4(qd, kd, vd, global_scale=g, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    deq = oracle.dequantize_nvfp4(codes, scales, g)
    st = np.repeat(_decode_scales(scales), 16, axis=-1) * g
    y = np.maximum(np.abs(o_ref), np.abs(deq)) / np.where(st > 0, st, 1.0)
    half_step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0)) * st
    assert (np.abs(deq - o_ref) <= half_step + 1e-2).all()
    _, s_ref = oracle.quantize_nvfp4(o_ref.astype(np.float32), g)
    diff = np.abs(scales.astype(np.int64) - s_ref.astype(np.int64))
    assert diff.max() <= 1 and (diff == 0).mean() >= 0.95
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_ATOL


def test_pair_and_one_tile_kernels_agree(path):
    w = W("pair_vs_tile", 1, 32, 4, 128, 1300, 128, causal=True)
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=25)
    outs = {}
    for which in (2, 4):
        path(which)
        o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, causal=True)
        torch.cuda.synchronize()
        binding.fmha_check_device_status()
        outs[which] = (o.float(), lse)
    assert (outs[2][0] - outs[4][0]).abs().max().item() <= 1.5e-2
    assert (outs[2][1] - outs[4][1]).abs().max().item() <= 1e-3
