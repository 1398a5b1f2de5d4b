"""NVFP4 output quantisation on the GPU against the oracle.

* The block quantiser the epilogues fuse, run on its own through the C ABI
  (fmha_quantize_nvfp4), gives the oracle's codes and scales bit for bit on
  the same fp32 inputs: both decide each code on the same fp32 numbers.
* fmha_fwd_nvfp4 on shapes that each kernel writes (decode, row-tile and hd-512
  tensor-core kernels, unsplit and through the merge): the dequantised output
  g * s * e is within the quantisation step of the oracle's fp64 O (half an
  E2M1 step at |O| / (g s), times g s, plus the 1e-2 allowed for the fp32 O
  the kernel quantises), the block scales are the oracle's E4M3 code of the
  block's amax or a neighbouring code, and the LSE meets the usual tolerance.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from check_utils import LSE_ATOL, device_inputs, oracle_full
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_hand_worked.json")


def _rows_for_bitwise():
    """fp32 rows of many magnitudes, the hand-worked blocks, exact midpoints
    of the E2M1 grid at several scales, zeros and huge values."""
    rng = np.random.default_rng(31)
    parts = [rng.standard_normal((512, 64)) * np.exp2(rng.uniform(-14, 12, (512, 1))),
             rng.uniform(-1, 1, (64, 64)) * 6.0,
             np.zeros((4, 64)),
             rng.standard_normal((8, 64)) * 1e6]
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    ties = np.concatenate([mids, -mids])[None, :] * np.exp2(np.arange(-8, 8))[:, None]
    parts.append(np.concatenate([ties, ties[:, ::-1], ties, -ties], axis=1))
    for c in json.load(open(GOLDEN))["cases"]:
        if c["global_scale"] == 1.0:
            x = np.asarray(c["x"])
            parts.append(np.tile(x, 64 // x.size)[None, :])
    return np.concatenate(parts).astype(np.float32)


@pytest.mark.parametrize("g", [1.0, 0.125, 3.0])
def test_block_quantiser_matches_oracle_bitwise(g):
    x = _rows_for_bitwise()
    codes, scales = binding.fmha_quantize_nvfp4(torch.from_numpy(x).cuda(), global_scale=g)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    c_ref, s_ref = oracle.quantize_nvfp4(x, g)
    np.testing.assert_array_equal(scales.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)


SHAPES = [
    # decode kernel, unsplit and split (merge of fp32 partials)
    W("dec_unsplit_hd128", 2, 8, 2, 1, 300, 128),
    W("dec_split_window", 1, 8, 1, 1, 4096, 128, window=3000),
    W("dec_hd64_T3_window_causal", 2, 6, 3, 3, 150, 64, window=40, causal=True),
    W("dec_hd64_R48_causal_long", 1, 8, 1, 6, 16500, 64, causal=True),
    W("dec_hd512", 1, 4, 4, 1, 100, 512),
    # row-tile tensor-core kernel, unsplit and split
    W("tc_causal_hd64", 1, 2, 2, 128, 300, 64, causal=True),
    W("tc_causal_hd256", 1, 4, 4, 64, 200, 256, causal=True),
    W("tc_split_mqa_hd128", 2, 128, 1, 1, 4096, 128),
    # hd-512 tensor-core kernel, unsplit and split (merge of fp16 partials)
    W("wide_hd512_T128", 1, 2, 2, 128, 130, 512),
    W("wide_split_mqa", 2, 128, 1, 1, 512, 512),
    W("wide_hd512_T32_q32", 4, 16, 16, 32, 512, 512, causal=True),
    # no key at all: O = 0 -> zero scales and codes, LSE = -inf
    W("no_key", 1, 2, 1, 2, 0, 64),
]


def _decode_scales(s):
    c = s.astype(np.int64)
    return np.where(c >> 3 == 0, (c & 7) / 8.0 * 2.0 ** -6, (1 + (c & 7) / 8.0) * np.exp2((c >> 3) - 7.0))


@pytest.mark.parametrize("g", [1.0, 0.25])
@pytest.mark.parametrize("w", SHAPES, ids=[w.name for w in SHAPES])
def test_fwd_nvfp4_matches_oracle(w, g):
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=41)
    codes, scales, lse = binding.fmha_fwd_nvfp4(qd, kd, vd, global_scale=g, scale=w.scale, window=w.window,
                                                causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    deq = oracle.dequantize_nvfp4(codes, scales, g)
    # quantisation step of each element at the GPU's block scale
    s = np.repeat(_decode_scales(scales), 16, axis=-1) * g
    y = np.maximum(np.abs(o_ref), np.abs(deq)) / np.where(s > 0, s, 1.0)
    half_step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0)) * s
    err = np.abs(deq - o_ref)
    assert (err <= half_step + 1e-2).all(), "%s: max excess %.3e" % (w.name, (err - half_step).max())
    # block scales: the oracle's code of the exact block amax, or a neighbour
    _, s_ref = oracle.quantize_nvfp4(o_ref.astype(np.float32), g)
    diff = np.abs(scales.astype(np.int64) - s_ref.astype(np.int64))
    assert diff.max() <= 1, w.name
    assert (diff == 0).mean() >= 0.95, "%s: %.3f of the scales agree" % (w.name, (diff == 0).mean())
    lg = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert (np.isinf(lg) == ~fin).all()
    if fin.any():
        assert np.abs(lg[fin] - lse_ref[fin]).max() <= LSE_ATOL


def test_fwd_nvfp4_lse_and_values_track_the_bf16_forward():
    """The NVFP4 forward runs the bf16 forward's split kernel: the same LSE up to
    the merge's summation order (the NVFP4 merge adds the chunk weights one
    thread at a time, the bf16 merge across a warp), and its dequantised output
    within one quantisation step of the bf16 O."""
    w = W("mqa_hd512", 4, 128, 1, 1, 512, 512)
    (_, _, _), (qd, kd, vd) = device_inputs(w, seed=42)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale)
    codes, scales, lse4 = binding.fmha_fwd_nvfp4(qd, kd, vd, scale=w.scale)
    torch.cuda.synchronize()
    assert (lse - lse4).abs().max().item() <= 1e-5
    deq = oracle.dequantize_nvfp4(codes.cpu().numpy(), scales.cpu().numpy())
    s = np.repeat(_decode_scales(scales.cpu().numpy()), 16, axis=-1)
    ob = o.float().cpu().numpy()
    assert (np.abs(deq - ob) <= 1.0 * s + 2e-2).all()
