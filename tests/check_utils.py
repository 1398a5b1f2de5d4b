"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the fp64 oracle on the same seeded bf16 inputs.

Tolerances (stated once, used everywhere):
  * max |O_gpu - O_oracle| <= 1.5e-2 over the bf16 output,
  * |LSE_gpu - LSE_oracle| <= 1e-3,
  * cosine(O_gpu, O_oracle) >= 0.99999 per (batch, head), over the T x hd block.
"""
import numpy as np
import torch

import oracle
from head_attention_forward_fmha_gb300 import inputs

O_ATOL = 1.5e-2
LSE_ATOL = 1e-3
COS_MIN = 0.99999


def to_np_bits(t):
    return inputs.bf16_bits(t.cpu())


def oracle_full(w, q, k, v):
    return oracle.attention(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, w.window, w.causal)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, label=""):
    """o_gpu: torch bf16/fp32 [..., hd]; lse_gpu torch fp32 [...]; refs float64 numpy."""
    og = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert og.shape == o_ref.shape, (og.shape, o_ref.shape)
    assert np.isfinite(og).all(), label + ": non-finite O"
    err = np.abs(og - o_ref).max() if og.size else 0.0
    assert err <= O_ATOL, "%s: max|dO| = %.3e > %.1e" % (label, err, O_ATOL)
    inf_ref = np.isinf(lse_ref)
    assert (np.isinf(lg) == inf_ref).all(), label + ": -inf LSE pattern differs"
    if (~inf_ref).any():
        lerr = np.abs(lg[~inf_ref] - lse_ref[~inf_ref]).max()
        assert lerr <= LSE_ATOL, "%s: max|dLSE| = %.3e > %.1e" % (label, lerr, LSE_ATOL)
    return err


def cosine_per_head(o_gpu, o_ref, label=""):
    """o: [b, n_h, T, hd]; cosine over T*hd per (b, h)."""
    og = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    b, n_h = og.shape[:2]
    a = og.reshape(b, n_h, -1)
    r = o_ref.reshape(b, n_h, -1)
    num = (a * r).sum(-1)
    den = np.sqrt((a * a).sum(-1) * (r * r).sum(-1))
    ok = den > 0
    cos = np.where(ok, num / np.where(ok, den, 1.0), 1.0)
    # rows whose reference is exactly zero must be zero on the GPU too
    assert (np.abs(a[~ok]) == 0).all() if (~ok).any() else True
    worst = cos.min() if cos.size else 1.0
    assert worst >= COS_MIN, "%s: min cosine %.7f < %.5f" % (label, worst, COS_MIN)
    return worst


def device_inputs(w, seed=0):
    q, k, v = inputs.make_inputs(w, seed)
    return (q, k, v), (q.cuda(), k.cuda(), v.cuda())
