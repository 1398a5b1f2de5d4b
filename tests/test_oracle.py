"""Pins of the fp64 oracle to things other than itself (CPU only).

Each pin checks the oracle against what the pages or the mathematics fix:
hand-worked closed forms (``tests/golden/hand_worked.json``), an independent
brute-force evaluation on tiny shapes, invariants (softmax rows sum to one,
uniform V returns V, key permutation invariance), closed forms (Q = 0 gives
lse = ln|J| and the mean of the attended V rows; one dominant key returns its V
row), split-KV merge equal to the single pass, and the unmasked case equal to
``torch.softmax`` in float64; with an attention sink (the reading the oracle
states: one more logit in the denominator only) the same brute force with the
sink's column, Q = 0 giving lse = ln(n + e^sigma), sigma = -inf equal to no
sink, an empty key range giving lse = sigma, and the split merge adding the
sink once; for the NVFP4 output quantisation (the format the oracle states)
hand-worked blocks (``tests/golden/nvfp4_hand_worked.json``), the E2M1
rounding against a construction from Python's round-half-even, the E4M3 scale
against torch's float8_e4m3fn cast, exact round trips of representable blocks
and the half-step error bound.  ``test_pins_catch_planted_mistakes`` plants
plausible mistakes in a copy of the oracle's C source and checks that the pins
reject every one.
"""
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from head_attention_forward_fmha_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_SRC = os.path.join(os.path.dirname(HERE), "oracle", "fmha_oracle.c")


def _arr(spec, n):
    if spec == "zeros":
        return np.zeros(n)
    if spec == "ones":
        return np.ones(n)
    return np.asarray(spec, dtype=np.float64)


# ----------------------------------------------------------------------------
# independent brute force: materialise the score matrix and the mask matrix
# ----------------------------------------------------------------------------
def brute_force(q, k, v, scale, window, causal, sink=None):
    """sink: optional [n_h] logits, one more column of the score matrix whose
    value row is zero."""
    b, n_h, T, hd = q.shape
    _, n_kv_h, s_k, _ = k.shape
    G = n_h // n_kv_h
    o = np.zeros((b, n_h, T, hd))
    lse = np.zeros((b, n_h, T))
    for bi in range(b):
        for h in range(n_h):
            kh = h // G
            S = np.zeros((T, s_k))
            allowed = np.zeros((T, s_k), dtype=bool)
            for t in range(T):
                pos = s_k - T + t
                for j in range(s_k):
                    S[t, j] = scale * sum(float(q[bi, h, t, d]) * float(k[bi, kh, j, d]) for d in range(hd))
                    ok = True
                    if causal and j > pos:
                        ok = False
                    if window > 0 and j <= pos - window:
                        ok = False
                    allowed[t, j] = ok
            sg = -math.inf if sink is None else float(sink[h])
            for t in range(T):
                idx = [j for j in range(s_k) if allowed[t, j]]
                if not idx:
                    lse[bi, h, t] = sg
                    continue
                mx = max([S[t, j] for j in idx] + [sg])
                e = {j: math.exp(S[t, j] - mx) for j in idx}
                tot = sum(e.values()) + (0.0 if sg == -math.inf else math.exp(sg - mx))
                for d in range(hd):
                    o[bi, h, t, d] = sum(e[j] / tot * float(v[bi, kh, j, d]) for j in idx)
                lse[bi, h, t] = mx + math.log(tot)
    return o, lse


# ----------------------------------------------------------------------------
# pins: each raises AssertionError when the oracle disagrees
# ----------------------------------------------------------------------------
def pin_golden_cases():
    data = json.load(open(GOLDEN))
    for c in data["cases"]:
        sh = c["shape"]
        q = _arr(c["q"], sh["batch"] * sh["n_h"] * sh["T"] * sh["hd"]).reshape(
            sh["batch"], sh["n_h"], sh["T"], sh["hd"])
        nkv = sh["batch"] * sh["n_kv_h"] * sh["s_k"] * sh["hd"]
        k = _arr(c["k"], nkv).reshape(sh["batch"], sh["n_kv_h"], sh["s_k"], sh["hd"])
        v = _arr(c["v"], nkv).reshape(k.shape)
        o, lse = oracle.attention(q, k, v, c["scale"], c["window"], c["causal"])
        np.testing.assert_allclose(o.ravel(), c["expect"]["o"], rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse.ravel(), c["expect"]["lse"], rtol=0, atol=1e-12, err_msg=c["name"])
    for c in data["merge_cases"]:
        op = np.asarray(c["o_parts"], dtype=np.float64).reshape(len(c["o_parts"]), 1, c["hd"])
        lp = np.asarray([float(x) for x in c["lse_parts"]], dtype=np.float64).reshape(-1, 1)
        o, lse = oracle.merge(op, lp)
        np.testing.assert_allclose(o.ravel(), c["expect"]["o"], rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse.ravel(), c["expect"]["lse"], rtol=0, atol=1e-12, err_msg=c["name"])


TINY = [
    # batch, n_h, n_kv_h, T, s_k, hd, window, causal
    (1, 1, 1, 1, 1, 1, 0, False),
    (1, 2, 1, 3, 5, 2, 0, True),
    (2, 4, 2, 5, 9, 3, 3, True),
    (1, 4, 4, 2, 7, 64, 0, False),
    (2, 2, 1, 4, 6, 2, 2, False),
    (1, 3, 1, 5, 5, 4, 1, True),
    (1, 2, 2, 6, 4, 2, 0, False),   # T > s_k, no causal
]


def pin_brute_force_tiny():
    rng = np.random.default_rng(1)
    for (b, n_h, n_kv_h, T, s_k, hd, window, causal) in TINY:
        q = rng.standard_normal((b, n_h, T, hd))
        k = rng.standard_normal((b, n_kv_h, s_k, hd)) * 2.0
        v = rng.standard_normal((b, n_kv_h, s_k, hd))
        scale = 0.7
        o, lse = oracle.attention(q, k, v, scale, window, causal)
        ob, lb = brute_force(q, k, v, scale, window, causal)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isinf(lse), np.isinf(lb))
        fin = np.isfinite(lb)
        np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-12)


def pin_softmax_rows_sum_to_one():
    # V = identity over keys: O[t, j] is the softmax weight P[t, j].
    rng = np.random.default_rng(2)
    for window, causal in ((0, False), (3, False), (0, True), (4, True)):
        s_k, hd = 12, 16
        q = rng.standard_normal((1, 2, 4, hd))
        k = rng.standard_normal((1, 1, s_k, hd))
        v = np.zeros((1, 1, s_k, hd))
        for j in range(s_k):
            v[0, 0, j, j] = 1.0
        o, _ = oracle.attention(q, k, v, 0.5, window, causal)
        assert (o >= 0).all()
        np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-12)
        # masked keys get exactly zero weight
        for t in range(4):
            pos = s_k - 4 + t
            for j in range(s_k):
                masked = (causal and j > pos) or (window > 0 and j <= pos - window)
                if masked:
                    assert (o[0, :, t, j] == 0).all()
                else:
                    assert (o[0, :, t, j] > 0).all()


def pin_uniform_v_returns_v():
    rng = np.random.default_rng(3)
    for (b, n_h, n_kv_h, T, s_k, hd, window, causal) in TINY[1:] + [(2, 8, 2, 3, 40, 8, 7, True)]:
        q = rng.standard_normal((b, n_h, T, hd)) * 3
        k = rng.standard_normal((b, n_kv_h, s_k, hd))
        c = rng.standard_normal(hd)
        v = np.broadcast_to(c, (b, n_kv_h, s_k, hd)).copy()
        o, lse = oracle.attention(q, k, v, 1.0, window, causal)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)


def pin_key_permutation_invariance():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((2, 4, 3, 8))
    k = rng.standard_normal((2, 2, 17, 8))
    v = rng.standard_normal((2, 2, 17, 8))
    perm = rng.permutation(17)
    o1, l1 = oracle.attention(q, k, v, 0.4)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def pin_q_zero_closed_form():
    # q = 0: every attended score is 0, lse = ln|J| and O = mean of attended V.
    rng = np.random.default_rng(5)
    # causal prefill layout: 8 new queries after 24 cached keys
    T, s_k, hd = 8, 32, 4
    q = np.zeros((1, 2, T, hd))
    k = rng.standard_normal((1, 2, s_k, hd))
    v = rng.standard_normal((1, 2, s_k, hd))
    o, lse = oracle.attention(q, k, v, 0.3, 0, True)
    for t in range(T):
        n = s_k - T + t + 1
        np.testing.assert_allclose(lse[0, :, t], math.log(n), rtol=0, atol=1e-12)
        np.testing.assert_allclose(o[0, :, t], v[0, :, :n].mean(axis=1), rtol=0, atol=1e-12)
    # sliding window, decode: lse = ln(window), O = mean of the last `window` rows
    o, lse = oracle.attention(q[:, :, :1], k, v, 0.3, 5, False)
    np.testing.assert_allclose(lse, math.log(5), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[0, :, 0], v[0, :, s_k - 5:].mean(axis=1), rtol=0, atol=1e-12)


def pin_dominant_key():
    rng = np.random.default_rng(6)
    s_k, hd = 20, 8
    k = rng.standard_normal((1, 1, s_k, hd)) * 0.01
    v = rng.standard_normal((1, 1, s_k, hd))
    jstar = 13
    q = np.zeros((1, 1, 1, hd))
    q[0, 0, 0, 0] = 1.0
    k[0, 0, jstar, 0] = 100.0
    o, lse = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, jstar], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0, 0], float(q[0, 0, 0] @ k[0, 0, jstar]), rtol=0, atol=1e-12)


def pin_single_attended_key():
    # window 1: each row attends exactly its own position
    rng = np.random.default_rng(7)
    T, s_k, hd = 3, 6, 5
    q = rng.standard_normal((1, 1, T, hd))
    k = rng.standard_normal((1, 1, s_k, hd))
    v = rng.standard_normal((1, 1, s_k, hd))
    o, lse = oracle.attention(q, k, v, 0.9, 1, True)
    for t in range(T):
        j = s_k - T + t
        np.testing.assert_allclose(o[0, 0, t], v[0, 0, j], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, 0, t], 0.9 * float(q[0, 0, t] @ k[0, 0, j]), rtol=0, atol=1e-12)


def pin_split_merge_equals_single_pass():
    rng = np.random.default_rng(8)
    for (T, s_k, window, causal) in ((1, 600, 0, False), (4, 300, 100, True), (3, 257, 0, True)):
        q = rng.standard_normal((1, 4, T, 8))
        k = rng.standard_normal((1, 2, s_k, 8))
        v = rng.standard_normal((1, 2, s_k, 8))
        o, lse = oracle.attention(q, k, v, 0.35, window, causal)
        for chunk in (1, 7, 128, 512, s_k):
            op, lp = oracle.partials(q, k, v, 0.35, chunk, window, causal)
            om, lm = oracle.merge(op, lp)
            np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)


def pin_split_layout():
    # chunks start at the first key row 0 attends and cover every attended key
    assert oracle.split_layout(1, 8192, 4096, 512) == (4096, 8)
    assert oracle.split_layout(1, 512, 0, 512) == (0, 1)
    assert oracle.split_layout(128, 512, 0, 100) == (0, 6)
    assert oracle.split_layout(4, 100, 10, 3) == (87, 5)


def pin_torch_softmax_unmasked():
    # special case that reduces to a library routine: T = 1, no mask
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 6, 1, 16))
    k = rng.standard_normal((2, 3, 33, 16))
    v = rng.standard_normal((2, 3, 33, 16))
    o, lse = oracle.attention(q, k, v, 0.25)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    tk = tk.repeat_interleave(2, dim=1)
    tv = tv.repeat_interleave(2, dim=1)
    s = (tq @ tk.transpose(-1, -2)) * 0.25
    np.testing.assert_allclose(o, (torch.softmax(s, -1) @ tv).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def pin_bf16_widening_is_exact():
    w = inputs.Workload("t", 1, 2, 1, 2, 40, 64, window=9, causal=True)
    q, k, v = inputs.make_inputs(w, seed=11)
    o1, l1 = oracle.attention(inputs.bf16_bits(q), inputs.bf16_bits(k), inputs.bf16_bits(v),
                              w.scale, w.window, w.causal)
    o2, l2 = oracle.attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                              w.scale, w.window, w.causal)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def pin_rows_api_matches_full():
    w = inputs.Workload("t", 2, 4, 2, 3, 50, 16, window=20, causal=True)
    q, k, v = (inputs.bf16_bits(x) for x in inputs.make_inputs(w, seed=12))
    o, lse = oracle.attention(q, k, v, w.scale, w.window, w.causal)
    rows = np.array([0, 5, 7, 23], dtype=np.int64)
    orow, lrow = oracle.attention_rows(q, k, v, rows, w.scale, w.window, w.causal)
    np.testing.assert_array_equal(orow, o.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(lrow, lse.reshape(-1)[rows])


SINKS = [None, "zero", "neg_inf", "big", "mixed"]


def _sinks(kind, n_h, rng):
    if kind is None:
        return None
    if kind == "zero":
        return np.zeros(n_h)
    if kind == "neg_inf":
        return np.full(n_h, -np.inf)
    if kind == "big":
        return np.full(n_h, 30.0)  # dominates every score
    return rng.standard_normal(n_h) * 2.0 + np.arange(n_h)  # a different logit per head


def pin_sink_brute_force_tiny():
    rng = np.random.default_rng(11)
    for (b, n_h, n_kv_h, T, s_k, hd, window, causal) in TINY:
        for kind in SINKS[1:]:
            q = rng.standard_normal((b, n_h, T, hd))
            k = rng.standard_normal((b, n_kv_h, s_k, hd)) * 2.0
            v = rng.standard_normal((b, n_kv_h, s_k, hd))
            sink = _sinks(kind, n_h, rng)
            o, lse = oracle.attention(q, k, v, 0.7, window, causal, sink=sink)
            ob, lb = brute_force(q, k, v, 0.7, window, causal, sink=sink)
            np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12, err_msg=kind)
            np.testing.assert_array_equal(np.isinf(lse), np.isinf(lb))
            fin = np.isfinite(lb)
            np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-12, err_msg=kind)


def pin_sink_q_zero_closed_form():
    # all n scores 0: l = n + e^sigma, O = sum_j v_j / (n + e^sigma)
    rng = np.random.default_rng(12)
    n, hd = 9, 5
    v = rng.standard_normal((1, 1, n, hd))
    for sg in (-3.0, 0.0, 1.5, 20.0):
        o, lse = oracle.attention(np.zeros((1, 1, 1, hd)), rng.standard_normal((1, 1, n, hd)), v, 0.3,
                                  sink=[sg])
        np.testing.assert_allclose(lse.ravel(), [math.log(n + math.exp(sg))], rtol=0, atol=1e-12)
        np.testing.assert_allclose(o.ravel(), v.sum(axis=2).ravel() / (n + math.exp(sg)), rtol=0, atol=1e-12)


def pin_sink_neg_inf_is_no_sink():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((2, 4, 3, 8))
    k = rng.standard_normal((2, 2, 11, 8))
    v = rng.standard_normal((2, 2, 11, 8))
    o0, l0 = oracle.attention(q, k, v, 0.4, 5, True)
    o1, l1 = oracle.attention(q, k, v, 0.4, 5, True, sink=np.full(4, -np.inf))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


def pin_sink_empty_key_range():
    # no attended key: O = 0 and lse = sigma (the sink alone is the denominator)
    rng = np.random.default_rng(14)
    q = rng.standard_normal((1, 3, 2, 4))
    k = rng.standard_normal((1, 1, 6, 4))
    sink = np.array([-1.0, 0.5, 7.0])
    o, lse = oracle.attention(q, k, k, 1.0, key_begin=3, key_end=3, sink=sink)
    np.testing.assert_array_equal(o, np.zeros_like(o))
    np.testing.assert_array_equal(lse, np.repeat(sink[None, :, None], 2, axis=2))


def pin_sink_split_merge_equals_single_pass():
    # partials carry no sink; the merge adds it once
    rng = np.random.default_rng(15)
    q = rng.standard_normal((2, 4, 3, 6))
    k = rng.standard_normal((2, 2, 40, 6)) * 1.5
    v = rng.standard_normal((2, 2, 40, 6))
    sink = rng.standard_normal(4) * 3.0
    o1, l1 = oracle.attention(q, k, v, 0.5, 25, True, sink=sink)
    rows_sink = np.broadcast_to(sink[None, :, None], l1.shape)
    for chunk in (1, 7, 16, 40):
        op, lp = oracle.partials(q, k, v, 0.5, chunk, 25, True)
        om, lm = oracle.merge(op, lp, sink=rows_sink)
        np.testing.assert_allclose(om, o1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lm, l1, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# NVFP4 quantisation (the format the oracle states: 16-element blocks, E2M1
# codes, E4M3 scale of amax / (6 g), both roundings to nearest-even, saturating)
# ----------------------------------------------------------------------------
NVFP4_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_hand_worked.json")


def pin_nvfp4_golden_blocks():
    for c in json.load(open(NVFP4_GOLDEN))["cases"]:
        x = np.asarray(c["x"], dtype=np.float32)[None]
        codes, scales = oracle.quantize_nvfp4(x, c["global_scale"])
        assert list(scales[0]) == c["scales"], (c["name"], list(scales[0]))
        assert list(codes[0]) == c["codes"], (c["name"], list(codes[0]))


def _e2m1_by_round(a):
    """E2M1 magnitude code of a >= 0 built from Python's round() (half to even)
    on the exponent / mantissa view: step 0.5 below 2, 1 in [2, 4), 2 in [4, 6]."""
    if a >= 6.0:
        return 7
    if a < 2.0:
        return round(a * 2.0)           # codes 0..4 are 0, 0.5, 1, 1.5, 2
    if a < 4.0:
        return round(a) + 2             # 2, 3, 4 -> codes 4, 5, 6
    return 6 if round(a / 2.0) == 2 else 7


def pin_nvfp4_e2m1_rounding_matches_round_half_even():
    rng = np.random.default_rng(21)
    ys = np.concatenate([rng.uniform(0, 6, 600), np.arange(0, 6.01, 0.25)]).astype(np.float32)
    # one block per value: amax 6 (s = 1) so the element is quantised as is
    # (saturation beyond 6 is covered by the hand-worked blocks)
    x = np.zeros((ys.size, 16), np.float32)
    x[:, 0] = 6.0
    x[:, 1] = ys
    codes, scales = oracle.quantize_nvfp4(x)
    assert (scales == 56).all()
    got = (codes[:, 0] >> 4) & 7
    want = np.array([_e2m1_by_round(float(y)) for y in ys])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(ys[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def pin_nvfp4_e4m3_scale_matches_torch_float8():
    # amax / 6 for amax = 6 v is exactly v when v has at most 20 significant
    # bits; torch's float8_e4m3fn cast (round-to-nearest-even) gives its code
    rng = np.random.default_rng(22)
    v = np.concatenate([np.exp2(rng.uniform(-11, 8.8, 800)), [2.0 ** -10, 3 * 2.0 ** -11, 1.0625, 1.1875, 240.0]])
    v = v[v <= 448.0]
    m, e = np.frexp(v)
    v = np.ldexp(np.round(m * 2 ** 20) / 2 ** 20, e).astype(np.float32)
    x = np.zeros((v.size, 16), np.float32)
    x[:, 3] = 6.0 * v
    assert (x[:, 3] / np.float32(6.0) == v).all()
    _, scales = oracle.quantize_nvfp4(x)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(scales[:, 0] != want)[0]
    assert bad.size == 0, [(float(v[i]), int(scales[i, 0]), int(want[i])) for i in bad[:5]]


def pin_nvfp4_round_trip_of_representable_blocks():
    # blocks of s * E2M1 values with s an E4M3 value and amax = 6 s come back exactly
    rng = np.random.default_rng(23)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for trial in range(50):
        s = float(np.ldexp(1.0 + rng.integers(0, 8) / 8.0, int(rng.integers(-6, 6))))
        g = float(rng.choice([0.5, 1.0, 4.0]))
        e = grid[rng.integers(0, 8, 32)] * rng.choice([-1.0, 1.0], 32)
        e[0], e[16] = 6.0, -6.0
        x = (g * s * e).astype(np.float32)[None]
        codes, scales = oracle.quantize_nvfp4(x, g)
        np.testing.assert_array_equal(oracle.dequantize_nvfp4(codes, scales, g), x.astype(np.float64))


def pin_nvfp4_error_bound_on_random_rows():
    # |x - deq| <= half the E2M1 step at |x| / (g s), times g s, away from saturation
    rng = np.random.default_rng(24)
    x = (rng.standard_normal((64, 64)) * np.exp2(rng.uniform(-4, 4, (64, 1)))).astype(np.float32)
    codes, scales = oracle.quantize_nvfp4(x, 1.0)
    deq = oracle.dequantize_nvfp4(codes, scales, 1.0)
    c = scales.astype(np.int64)
    s = np.where(c >> 3 == 0, (c & 7) / 8.0 * 2.0 ** -6, (1 + (c & 7) / 8.0) * np.exp2((c >> 3) - 7.0))
    s = np.repeat(s, 16, axis=-1)
    y = np.abs(x) / s
    half_step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
    inside = y <= 6.0
    assert (np.abs(x - deq)[inside] <= (half_step * s)[inside] * (1 + 1e-6)).all()


ALL_PINS = [pin_golden_cases, pin_brute_force_tiny, pin_softmax_rows_sum_to_one,
            pin_uniform_v_returns_v, pin_key_permutation_invariance, pin_q_zero_closed_form,
            pin_dominant_key, pin_single_attended_key, pin_split_merge_equals_single_pass,
            pin_split_layout, pin_torch_softmax_unmasked, pin_bf16_widening_is_exact,
            pin_rows_api_matches_full, pin_sink_brute_force_tiny, pin_sink_q_zero_closed_form,
            pin_sink_neg_inf_is_no_sink, pin_sink_empty_key_range, pin_sink_split_merge_equals_single_pass,
            pin_nvfp4_golden_blocks, pin_nvfp4_e2m1_rounding_matches_round_half_even,
            pin_nvfp4_e4m3_scale_matches_torch_float8, pin_nvfp4_round_trip_of_representable_blocks,
            pin_nvfp4_error_bound_on_random_rows]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin()


# ----------------------------------------------------------------------------
# planted mistakes: each mutant of the oracle source must fail at least one pin
# ----------------------------------------------------------------------------
MUTANTS = {
    "dropped_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "gqa_modulo_map": ("int kvh = h / group;", "int kvh = h % n_kv_h;"),
    "causal_off_by_one": ("if (causal && p < h) h = p;", "if (causal && p - 1 < h) h = p - 1;"),
    "window_off_by_one": ("l = p - window + 1;", "l = p - window;"),
    "top_left_alignment": ("long p = (long)s_k - T + t;", "long p = t;"),
    "lse_missing_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "double_divide": ("double w = exp(s[j] - m) / l;", "double w = exp(s[j] - m) / l / l;"),
    "v_for_k": ("dot += qd[d] * load_elem(k, kj", "dot += qd[d] * load_elem(v, kj"),
    "merge_plain_mean": ("double w = exp(lse_parts[(size_t)i * rows + r] - mx) / den;",
                         "double w = 1.0 / n_splits;"),
    "merge_lse_log2": ("lse[r] = mx + log(den);", "lse[r] = mx + log2(den);"),
    "sink_unshifted": ("if (sink != -INFINITY) l += exp(sink - m);", "if (sink != -INFINITY) l += exp(sink);"),
    "sink_per_kv_head": ("sink ? sink[h] : -INFINITY", "sink ? sink[kvh] : -INFINITY"),
    "sink_empty_row_lse": ("*lse_out = sink;  /* -inf without a sink */", "*lse_out = -INFINITY;"),
    "merge_sink_dropped": ("if (sg != -INFINITY) den += exp(sg - mx);", ";"),
    "nvfp4_e2m1_ties_up": ("if (d_new < d_best || (d_new == d_best && (c & 1) == 0)) best = c;\n    }\n    return best;\n}\n\n/* x:",
                           "if (d_new <= d_best) best = c;\n    }\n    return best;\n}\n\n/* x:"),
    "nvfp4_e4m3_ties_up": ("if (d_new < d_best || (d_new == d_best && (c & 1) == 0)) best = c;\n    }\n    return best;\n}\n\nstatic const",
                           "if (d_new <= d_best) best = c;\n    }\n    return best;\n}\n\nstatic const"),
    "nvfp4_amax_over_4": ("const float six_g = 6.0f * g;", "const float six_g = 4.0f * g;"),
    "nvfp4_half_block_amax": ("for (int i = 0; i < 16; ++i)\n                if (fabsf(xb[i]) > amax)",
                              "for (int i = 0; i < 8; ++i)\n                if (fabsf(xb[i]) > amax)"),
    "nvfp4_sign_dropped": ("if (y < 0.0f && code != 0) code |= 8;", ";"),
    "nvfp4_nibble_order": ("(uint8_t)(nib[0] | (nib[1] << 4))", "(uint8_t)(nib[1] | (nib[0] << 4))"),
    "nvfp4_e4m3_no_saturation": ("for (int c = 1; c <= 0x7E; ++c)", "for (int c = 1; c <= 0x7F; ++c)"),
    "nvfp4_global_scale_ignored": ("const float gs = g * s;", "const float gs = s;"),
    "merge_sink_in_numerator": ("        if (sg != -INFINITY) den += exp(sg - mx);",
                                "        if (sg != -INFINITY) { den += exp(sg - mx); orow[0] += exp(sg - mx); }"),
}


def _build_mutant(src_text, tmpdir, name):
    path = os.path.join(tmpdir, name + ".c")
    with open(path, "w") as f:
        f.write(src_text)
    lib = os.path.join(tmpdir, "lib" + name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", path, "-o", lib, "-lm"], check=True)
    return lib


def test_pins_catch_planted_mistakes():
    src = open(ORACLE_SRC).read()
    tmpdir = tempfile.mkdtemp(prefix="oracle_mutants_")
    saved = oracle._lib
    survivors = []
    try:
        for name, (old, new) in MUTANTS.items():
            assert src.count(old) == 1, "mutation target not found exactly once: " + name
            lib = _build_mutant(src.replace(old, new), tmpdir, name)
            oracle._lib = oracle._bind(lib)
            caught = False
            for pin in ALL_PINS:
                try:
                    pin()
                except (AssertionError, ValueError):
                    caught = True
                    break
            if not caught:
                survivors.append(name)
    finally:
        oracle._lib = saved
        shutil.rmtree(tmpdir, ignore_errors=True)
    assert not survivors, "planted mistakes no pin rejects: %s" % survivors
