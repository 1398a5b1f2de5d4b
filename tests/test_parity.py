"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every case draws seeded bf16 inputs, runs the library, runs the oracle on the
same bits and compares element by element (tolerances in ``check_utils``).
The named workloads run at their full sizes with the full oracle; the MHA
shape sweep runs at full size and checks a sample of rows computed one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from check_utils import compare, cosine_per_head, device_inputs, oracle_full, to_np_bits
from head_attention_forward_fmha_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

SMALL = [
    # name, batch, n_h, n_kv_h, T, s_k, hd, window, causal
    W("s1_tiny_sk1", 1, 1, 1, 1, 1, 64),
    W("s2_sk_below_tile", 2, 4, 2, 1, 37, 128),
    W("s3_ragged_tail", 2, 8, 2, 1, 200, 64),
    W("s4_gqa8", 2, 16, 2, 1, 300, 128),
    W("s5_mqa_hd256", 1, 16, 1, 1, 129, 256),
    W("s6_hd512", 1, 4, 4, 1, 100, 512),
    W("s7_T4_causal", 2, 8, 8, 4, 70, 64, causal=True),
    W("s8_T3_window", 1, 4, 2, 3, 90, 128, window=17),
    W("s9_T5_window_causal", 2, 6, 3, 5, 150, 256, window=40, causal=True),
    W("s10_T32_causal", 1, 4, 4, 32, 96, 128, causal=True),
    W("s11_T128_causal", 1, 2, 2, 128, 300, 64, causal=True),
    W("s12_T128_hd512", 1, 2, 2, 128, 130, 512),
    W("s13_T_gt_sk", 1, 2, 1, 7, 3, 64),
    W("s14_sk0", 1, 2, 1, 2, 0, 64),  # no cached key at all: O = 0, LSE = -inf
    W("s15_T17_G3_window_causal", 1, 6, 2, 17, 64, 128, window=8, causal=True),
    W("s16_window1", 1, 2, 2, 3, 50, 64, window=1, causal=True),
    W("s17_gqa16_T2", 1, 32, 2, 2, 513, 128, window=300),
    W("s18_hd256_T128_window", 1, 2, 1, 128, 700, 256, window=100, causal=True),
    W("s19_long_sk", 1, 4, 1, 1, 5000, 128),
    W("s20_mqa_G128_hd128", 2, 128, 1, 1, 257, 128),
    # 32-row decode blocks: hd 64, 17 to 63 rows per KV head, >= 16384 attended keys
    W("s21_hd64_T32_causal_long", 1, 4, 4, 32, 16400, 64, causal=True),
    W("s22_hd64_R40_window_long", 1, 8, 2, 10, 20000, 64, window=16380),
    W("s23_hd64_R24_window_causal", 2, 6, 2, 8, 200, 64, window=50, causal=True),  # 16-row blocks
    W("s24_hd64_R63_long", 1, 9, 1, 7, 16500, 64),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_fwd_small_shapes(w):
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=1)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, w.name)
    cosine_per_head(o, o_ref, w.name)


NAMED = ["single_head_decode", "mqa_decode", "gqa_swa_decode", "causal_prefill"]


@pytest.mark.parametrize("name", NAMED)
def test_fwd_named_workloads_full_oracle(name):
    w = inputs.WORKLOADS[name]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=0)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, name)
    cosine_per_head(o, o_ref, name)


def test_mqa_decode_uniform_v_returns_v():
    w = inputs.WORKLOADS["mqa_decode_vconst"]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=0)
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale)
    torch.cuda.synchronize()
    c = v[0, 0, 0].double().numpy()
    err = np.abs(o.double().cpu().numpy() - c).max()
    # P is rounded to bf16 before PV while the sum uses fp32 P: |O - c| <= |c| * 2^-8
    assert err <= max(1e-2, 2.0 ** -8 * np.abs(c).max()), err
    _, lse_ref = oracle_full(w, q, k, v)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


def test_gqa_swa_decode_split_512_matches_oracle_partials_and_merge():
    w = inputs.WORKLOADS["gqa_swa_decode"]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=2)
    op, lp = binding.fmha_fwd_splitkv(qd, kd, vd, 512, scale=w.scale, window=w.window, causal=w.causal)
    o, lse = binding.fmha_merge(op, lp)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    assert op.shape[0] == 8
    # partials of two chunks against the oracle restricted to those keys
    for i in (0, 7):
        lo = 4096 + 512 * i
        o_i, l_i = oracle.attention(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, w.window, w.causal,
                                    key_begin=lo, key_end=lo + 512)
        compare(op[i], lp[i], o_i, l_i, "partial %d" % i)
    o_ref, lse_ref = oracle_full(w, q, k, v)
    compare(o, lse, o_ref, lse_ref, "merged")
    cosine_per_head(o, o_ref, "merged")


SPLIT_CASES = [
    (W("sp1", 1, 4, 2, 1, 40, 64), 1),
    (W("sp2", 2, 4, 1, 3, 300, 128, window=100, causal=True), 7),
    (W("sp3", 1, 8, 8, 4, 257, 256, causal=True), 64),
    (W("sp4", 1, 2, 1, 2, 200, 512), 100),
    (W("sp5", 1, 16, 2, 1, 129, 128), 129),
    (W("sp6_hd64_R32_long", 1, 8, 2, 8, 17000, 64, causal=True), 4096),
]


@pytest.mark.parametrize("w,chunk", SPLIT_CASES, ids=[c[0].name for c in SPLIT_CASES])
def test_splitkv_partials_and_merge(w, chunk):
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=3)
    op, lp = binding.fmha_fwd_splitkv(qd, kd, vd, chunk, scale=w.scale, window=w.window, causal=w.causal)
    o, lse = binding.fmha_merge(op, lp)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    op_ref, lp_ref = oracle.partials(to_np_bits(q), to_np_bits(k), to_np_bits(v), w.scale, chunk, w.window,
                                     w.causal)
    assert op.shape[0] == op_ref.shape[0]
    compare(op, lp, op_ref, lp_ref, w.name + " partials")
    o_ref, lse_ref = oracle.merge(op_ref, lp_ref)
    compare(o, lse, o_ref, lse_ref, w.name + " merged")
    # and the merged result equals the single pass
    o1, l1 = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
    torch.cuda.synchronize()
    assert (o1.float() - o.float()).abs().max().item() <= 1.5e-2
    assert (l1 - lse).abs().max().item() <= 1e-3


@pytest.mark.parametrize("hd", [64, 128, 256, 512])
def test_merge_kernel_against_oracle(hd):
    g = torch.Generator().manual_seed(hd)
    n, b, n_h, T = 5, 2, 3, 4
    # partial outputs are convex combinations of N(0,1) V rows: |O_i| < 4, where
    # bf16 rounding of the merged output stays inside the 1.5e-2 bound
    op = torch.randn((n, b, n_h, T, hd), generator=g).clamp_(-3.9, 3.9)
    lp = torch.randn((n, b, n_h, T), generator=g) * 3
    lp[1, 0, 0, 0] = -math.inf          # one empty partial
    lp[:, 1, 2, 3] = -math.inf          # a row with no key at all
    op[:, 1, 2, 3] = 0
    o, lse = binding.fmha_merge(op.cuda(), lp.cuda())
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge(op.double().numpy(), lp.double().numpy())
    compare(o, lse, o_ref, lse_ref, "merge hd%d" % hd)


SWEEP = inputs.sweep()


def _sweep_slabs(w, n, seed):
    """n distinct (batch, head) pairs: the first, the last and seeded others."""
    rng = np.random.default_rng(seed)
    pairs = [(0, 0), (w.batch - 1, w.n_h - 1)]
    while len(pairs) < n:
        p = (int(rng.integers(w.batch)), int(rng.integers(w.n_h)))
        if p not in pairs:
            pairs.append(p)
    return pairs


@pytest.mark.parametrize("w", SWEEP, ids=[w.name for w in SWEEP])
def test_sweep_full_size_sampled_rows(w):
    """Full-size run; the oracle recomputes 48 sampled rows plus every row of
    four whole (batch, head) slabs, so that all three tolerances -- max |dO|,
    |dLSE| and the per-(batch, head) cosine over the T x hd block -- are
    asserted at every point of the sweep."""
    qd, kd, vd = inputs.make_inputs(w, seed=5, device="cuda")
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    slabs = _sweep_slabs(w, 4, seed=5)
    slab_rows = np.concatenate([(b * w.n_h + h) * w.T + np.arange(w.T, dtype=np.int64) for b, h in slabs])
    rows = np.union1d(inputs.sample_rows(w, 48, seed=5), slab_rows)
    o_ref, lse_ref = oracle.attention_rows(to_np_bits(qd), to_np_bits(kd), to_np_bits(vd), rows, w.scale)
    idx = torch.from_numpy(rows).cuda()
    og = o.reshape(-1, w.hd)[idx]
    lg = lse.reshape(-1)[idx]
    compare(og, lg, o_ref, lse_ref, w.name)
    pos = np.searchsorted(rows, slab_rows)
    og_slabs = og[torch.from_numpy(pos).cuda()].reshape(1, len(slabs), w.T, w.hd)
    cosine_per_head(og_slabs, o_ref[pos].reshape(1, len(slabs), w.T, w.hd), w.name)
    del qd, kd, vd, o, lse
    torch.cuda.empty_cache()


def test_gqa_prefill_full_size_sampled_rows():
    """The GQA short prefill bench.py times (two-row-tile kernel) at full size:
    48 sampled rows plus every row of four whole (batch, head) slabs against
    the oracle, all three tolerances."""
    w = inputs.WORKLOADS["gqa_prefill"]
    n, _, kern = binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window, w.causal,
                                       with_kernel=True)
    assert kern == "fwd_tc_pair", kern
    qd, kd, vd = inputs.make_inputs(w, seed=9, device="cuda")
    o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, causal=True)
    torch.cuda.synchronize()
    binding.fmha_check_device_status()
    slabs = _sweep_slabs(w, 4, seed=9)
    slab_rows = np.concatenate([(b * w.n_h + h) * w.T + np.arange(w.T, dtype=np.int64) for b, h in slabs])
    rows = np.union1d(inputs.sample_rows(w, 48, seed=9), slab_rows)
    o_ref, lse_ref = oracle.attention_rows(to_np_bits(qd), to_np_bits(kd), to_np_bits(vd), rows, w.scale,
                                           causal=True)
    idx = torch.from_numpy(rows).cuda()
    og = o.reshape(-1, w.hd)[idx]
    compare(og, lse.reshape(-1)[idx], o_ref, lse_ref, w.name)
    pos = np.searchsorted(rows, slab_rows)
    og_slabs = og[torch.from_numpy(pos).cuda()].reshape(1, len(slabs), w.T, w.hd)
    cosine_per_head(og_slabs, o_ref[pos].reshape(1, len(slabs), w.T, w.hd), w.name)


CHAIN = [
    # each kernel family, split and unsplit; O of one call is Q of the next
    W("chain_hd512_mqa_split", 2, 128, 1, 1, 512, 512),
    W("chain_gqa_decode_split", 4, 16, 2, 1, 2000, 128),
    W("chain_tc_prefill", 2, 4, 4, 128, 256, 256, causal=True),
]


@pytest.mark.parametrize("w", CHAIN, ids=[w.name for w in CHAIN])
def test_back_to_back_calls_see_previous_output(w):
    """Consecutive calls on one stream may overlap their set-up with the
    previous kernel (programmatic launches); each must still read the complete
    output of the call before it.  Four calls are queued with no host sync,
    call i+1 taking call i's O as its Q, into buffers that first hold NaN."""
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=21)
    n = 4
    outs = [torch.full_like(qd, float("nan")) for _ in range(n)]
    lses = [torch.full(qd.shape[:-1], float("nan"), dtype=torch.float32, device="cuda") for _ in range(n)]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        src = qd
        for i in range(n):
            binding.fmha_fwd(src, kd, vd, outs[i], lses[i], scale=w.scale, window=w.window, causal=w.causal,
                             stream=stream)
            src = outs[i]
    stream.synchronize()
    binding.fmha_check_device_status()
    src = q
    for i in range(n):
        o_ref, lse_ref = oracle_full(w, src, k, v)
        compare(outs[i], lses[i], o_ref, lse_ref, "%s call %d" % (w.name, i))
        src = outs[i].cpu()


def _random_shapes(n, seed):
    """Seeded random small shapes over every knob: batch, heads and grouping,
    T, s_k (ragged), hd, window and causal."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        hd = int(rng.choice([64, 128, 256, 512]))
        n_kv_h = int(rng.choice([1, 2, 4]))
        G = int(rng.choice([1, 2, 8, 16, 64]))
        T = int(rng.choice([1, 2, 3, 8, 33, 128]))
        causal = bool(rng.random() < 0.4)
        s_k = int(rng.integers(max(T, 1) if causal else 1, 700))
        window = int(rng.choice([0, 0, 1, 17, 256]))
        b = int(rng.integers(1, 3))
        out.append(W("rand%d_hd%d_G%d_T%d_sk%d_w%d_c%d" % (i, hd, G, T, s_k, window, causal), b, n_kv_h * G,
                     n_kv_h, T, s_k, hd, window=window, causal=causal))
    return out


RANDOM = _random_shapes(24, 2024)


@pytest.mark.parametrize("i", range(len(RANDOM)), ids=[w.name for w in RANDOM])
def test_random_shapes_match_oracle(i):
    """fmha_fwd under the automatic plan and, rotating, each forced kernel
    family; then an explicit split into seeded chunk lengths plus the merge."""
    w = RANDOM[i]
    (q, k, v), (qd, kd, vd) = device_inputs(w, seed=51)
    o_ref, lse_ref = oracle_full(w, q, k, v)
    try:
        binding.fmha_set_kernel_path(i % 3)
        o, lse = binding.fmha_fwd(qd, kd, vd, scale=w.scale, window=w.window, causal=w.causal)
        chunk = int(np.random.default_rng(i).integers(16, 320))
        op, lp = binding.fmha_fwd_splitkv(qd, kd, vd, chunk, scale=w.scale, window=w.window, causal=w.causal)
        om, lm = binding.fmha_merge(op, lp)
        torch.cuda.synchronize()
    finally:
        binding.fmha_set_kernel_path(0)
    binding.fmha_check_device_status()
    compare(o, lse, o_ref, lse_ref, "%s path %d" % (w.name, i % 3))
    cosine_per_head(o, o_ref, w.name)
    compare(om, lm, o_ref, lse_ref, "%s split %d" % (w.name, chunk))
