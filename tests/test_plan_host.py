"""fmha_fwd_plan on the host (no GPU): the kernel family follows the rule the
header documents, the chunk count is the one fmha_split_layout gives for the
chosen chunk, chunks are whole KV tiles of that kernel, and every chunk holds
keys that some query row attends."""
import itertools

import pytest

import oracle
from head_attention_forward_fmha_gb300 import binding, build

KV_TILE = {  # keys per tile of each kernel family and head dim
    "decode_splitkv": {64: 64, 128: 64, 256: 32, 512: 32},
    "fwd_tc": {64: 128, 128: 128, 256: 64},
    "fwd_tc_wide": {512: 128},
    "fwd_tc_pair": {64: 128, 128: 128},
}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load()


def expected_families(n_h, n_kv_h, T, hd):
    rows = (n_h // n_kv_h) * T  # query rows per KV head
    if rows >= (64 if hd <= 128 else 32):
        if hd == 512:
            return {"fwd_tc_wide"}
        # more than one 128-row tile per KV head at hd <= 128: one or two tiles per block
        return {"fwd_tc", "fwd_tc_pair"} if rows > 128 and hd <= 128 else {"fwd_tc"}
    return {"decode_splitkv"}


SHAPES = list(itertools.product(
    [1, 4, 16],                 # batch
    [(8, 8), (64, 8), (128, 1)],  # (n_h, n_kv_h)
    [1, 4, 32, 128],            # T
    [128, 700, 4096],           # s_k
    [64, 128, 256, 512],        # hd
    [(0, 0), (300, 0), (0, 1)],  # (window, causal)
))


@pytest.mark.parametrize("batch,heads,T,s_k,hd,mask", SHAPES[::7])
def test_plan_follows_documented_rules(batch, heads, T, s_k, hd, mask):
    n_h, n_kv_h = heads
    window, causal = mask
    if causal and T > s_k:
        return
    n, chunk, family = binding.fmha_fwd_plan(batch, n_h, n_kv_h, T, s_k, hd, window, causal, with_kernel=True)
    assert family in expected_families(n_h, n_kv_h, T, hd)
    assert n >= 1 and chunk >= 1
    first, n_layout = binding.fmha_split_layout(T, s_k, window, chunk)
    assert n == n_layout
    if n > 1:
        assert chunk % KV_TILE[family][hd] == 0
    # the oracle's layout agrees, and no chunk is empty of attended keys
    first_o, n_o = oracle.split_layout(T, s_k, window, chunk)
    assert (first_o, n_o) == (first, n)
    assert first + (n - 1) * chunk < s_k


def test_forced_families():
    try:
        binding.fmha_set_kernel_path(1)
        assert binding.fmha_fwd_plan(2, 64, 8, 128, 4096, 128, with_kernel=True)[2] == "decode_splitkv"
        binding.fmha_set_kernel_path(2)
        assert binding.fmha_fwd_plan(2, 8, 8, 1, 4096, 128, with_kernel=True)[2] == "fwd_tc"
        assert binding.fmha_fwd_plan(2, 8, 8, 1, 4096, 512, with_kernel=True)[2] == "fwd_tc_wide"
        # two row tiles per block wherever that kernel applies (hd 64 / 128, > 128 rows per KV head)
        assert binding.fmha_fwd_plan(2, 64, 8, 128, 4096, 128, with_kernel=True)[2] == "fwd_tc_pair"
        assert binding.fmha_fwd_plan(2, 64, 8, 32, 4096, 64, with_kernel=True)[2] == "fwd_tc_pair"
        assert binding.fmha_fwd_plan(2, 64, 8, 16, 4096, 128, with_kernel=True)[2] == "fwd_tc"    # 128 rows
        assert binding.fmha_fwd_plan(2, 64, 8, 128, 4096, 256, with_kernel=True)[2] == "fwd_tc"   # hd 256
        binding.fmha_set_kernel_path(4)
        assert binding.fmha_fwd_plan(2, 64, 8, 128, 4096, 128, with_kernel=True)[2] == "fwd_tc"
        binding.fmha_set_kernel_path(3)
        assert binding.fmha_fwd_plan(2, 64, 8, 128, 4096, 128, with_kernel=True)[2] == "fwd_tc"
    finally:
        binding.fmha_set_kernel_path(0)
