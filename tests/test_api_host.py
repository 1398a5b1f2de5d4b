"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* the library builds for sm_103a and loads,
* it exports every function ``include/fmha.h`` declares, and the binding
  declares a signature for each,
* argument errors return their codes (and a message) before any CUDA call,
* the split-KV layout (pure host arithmetic) agrees with the oracle's.
"""
import ctypes
import os
import re

import pytest

import oracle
from head_attention_forward_fmha_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_ \*]*?)\b(fmha_[a-z0-9_]+)\s*\(", text):
            names.append(m.group(2))
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("fmha_fwd", "fmha_fwd_splitkv", "fmha_merge", "fmha_split_layout", "fmha_check_device_status",
              "fmha_get_last_error", "fmha_release", "fmha_version", "fmha_splitkv_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), "missing export " + name
        assert name in binding.SIGNATURES, "binding lacks a signature for " + name


def test_version(lib):
    assert binding.fmha_version() >= 100


CASES = [
    # T, s_k, window, chunk
    (1, 8192, 4096, 512), (1, 128, 0, 64), (128, 512, 0, 100), (4, 100, 10, 3), (1, 0, 0, 7),
    (6, 4, 0, 2), (6, 4, 3, 1), (1, 5, 2, 1), (3, 257, 0, 128), (1, 32768, 0, 4096),
]


@pytest.mark.parametrize("T,s_k,window,chunk", CASES)
def test_split_layout_matches_oracle(lib, T, s_k, window, chunk):
    assert binding.fmha_split_layout(T, s_k, window, chunk) == oracle.split_layout(T, s_k, window, chunk)


def test_workspace_bytes(lib):
    assert binding.fmha_splitkv_workspace_bytes(32, 64, 1, 128, 8) == 8 * 32 * 64 * (128 + 1) * 4


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, batch=1, n_h=2, n_kv_h=1, T=1, s_k=8, hd=64, scale=0.125,
         window=0, causal=0):
    return lib.fmha_fwd(q, k, v, o, lse, batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(hd=96), -3), (dict(hd=0), -3),
    (dict(n_h=3, n_kv_h=2), -4), (dict(n_kv_h=0), -4),
    (dict(batch=-1), -5), (dict(T=-2), -5), (dict(s_k=-1), -5),
    (dict(causal=1, T=9, s_k=8), -5), (dict(window=-1), -5), (dict(causal=2), -5),
    (dict(scale=float("inf")), -5), (dict(batch=70000, n_h=1, n_kv_h=1), -5),
    (dict(q=0), -1), (dict(v=0), -1), (dict(o=0), -1), (dict(lse=0), -1),
    (dict(k=24), -2), (dict(o=8), -2), (dict(lse=2), -2),
])
def test_fwd_argument_errors(lib, kw, code):
    assert _fwd(lib, **kw) == code
    assert len(binding.fmha_get_last_error()) > 0


def test_fwd_empty_problem_is_a_no_op(lib):
    # nothing to compute: returns OK without touching (fake) pointers or the GPU
    assert _fwd(lib, batch=0) == 0
    assert _fwd(lib, T=0) == 0


def test_splitkv_and_merge_argument_errors(lib):
    f = lib.fmha_fwd_splitkv
    assert f(16, 16, 16, 16, 16, 0, 1, 1, 1, 1, 8, 64, 0.1, 0, 0, None) == -5     # chunk 0
    assert f(16, 16, 16, 0, 16, 64, 1, 1, 1, 1, 8, 64, 0.1, 0, 0, None) == -1     # o_parts NULL
    assert f(16, 16, 16, 20, 16, 64, 1, 1, 1, 1, 8, 64, 0.1, 0, 0, None) == -2    # o_parts misaligned
    assert f(16, 16, 16, 16, 16, 64, 1, 1, 1, 1, 8, 80, 0.1, 0, 0, None) == -3
    m = lib.fmha_merge
    assert m(16, 16, 0, 16, 16, 1, 1, 1, 64, None) == -5                           # no partials
    assert m(16, 16, 2, 16, 16, 1, 1, 1, 65, None) == -3
    assert m(0, 16, 2, 16, 16, 1, 1, 1, 64, None) == -1
    assert m(16, 16, 2, 24, 16, 1, 1, 1, 64, None) == -2
    assert m(16, 16, 2, 16, 16, 0, 1, 1, 64, None) == 0                            # empty
    assert lib.fmha_split_layout(1, 10, 0, 0, None) == -5
    # chunk count limits: more than 65535 chunks, and chunks x batch x n_kv_h past 2^31 - 1
    assert f(16, 16, 16, 16, 16, 1, 1, 1, 1, 1, 70000, 64, 0.1, 0, 0, None) == -5
    assert "too many KV chunks" in binding.fmha_get_last_error()
    assert f(16, 16, 16, 16, 16, 1, 40000, 1, 1, 1, 60000, 64, 0.1, 0, 0, None) == -5
    assert "exceeds 2^31 - 1" in binding.fmha_get_last_error()
    assert lib.fmha_fwd(16, 16, 16, 16, 16, 60000, 1024, 1, 64, 64, 64, 0.1, 0, 0, None) == -5   # 3.9e9 rows
    assert "query rows exceeds" in binding.fmha_get_last_error()


def test_f16_partials_only_on_the_hd512_tensor_core_kernel(lib):
    f = lib.fmha_fwd_splitkv_ex
    # hd 128: the fp16 partial format does not exist there
    assert f(16, 16, 16, 16, 16, 16, 1, 64, 1, 64, 1, 1, 100, 128, 0.1, 0, 0, None) == -9
    # hd 512 with 8 query rows per KV head runs on the decode kernel: unsupported too
    assert f(16, 16, 16, 16, 16, 16, 1, 64, 1, 8, 1, 1, 100, 512, 0.1, 0, 0, None) == -9
    # hd 512 with 128 rows per KV head: accepted up to the pointer checks
    assert f(16, 16, 16, 16, 16, 0, 1, 128, 1, 128, 1, 1, 256, 512, 0.1, 0, 0, None) == -1   # range NULL
    assert f(16, 16, 16, 16, 16, 18, 1, 128, 1, 128, 1, 1, 256, 512, 0.1, 0, 0, None) == -2  # range misaligned
    assert f(16, 16, 16, 16, 16, 16, 7, 128, 1, 128, 1, 1, 256, 512, 0.1, 0, 0, None) == -5  # no such format
    m = lib.fmha_merge_ex
    assert m(16, 16, 16, 1, 2, None, 16, 16, 1, 1, 1, 128, None) == -9
    assert m(16, 16, 0, 1, 2, None, 16, 16, 1, 1, 1, 512, None) == -1
    assert m(16, 16, 16, 1, 2, None, 16, 16, 0, 1, 1, 512, None) == 0                # empty
    assert m(16, 16, None, 0, 2, 18, 16, 16, 1, 1, 1, 64, None) == -2                # sink misaligned


def test_fwd_sink_argument_errors(lib):
    f = lib.fmha_fwd_sink
    assert f(16, 16, 16, 16, 16, 18, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -2     # sink misaligned
    assert f(16, 16, 16, 16, 16, 16, 1, 2, 1, 1, 8, 80, 0.125, 0, 0, None) == -3
    assert f(16, 16, 16, 16, 16, 16, 0, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == 0      # empty problem



def test_nvfp4_argument_errors(lib):
    # every call here fails its argument checks (or has nothing to do) before
    # any launch: the fake pointers are never dereferenced
    f = lib.fmha_fwd_nvfp4
    # q, k, v, codes, scales, lse, g, batch, n_h, n_kv_h, T, s_k, hd, scale, window, causal, stream
    assert f(16, 16, 16, 0, 16, 16, 1.0, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -1     # codes NULL
    assert f(16, 16, 16, 16, 0, 16, 1.0, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -1     # scales NULL
    assert f(16, 16, 16, 24, 16, 16, 1.0, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -2    # codes misaligned
    assert f(16, 16, 16, 16, 18, 16, 1.0, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -2    # scales misaligned
    for g in (0.0, -1.0, float("inf"), float("nan")):
        assert f(16, 16, 16, 16, 16, 16, g, 1, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == -5
    assert f(16, 16, 16, 16, 16, 16, 1.0, 1, 2, 1, 1, 8, 96, 0.125, 0, 0, None) == -3
    assert f(16, 16, 16, 16, 16, 16, 1.0, 0, 2, 1, 1, 8, 64, 0.125, 0, 0, None) == 0     # empty problem
    qz = lib.fmha_quantize_nvfp4
    assert qz(16, 4, 24, 1.0, 16, 16, None) == -5                                       # hd not a multiple of 16
    assert qz(16, -1, 32, 1.0, 16, 16, None) == -5
    assert qz(16, 4, 32, 0.0, 16, 16, None) == -5
    assert qz(16, 0, 32, 1.0, 0, 0, None) == 0                                          # nothing to do
    assert qz(0, 4, 32, 1.0, 16, 16, None) == -1
    assert qz(8, 4, 32, 1.0, 16, 16, None) == -2                                        # x misaligned
    assert qz(16, 4, 32, 1.0, 12, 16, None) == -2                                       # codes misaligned


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(ImportError):
        binding.load(str(tmp_path / "nope.so"))
