"""fp64 CPU oracle for the fused attention forward (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Imported by the test suite, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py``; never by the library.  It shares no
code with the CUDA path; both sides only read the same seeded inputs.

What it computes is the plain definition of softmax attention (see
``fmha_oracle.c`` for the page citations and the readings taken):
``O = softmax(scale * Q K^T + mask) V`` per (batch, head, query row), in double
precision, with the natural-log LSE of the scaled, masked logits, and the
split-KV merge ``O = sum_i exp(lse_i) O_i / sum_i exp(lse_i)``.  An optional
per-head attention-sink logit joins the softmax denominator only (the reading
``fmha_oracle.c`` states for the pages' undefined "D5c sink").

Inputs are numpy arrays: ``float64``, or ``uint16`` holding bf16 bit patterns
(widened exactly inside the C code).  Shapes: q ``[batch, n_h, T, hd]``,
k/v ``[batch, n_kv_h, s_k, hd]``.
"""
import ctypes

import numpy as np

from . import build as _build

_F64, _BF16 = 0, 1
_lib = None


def _bind(path):
    """Load a build of ``fmha_oracle.c`` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, i32, vp, i64, i32, i32, i32, i32, i32, i32,
                                          f64, i32, i32, i32, i32, vp, vp]
    lib.oracle_attention_rows.restype = i32
    lib.oracle_attention_rows_sink.argtypes = [vp, vp, vp, i32, vp, i64, i32, i32, i32, i32, i32, i32,
                                               f64, i32, i32, i32, i32, vp, vp, vp]
    lib.oracle_attention_rows_sink.restype = i32
    lib.oracle_attention_sink.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                          f64, i32, i32, i32, i32, vp, vp, vp]
    lib.oracle_attention_sink.restype = i32
    lib.oracle_merge_sink.argtypes = [vp, vp, i32, i64, i32, vp, vp, vp]
    lib.oracle_merge_sink.restype = None
    lib.oracle_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                     f64, i32, i32, i32, i32, vp, vp]
    lib.oracle_attention.restype = i32
    lib.oracle_merge.argtypes = [vp, vp, i32, i64, i32, vp, vp]
    lib.oracle_merge.restype = None
    lib.oracle_split_layout.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32)]
    lib.oracle_split_layout.restype = i32
    lib.oracle_quantize_nvfp4.argtypes = [vp, i64, i32, ctypes.c_float, vp, vp]
    lib.oracle_quantize_nvfp4.restype = i32
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_max_threads.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(_build.build())
    return _lib


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _prep(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, _BF16
    if x.dtype == np.float64:
        return x, _F64
    raise TypeError("oracle inputs are float64 or uint16 (bf16 bits), got %s" % x.dtype)


def _check(q, k, v):
    (q, tq), (k, tk), (v, tv) = _prep(q), _prep(k), _prep(v)
    if not (tq == tk == tv):
        raise TypeError("q, k, v must share one element type")
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape:
        raise ValueError("q [b,n_h,T,hd], k/v [b,n_kv_h,s_k,hd] expected")
    b, n_h, T, hd = q.shape
    bk, n_kv_h, s_k, hdk = k.shape
    if bk != b or hdk != hd or n_h % n_kv_h != 0:
        raise ValueError("inconsistent shapes %s %s" % (q.shape, k.shape))
    return q, k, v, tq, (b, n_h, n_kv_h, T, s_k, hd)


def _sink_arg(sink, n_h):
    if sink is None:
        return None, None
    sink = np.ascontiguousarray(np.asarray(sink, dtype=np.float64).reshape(-1))
    if sink.size != n_h:
        raise ValueError("sink must hold one logit per query head (%d), got %d" % (n_h, sink.size))
    return sink, sink.ctypes.data


def attention(q, k, v, scale, window=0, causal=False, key_begin=0, key_end=None, sink=None):
    """Return (O [b,n_h,T,hd] float64, lse [b,n_h,T] float64).

    ``key_begin``/``key_end`` restrict the attended keys to that half-open
    range (one split-KV chunk); the default is every key.  ``sink``: optional
    [n_h] sink logits."""
    q, k, v, dt, (b, n_h, n_kv_h, T, s_k, hd) = _check(q, k, v)
    if key_end is None:
        key_end = s_k
    sink, sink_p = _sink_arg(sink, n_h)
    o = np.empty((b, n_h, T, hd), np.float64)
    lse = np.empty((b, n_h, T), np.float64)
    rc = _load().oracle_attention_sink(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt,
                                       b, n_h, n_kv_h, T, s_k, hd, float(scale), int(window),
                                       int(bool(causal)), int(key_begin), int(key_end), sink_p,
                                       o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return o, lse


def attention_rows(q, k, v, rows, scale, window=0, causal=False, key_begin=0, key_end=None, sink=None):
    """Attention for selected flattened rows ``((b*n_h)+h)*T+t``.

    Returns (O [len(rows), hd], lse [len(rows)]), float64."""
    q, k, v, dt, (b, n_h, n_kv_h, T, s_k, hd) = _check(q, k, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if key_end is None:
        key_end = s_k
    sink, sink_p = _sink_arg(sink, n_h)
    o = np.empty((rows.size, hd), np.float64)
    lse = np.empty((rows.size,), np.float64)
    rc = _load().oracle_attention_rows_sink(q.ctypes.data, k.ctypes.data, v.ctypes.data, dt,
                                            rows.ctypes.data, rows.size, b, n_h, n_kv_h, T, s_k, hd,
                                            float(scale), int(window), int(bool(causal)),
                                            int(key_begin), int(key_end), sink_p, o.ctypes.data,
                                            lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the rows or the shape")
    return o, lse


def split_layout(T, s_k, window, kv_chunk):
    """(first key of chunk 0, number of chunks) of the split-KV layout."""
    begin = ctypes.c_int(0)
    n = _load().oracle_split_layout(int(T), int(s_k), int(window), int(kv_chunk), ctypes.byref(begin))
    return begin.value, int(n)


def partials(q, k, v, scale, kv_chunk, window=0, causal=False):
    """Split-KV partial results: (O_i [n, b, n_h, T, hd], lse_i [n, b, n_h, T]).

    Partial i is the attention restricted to the keys of chunk i."""
    s_k = np.asarray(k).shape[2]
    begin, n = split_layout(np.asarray(q).shape[2], s_k, window, kv_chunk)
    os_, ls_ = [], []
    for i in range(n):
        lo = begin + i * kv_chunk
        o, lse = attention(q, k, v, scale, window, causal, key_begin=lo,
                           key_end=min(s_k, lo + kv_chunk))
        os_.append(o)
        ls_.append(lse)
    return np.stack(os_), np.stack(ls_)


def merge(o_parts, lse_parts, sink=None):
    """Merge split-KV partials: O [..., hd] float64 and lse [...] float64.

    ``sink``: optional sink logit per output row (shape ``lse_parts.shape[1:]``)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n = o_parts.shape[0]
    hd = o_parts.shape[-1]
    rows = int(np.prod(lse_parts.shape[1:], dtype=np.int64))
    if o_parts.shape[:-1] != lse_parts.shape:
        raise ValueError("o_parts [n,...,hd] and lse_parts [n,...] disagree")
    o = np.empty(o_parts.shape[1:], np.float64)
    lse = np.empty(lse_parts.shape[1:], np.float64)
    sink_p = None
    if sink is not None:
        sink = np.ascontiguousarray(np.broadcast_to(np.asarray(sink, dtype=np.float64), lse_parts.shape[1:]))
        sink_p = sink.ctypes.data
    _load().oracle_merge_sink(o_parts.ctypes.data, lse_parts.ctypes.data, n, rows, hd, sink_p,
                              o.ctypes.data, lse.ctypes.data)
    return o, lse


def quantize_nvfp4(x, global_scale=1.0):
    """NVFP4 quantisation of rows of fp32 values (the format ``fmha_oracle.c``
    states): x [..., hd] float32 with hd a multiple of 16.  Returns (codes
    [..., hd / 2] uint8, two E2M1 codes per byte, element 2i in the low
    nibble; scales [..., hd / 16] uint8 E4M3 codes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hd = x.shape[-1]
    rows = int(np.prod(x.shape[:-1], dtype=np.int64))
    codes = np.empty(x.shape[:-1] + (hd // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (hd // 16,), np.uint8)
    rc = _load().oracle_quantize_nvfp4(x.ctypes.data, rows, hd, float(global_scale), codes.ctypes.data,
                                       scales.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the NVFP4 arguments (hd %% 16 == 0, global_scale > 0 finite)")
    return codes, scales


_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def dequantize_nvfp4(codes, scales, global_scale=1.0):
    """Values g * s * e of NVFP4 codes and E4M3 scales (float64 [..., hd])."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
    e = _E2M1[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    c = scales.astype(np.int64)
    ex, m = c >> 3, c & 7
    s = np.where(ex == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(ex - 7.0))
    return float(global_scale) * np.repeat(s, 16, axis=-1) * e


__all__ = ["attention", "attention_rows", "split_layout", "partials", "merge",
           "quantize_nvfp4", "dequantize_nvfp4", "set_threads", "max_threads"]
