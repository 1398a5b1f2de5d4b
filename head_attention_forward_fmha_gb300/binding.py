"""Thin ctypes binding of ``libfmha_gb300.so`` (C ABI in ``include/fmha.h``).

Argument marshalling only: torch tensors are checked for dtype, shape,
contiguity and device, then their data pointers go to the C entry point of the
same name.  Every step of the attention forward runs in the library's CUDA
kernels; there is no CPU fallback, and a missing library raises.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# FMHA_GB300_LIB may name another build of the same library (for example the
# checked build, CHECKED_LIB_PATH) to load instead of the in-tree one.
LIB_PATH = os.environ.get("FMHA_GB300_LIB") or os.path.join(_PKG, "libfmha_gb300.so")
CHECKED_LIB_PATH = os.path.join(_PKG, "libfmha_gb300_checked.so")
FMHA_BUILD_CHECKED = 1

FMHA_OK = 0
ERRORS = {
    -1: "FMHA_ERR_NULL", -2: "FMHA_ERR_ALIGN", -3: "FMHA_ERR_HEADDIM", -4: "FMHA_ERR_HEADS",
    -5: "FMHA_ERR_SHAPE", -6: "FMHA_ERR_WORKSPACE", -7: "FMHA_ERR_LAUNCH", -8: "FMHA_ERR_DEVICE_TIMEOUT",
    -9: "FMHA_ERR_UNSUPPORTED", -10: "FMHA_ERR_DEVICE_BOUNDS",
}
# Partial formats (enum fmha_parts_format).
PARTS_F32, PARTS_F16 = 0, 1

# Every symbol include/fmha.h declares, with its ctypes signature.
_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fmha_fwd": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp], _i32),
    "fmha_fwd_plan": ([_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)],
                      _i32),
    "fmha_split_layout": ([_i32, _i32, _i32, _i32, ctypes.POINTER(_i32)], _i32),
    "fmha_fwd_splitkv": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp],
                         _i32),
    "fmha_merge": ([_vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _vp], _i32),
    "fmha_fwd_splitkv_ex": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                             _i32, _vp], _i32),
    "fmha_merge_ex": ([_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp], _i32),
    "fmha_fwd_sink": ([_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp], _i32),
    "fmha_splitkv_workspace_bytes": ([_i32, _i32, _i32, _i32, _i32], _sz),
    "fmha_workspace_bytes": ([_i32, _i32, _i32, _i32, _i32], _sz),
    "fmha_check_device_status": ([_vp], _i32),
    "fmha_get_last_error": ([], ctypes.c_char_p),
    "fmha_release": ([], None),
    "fmha_version": ([], _i32),
    "fmha_set_kernel_path": ([_i32], _i32),
    "fmha_selftest_wait_timeout": ([ctypes.c_uint, _vp], _i32),
    "fmha_fwd_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp], _i32),
    "fmha_build_flags": ([], _i32),
    "fmha_fwd_host": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp], _i32),
    "fmha_selftest_bounds_check": ([_vp], _i32),
    "fmha_fwd_nvfp4": ([_vp, _vp, _vp, _vp, _vp, _vp, _f32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp],
                       _i32),
    "fmha_quantize_nvfp4": ([_vp, ctypes.c_longlong, _i32, _f32, _vp, _vp, _vp], _i32),
}
# Size of the fixed split-KV scratch fmha_fwd_noalloc uses (FMHA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 << 20


_lib = None


class FmhaError(RuntimeError):
    def __init__(self, code, fn, msg):
        super().__init__("%s returned %s (%d): %s" % (fn, ERRORS.get(code, "?"), code, msg))
        self.code = code


def load(path=None):
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libfmha_gb300.so not found at %s: run head_attention_forward_fmha_gb300.build" % p)
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(rc, fn):
    if rc != FMHA_OK:
        raise FmhaError(rc, fn, load().fmha_get_last_error().decode(errors="replace"))


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _bf16(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CUDA bf16 tensor" % name)
    return t.data_ptr()


def _f32(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CUDA float32 tensor" % name)
    return t.data_ptr()


def _shapes(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or tuple(k.shape) != tuple(v.shape):
        raise ValueError("q [b,n_h,T,hd] and k, v [b,n_kv_h,s_k,hd] expected")
    b, n_h, T, hd = q.shape
    bk, n_kv_h, s_k, hdk = k.shape
    if bk != b or hdk != hd:
        raise ValueError("q %s and k %s disagree" % (tuple(q.shape), tuple(k.shape)))
    return b, n_h, n_kv_h, T, s_k, hd


def _check_outputs(q, o, lse):
    """o must be shaped like q and lse [b, n_h, T], both on q's device, so that
    the kernels never write past the end of a caller's buffer."""
    b, n_h, T, _ = q.shape
    if not isinstance(o, torch.Tensor) or tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must be shaped like q %s" % (tuple(q.shape),))
    if not isinstance(lse, torch.Tensor) or tuple(lse.shape) != (b, n_h, T):
        raise ValueError("lse must be [b,n_h,T] = %s" % ((b, n_h, T),))
    if o.device != q.device or lse.device != q.device:
        raise ValueError("o and lse must be on q's device (%s)" % q.device)


def _sink_ptr(sink, n_h):
    if sink is None:
        return None
    if sink.numel() != n_h:
        raise ValueError("sink must hold one logit per query head (%d), got %d" % (n_h, sink.numel()))
    return _f32(sink, "sink")


def fmha_fwd(q, k, v, o=None, lse=None, scale=None, window=0, causal=False, stream=None, sink=None):
    """O (bf16 [b,n_h,T,hd]) and LSE (fp32 [b,n_h,T]); allocates them if not given.
    sink: optional fp32 CUDA tensor of n_h attention-sink logits (fmha_fwd_sink)."""
    b, n_h, n_kv_h, T, s_k, hd = _shapes(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, n_h, T), dtype=torch.float32, device=q.device)
    qp, kp, vp = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    _check_outputs(q, o, lse)
    if scale is None:
        scale = hd ** -0.5
    if sink is None:
        rc = load().fmha_fwd(qp, kp, vp, _bf16(o, "o"), _f32(lse, "lse"),
                             b, n_h, n_kv_h, T, s_k, hd, float(scale), int(window), int(bool(causal)),
                             _stream(stream))
        _check(rc, "fmha_fwd")
    else:
        rc = load().fmha_fwd_sink(qp, kp, vp, _bf16(o, "o"), _f32(lse, "lse"),
                                  _sink_ptr(sink, n_h), b, n_h, n_kv_h, T, s_k, hd, float(scale), int(window),
                                  int(bool(causal)), _stream(stream))
        _check(rc, "fmha_fwd_sink")
    return o, lse


def _host(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous host (CPU) %s tensor" % (name, dtype))
    return t.data_ptr()


def fmha_fwd_host(q, k, v, o=None, lse=None, scale=None, window=0, causal=False, stream=None):
    """fmha_fwd on host tensors (fmha_fwd_host): q, k, v are contiguous CPU bf16
    tensors, preferably page-locked; O and LSE come back in CPU tensors
    (page-locked ones are allocated if not given).  Stream-ordered: the results
    are valid, and the inputs may be changed, once `stream` has passed the call."""
    b, n_h, n_kv_h, T, s_k, hd = _shapes(q, k, v)
    if o is None:
        o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((b, n_h, T), dtype=torch.float32).pin_memory()
    if tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (b, n_h, T):
        raise ValueError("o must be [b,n_h,T,hd] and lse [b,n_h,T]")
    if scale is None:
        scale = hd ** -0.5
    rc = load().fmha_fwd_host(_host(q, "q", torch.bfloat16), _host(k, "k", torch.bfloat16),
                              _host(v, "v", torch.bfloat16), _host(o, "o", torch.bfloat16),
                              _host(lse, "lse", torch.float32), b, n_h, n_kv_h, T, s_k, hd, float(scale),
                              int(window), int(bool(causal)), _stream(stream))
    _check(rc, "fmha_fwd_host")
    return o, lse


KERNELS = {1: "decode_splitkv", 2: "fwd_tc", 3: "fwd_tc_wide", 4: "fwd_tc_pair"}


def fmha_fwd_plan(batch, n_h, n_kv_h, T, s_k, hd, window=0, causal=False, with_kernel=False):
    """(n_splits, kv_chunk) that fmha_fwd uses for this shape, plus the kernel
    family name if ``with_kernel``."""
    chunk, kern = ctypes.c_int(0), ctypes.c_int(0)
    n = load().fmha_fwd_plan(batch, n_h, n_kv_h, T, s_k, hd, int(window), int(bool(causal)), ctypes.byref(chunk),
                             ctypes.byref(kern))
    _check(n if n < 0 else 0, "fmha_fwd_plan")
    if with_kernel:
        return n, chunk.value, KERNELS.get(kern.value, "?")
    return n, chunk.value


def fmha_split_layout(T, s_k, window, kv_chunk):
    """(first key of chunk 0, number of chunks)."""
    first = ctypes.c_int(0)
    n = load().fmha_split_layout(int(T), int(s_k), int(window), int(kv_chunk), ctypes.byref(first))
    _check(n if n < 0 else 0, "fmha_split_layout")
    return first.value, n


def fmha_fwd_splitkv(q, k, v, kv_chunk, o_parts=None, lse_parts=None, scale=None, window=0, causal=False,
                     stream=None):
    """fp32 partials O_i [n,b,n_h,T,hd] and lse_i [n,b,n_h,T] for chunks of kv_chunk keys."""
    b, n_h, n_kv_h, T, s_k, hd = _shapes(q, k, v)
    _, n = fmha_split_layout(T, s_k, window, kv_chunk)
    if o_parts is None:
        o_parts = torch.empty((n, b, n_h, T, hd), dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((n, b, n_h, T), dtype=torch.float32, device=q.device)
    if o_parts.numel() < n * b * n_h * T * hd or lse_parts.numel() < n * b * n_h * T:
        raise ValueError("partial buffers too small for %d chunks" % n)
    if scale is None:
        scale = hd ** -0.5
    rc = load().fmha_fwd_splitkv(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _f32(o_parts, "o_parts"),
                                 _f32(lse_parts, "lse_parts"), int(kv_chunk), b, n_h, n_kv_h, T, s_k, hd,
                                 float(scale), int(window), int(bool(causal)), _stream(stream))
    _check(rc, "fmha_fwd_splitkv")
    return o_parts, lse_parts


def fmha_merge(o_parts, lse_parts, o=None, lse=None, stream=None, sink=None):
    """Merge partials [n,b,n_h,T,hd] / [n,b,n_h,T] into bf16 O and fp32 LSE
    (with an optional [n_h] attention-sink tensor)."""
    if o_parts.dim() != 5 or lse_parts.dim() != 4 or tuple(o_parts.shape[:4]) != tuple(lse_parts.shape):
        raise ValueError("o_parts [n,b,n_h,T,hd] and lse_parts [n,b,n_h,T] expected")
    n, b, n_h, T, hd = o_parts.shape
    if o is None:
        o = torch.empty((b, n_h, T, hd), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((b, n_h, T), dtype=torch.float32, device=o_parts.device)
    if sink is None:
        rc = load().fmha_merge(_f32(o_parts, "o_parts"), _f32(lse_parts, "lse_parts"), n, _bf16(o, "o"),
                               _f32(lse, "lse"), b, n_h, T, hd, _stream(stream))
        _check(rc, "fmha_merge")
    else:
        rc = load().fmha_merge_ex(_f32(o_parts, "o_parts"), _f32(lse_parts, "lse_parts"), None, PARTS_F32, n,
                                  _sink_ptr(sink, n_h), _bf16(o, "o"), _f32(lse, "lse"), b, n_h, T, hd,
                                  _stream(stream))
        _check(rc, "fmha_merge_ex")
    return o, lse


def fmha_fwd_splitkv_f16(q, k, v, kv_chunk, o_parts=None, lse_parts=None, range_parts=None, scale=None, window=0,
                         causal=False, stream=None):
    """fp16 partials (FMHA_PARTS_F16): O_i * 2^-k as fp16 [n,b,n_h,T,hd], lse_i fp32 [n,b,n_h,T] and the
    factors 2^k fp32 [n,b,n_h,T,2] (one per 256-column half row).  hd-512 tensor-core kernel only."""
    b, n_h, n_kv_h, T, s_k, hd = _shapes(q, k, v)
    _, n = fmha_split_layout(T, s_k, window, kv_chunk)
    if o_parts is None:
        o_parts = torch.empty((n, b, n_h, T, hd), dtype=torch.float16, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((n, b, n_h, T), dtype=torch.float32, device=q.device)
    if range_parts is None:
        range_parts = torch.empty((n, b, n_h, T, 2), dtype=torch.float32, device=q.device)
    if (o_parts.dtype != torch.float16 or not o_parts.is_cuda or not o_parts.is_contiguous()
            or o_parts.numel() < n * b * n_h * T * hd or lse_parts.numel() < n * b * n_h * T
            or range_parts.numel() < n * b * n_h * T * 2):
        raise ValueError("fp16 partial buffers too small or of the wrong type for %d chunks" % n)
    if scale is None:
        scale = hd ** -0.5
    rc = load().fmha_fwd_splitkv_ex(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), o_parts.data_ptr(),
                                    _f32(lse_parts, "lse_parts"), _f32(range_parts, "range_parts"), PARTS_F16,
                                    int(kv_chunk), b, n_h, n_kv_h, T, s_k, hd, float(scale), int(window),
                                    int(bool(causal)), _stream(stream))
    _check(rc, "fmha_fwd_splitkv_ex")
    return o_parts, lse_parts, range_parts


def fmha_merge_f16(o_parts, lse_parts, range_parts, o=None, lse=None, stream=None, sink=None):
    """Merge FMHA_PARTS_F16 partials into bf16 O and fp32 LSE."""
    if o_parts.dim() != 5 or o_parts.dtype != torch.float16 or not o_parts.is_contiguous():
        raise ValueError("o_parts: contiguous fp16 [n,b,n_h,T,hd] expected")
    n, b, n_h, T, hd = o_parts.shape
    if tuple(lse_parts.shape) != (n, b, n_h, T) or tuple(range_parts.shape) != (n, b, n_h, T, 2):
        raise ValueError("lse_parts [n,b,n_h,T] and range_parts [n,b,n_h,T,2] expected")
    if o is None:
        o = torch.empty((b, n_h, T, hd), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((b, n_h, T), dtype=torch.float32, device=o_parts.device)
    rc = load().fmha_merge_ex(o_parts.data_ptr(), _f32(lse_parts, "lse_parts"), _f32(range_parts, "range_parts"),
                              PARTS_F16, n, _sink_ptr(sink, n_h), _bf16(o, "o"), _f32(lse, "lse"), b, n_h, T, hd,
                              _stream(stream))
    _check(rc, "fmha_merge_ex")
    return o, lse


def fmha_splitkv_workspace_bytes(batch, n_h, T, hd, n_splits):
    return int(load().fmha_splitkv_workspace_bytes(batch, n_h, T, hd, n_splits))


def fmha_workspace_bytes(batch, n_h, T, hd, n_splits):
    """Bytes of the caller buffers fmha_fwd_splitkv + fmha_merge need for n_splits chunks."""
    return int(load().fmha_workspace_bytes(batch, n_h, T, hd, n_splits))


def fmha_check_device_status(stream=None):
    rc = load().fmha_check_device_status(_stream(stream))
    _check(rc, "fmha_check_device_status")


def fmha_get_last_error():
    return load().fmha_get_last_error().decode(errors="replace")


def _u8(t, name):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CUDA uint8 tensor" % name)
    return t.data_ptr()


def fmha_fwd_nvfp4(q, k, v, codes=None, scales=None, lse=None, global_scale=1.0, scale=None, window=0,
                   causal=False, stream=None):
    """fmha_fwd with O quantised to NVFP4 (see include/fmha.h): returns
    (codes uint8 [b,n_h,T,hd/2], scales uint8 [b,n_h,T,hd/16] E4M3, lse fp32 [b,n_h,T])."""
    b, n_h, n_kv_h, T, s_k, hd = _shapes(q, k, v)
    if codes is None:
        codes = torch.empty((b, n_h, T, hd // 2), dtype=torch.uint8, device=q.device)
    if scales is None:
        scales = torch.empty((b, n_h, T, hd // 16), dtype=torch.uint8, device=q.device)
    if lse is None:
        lse = torch.empty((b, n_h, T), dtype=torch.float32, device=q.device)
    qp, kp, vp = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    if (tuple(codes.shape) != (b, n_h, T, hd // 2) or tuple(scales.shape) != (b, n_h, T, hd // 16)
            or tuple(lse.shape) != (b, n_h, T)):
        raise ValueError("codes [b,n_h,T,hd/2], scales [b,n_h,T,hd/16] and lse [b,n_h,T] expected")
    if codes.device != q.device or scales.device != q.device or lse.device != q.device:
        raise ValueError("codes, scales and lse must be on q's device (%s)" % q.device)
    if scale is None:
        scale = hd ** -0.5
    rc = load().fmha_fwd_nvfp4(qp, kp, vp, _u8(codes, "codes"), _u8(scales, "scales"), _f32(lse, "lse"),
                               float(global_scale), b, n_h, n_kv_h, T, s_k, hd, float(scale), int(window),
                               int(bool(causal)), _stream(stream))
    _check(rc, "fmha_fwd_nvfp4")
    return codes, scales, lse


def fmha_quantize_nvfp4(x, global_scale=1.0, stream=None):
    """NVFP4 codes and E4M3 scales of fp32 rows x [..., hd] (the fused epilogues' quantiser)."""
    if x.dim() < 1 or x.shape[-1] % 16 != 0:
        raise ValueError("x [..., hd] with hd a multiple of 16 expected")
    hd = x.shape[-1]
    rows = x.numel() // hd
    codes = torch.empty(tuple(x.shape[:-1]) + (hd // 2,), dtype=torch.uint8, device=x.device)
    scales = torch.empty(tuple(x.shape[:-1]) + (hd // 16,), dtype=torch.uint8, device=x.device)
    rc = load().fmha_quantize_nvfp4(_f32(x, "x"), rows, hd, float(global_scale), _u8(codes, "codes"),
                                    _u8(scales, "scales"), _stream(stream))
    _check(rc, "fmha_quantize_nvfp4")
    return codes, scales


def fmha_release():
    load().fmha_release()


def fmha_version():
    return int(load().fmha_version())


def fmha_build_flags():
    """FMHA_BUILD_CHECKED if the loaded library is the checked build, else 0."""
    return int(load().fmha_build_flags())


def fmha_selftest_bounds_check(stream=None):
    """One failing index check on the device (recorded only by the checked build)."""
    _check(load().fmha_selftest_bounds_check(_stream(stream)), "fmha_selftest_bounds_check")


def fmha_selftest_wait_timeout(timeout_us, stream=None):
    """Launch the bounded-wait self-test kernel (see include/fmha.h)."""
    _check(load().fmha_selftest_wait_timeout(int(timeout_us), _stream(stream)), "fmha_selftest_wait_timeout")


def fmha_set_kernel_path(path):
    """0 automatic, 1 decode kernel, 2 tensor-core kernels (two row tiles per block where that
    kernel applies), 3 tensor-core kernels, one row tile per block, with the row-tile kernel's
    P V in the SS form (P through shared memory) instead of the TS form, 4 tensor-core kernels,
    one row tile per block (TS form)."""
    _check(load().fmha_set_kernel_path(int(path)), "fmha_set_kernel_path")


def fmha_fwd_noalloc(q, k, v, o, lse, scale=None, window=0, causal=False, stream=None):
    """fmha_fwd for callers that cannot allocate device memory: O and LSE must be
    given, and split-KV partials use the library's fixed scratch array instead
    of a workspace (see include/fmha.h)."""
    b, n_h, n_kv_h, T, s_k, hd = _shapes(q, k, v)
    qp, kp, vp = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    _check_outputs(q, o, lse)
    if scale is None:
        scale = hd ** -0.5
    rc = load().fmha_fwd_noalloc(qp, kp, vp, _bf16(o, "o"), _f32(lse, "lse"),
                                 b, n_h, n_kv_h, T, s_k, hd, float(scale), int(window), int(bool(causal)),
                                 _stream(stream))
    _check(rc, "fmha_fwd_noalloc")
    return o, lse
