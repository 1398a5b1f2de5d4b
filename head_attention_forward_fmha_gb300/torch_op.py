"""``torch.ops.fmha_gb300.fwd``: the attention forward as a PyTorch custom op.

Registers one operator around the C ABI (``fmha_fwd``) with a fake (meta)
implementation, so that ``torch.compile`` can trace programs that call it
without running it.  The real implementation is the library's CUDA kernels;
like the binding, it accepts contiguous CUDA bf16 tensors only.

    q [b, n_h, T, hd], k, v [b, n_kv_h, s_k, hd]  ->  (O [b, n_h, T, hd] bf16, LSE [b, n_h, T] fp32)

An optional ``sink`` tensor (fp32, n_h attention-sink logits) selects
``fmha_fwd_sink``.
"""
from typing import Optional, Tuple

import torch

from . import binding


@torch.library.custom_op("fmha_gb300::fwd", mutates_args=())
def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float, window: int,
        causal: bool, sink: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    return binding.fmha_fwd(q, k, v, scale=scale, window=window, causal=causal, sink=sink)


@fwd.register_fake
def _fwd_fake(q, k, v, scale, window, causal, sink=None):
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q [b,n_h,T,hd] and k, v [b,n_kv_h,s_k,hd] expected")
    b, n_h, T, hd = q.shape
    return torch.empty_like(q), q.new_empty((b, n_h, T), dtype=torch.float32)


def attention(q, k, v, scale=None, window=0, causal=False, sink=None):
    """Convenience wrapper: ``torch.ops.fmha_gb300.fwd`` with scale defaulting to 1/sqrt(hd)."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return torch.ops.fmha_gb300.fwd(q, k, v, float(scale), int(window), bool(causal), sink)
