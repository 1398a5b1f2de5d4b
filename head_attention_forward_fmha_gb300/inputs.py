"""Seeded synthetic inputs for the attention forward workloads.

This module holds shapes and random numbers only -- none of the attention
arithmetic.  The CUDA path and the fp64 oracle both read the bf16 tensors made
here, so they see identical bits.

Recipe: ``torch.Generator().manual_seed(seed)`` on the CPU, ``randn`` in fp32,
optionally multiplied (the shape sweep scales K by 3 to sharpen the softmax),
then rounded to bf16 (round-to-nearest-even).  The constant-V variant sets every
V row of every KV head to one seeded random row ``c``, so the exact output is
``O == c``.  No dataset or trained weights are involved.

The named workloads are the ones the attention forward is specified and
measured on: single-head decode, MQA decode (hd 512, 128 query heads on one KV
head), GQA decode with a 4096-key sliding window over 8192 cached keys split in
512-key chunks, a causal 128-query prefill after 384 cached keys (hd 256), and
an MHA shape sweep.
"""
from dataclasses import dataclass, replace
import math

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_h: int
    n_kv_h: int
    T: int
    s_k: int
    hd: int
    window: int = 0
    causal: bool = False
    k_mult: float = 1.0
    v_const_row: bool = False
    kv_chunk: int = 0  # split-KV chunk named by the workload (0: the library picks)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.hd)

    @property
    def group(self) -> int:
        return self.n_h // self.n_kv_h

    def q_shape(self):
        return (self.batch, self.n_h, self.T, self.hd)

    def kv_shape(self):
        return (self.batch, self.n_kv_h, self.s_k, self.hd)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "single_head_decode": Workload("single_head_decode", 1, 1, 1, 1, 128, 64),
    "mqa_decode": Workload("mqa_decode", 16, 128, 1, 1, 512, 512),
    "mqa_decode_vconst": Workload("mqa_decode_vconst", 16, 128, 1, 1, 512, 512, v_const_row=True),
    "gqa_swa_decode": Workload("gqa_swa_decode", 32, 64, 8, 1, 8192, 128, window=4096, kv_chunk=512),
    "causal_prefill": Workload("causal_prefill", 8, 32, 32, 128, 512, 256, causal=True),
    # Not one of the listed configurations: a GQA short prefill (T = 128, eight
    # query heads per KV head, 4096 cached keys, bottom-right causal), the
    # compute-bound end of the path (its FLOPs take 2x its bytes' time at the
    # peaks), where the two-row-tile tensor-core kernel runs.
    "gqa_prefill": Workload("gqa_prefill", 4, 64, 8, 128, 4096, 128, causal=True),
}

SWEEP_HD = (64, 128, 256, 512)
SWEEP_T = (1, 4, 32, 128)
SWEEP_SK = (128, 256, 384, 512, 4096, 32768)


def sweep():
    """The MHA shape sweep: batch 4, 16 heads, K x3, no mask."""
    out = []
    for hd in SWEEP_HD:
        for T in SWEEP_T:
            for s_k in SWEEP_SK:
                out.append(Workload("sweep_hd%d_T%d_sk%d" % (hd, T, s_k), 4, 16, 16, T, s_k, hd,
                                    k_mult=3.0))
    return out


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu"):
    """(q, k, v) as contiguous bf16 tensors with the workload's shapes.

    ``device="cpu"`` draws from the CPU generator; ``device="cuda"`` draws from
    the CUDA generator (faster for multi-GB shapes).  The two give different
    numbers for the same seed; a check copies the device tensors to the host so
    that both sides still read identical bits."""
    g = torch.Generator(device=device).manual_seed(int(seed))

    def draw(shape):
        return torch.randn(shape, generator=g, dtype=torch.float32, device=device)

    q = draw(w.q_shape()).to(torch.bfloat16)
    k = draw(w.kv_shape())
    if w.k_mult != 1.0:
        k.mul_(w.k_mult)
    k = k.to(torch.bfloat16)
    if w.v_const_row:
        c = draw((w.hd,))
        v = c.to(torch.bfloat16).expand(w.kv_shape()).contiguous()
    else:
        v = draw(w.kv_shape()).to(torch.bfloat16)
    return q.contiguous(), k.contiguous(), v.contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a CPU bf16 tensor, as a uint16 numpy array."""
    if t.dtype != torch.bfloat16:
        raise TypeError("bf16 tensor expected")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, n: int, seed: int = 0) -> np.ndarray:
    """``n`` distinct flattened query rows ((b*n_h)+h)*T+t, always including the
    first and the last row, for sampled checks at full size."""
    total = w.batch * w.n_h * w.T
    rng = np.random.default_rng(seed)
    n = min(n, total)
    picks = set([0, total - 1])
    if n > len(picks):
        extra = rng.choice(total, size=min(total, n + 8), replace=False)
        for r in extra:
            if len(picks) >= n:
                break
            picks.add(int(r))
    return np.array(sorted(picks), dtype=np.int64)
