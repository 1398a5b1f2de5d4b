#!/usr/bin/env python
"""Benchmark of the GB300 fused attention forward.

One step = one ``fmha_fwd`` call (the whole hot path: plan, Q/K/V streaming,
QK^T, mask, online softmax, PV, epilogue and -- when the plan splits the KV
range -- the LSE merge) over one batch of the workload.  Default workload: MQA
decode, batch 16, 128 query heads on one KV head, hd 512, 512 cached keys.

Timing: inputs are rotated over enough copies that the set touched by a step
exceeds twice the L2 size, so every step reads K/V from HBM; steps are
replayed from CUDA graphs and timed with CUDA events on the launching stream
(max over ranks).  ``value`` is algorithmic HBM bytes per second (Q + attended
K + attended V + O + LSE, split-KV partials not credited).

JSON line keys beyond the basic contract: ``roofline`` (the dominant kernel
timed alone, against the measured HBM copy bandwidth), ``cpu_baseline`` (the
fp64 oracle on the host cores, a bounded sample), ``e2e`` (the C ABI call with
host buffers, ``fmha_fwd_host``: per step the H2D copies of Q, K, V from
page-locked memory, the forward, and the D2H copies of O and LSE; steps
alternate between two streams), ``clocks``
(nvidia-smi sampled during the timed region), ``gpu_launches`` and
``secondary`` (the single-head decode -- launch-latency bound, read its
``us_per_step`` --, the GQA sliding-window decode, the causal prefill and a GQA
short prefill (T 128, group 8, hd 128, 4096 keys: compute-bound, read its
``frac_bf16_peak``), each with its own roofline figures, as ``fmha_fwd`` plans
them; for the GQA decode also ``split_512``: the same workload split literally
into 512-key chunks with ``fmha_fwd_splitkv`` + ``fmha_merge``).

``--impl reference`` times the fp64 oracle on the host cores instead (the only
reference implementation this project has), on the same workload and metric.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from head_attention_forward_fmha_gb300 import inputs  # noqa: E402

METRIC = "FMHA decode HBM GB/s (% of roofline) and prefill TFLOP/s (% bf16 peak)"
DEFAULT_WORKLOAD = "mqa_decode"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "head_attention_forward_fmha_gb300", "csrc")


# ----------------------------------------------------------------------------
# algorithmic counts
# ----------------------------------------------------------------------------
def attended_count(w, t):
    p = w.s_k - w.T + t
    lo, hi = 0, w.s_k - 1
    if w.causal:
        hi = min(hi, p)
    if w.window > 0:
        lo = max(lo, p - w.window + 1)
    return max(0, hi - lo + 1)


def kv_keys_read(w):
    """Keys of one KV head that some query row attends (read once from HBM)."""
    lo = w.s_k
    hi = -1
    for t in range(w.T):
        p = w.s_k - w.T + t
        a, b = 0, w.s_k - 1
        if w.causal:
            b = min(b, p)
        if w.window > 0:
            a = max(a, p - w.window + 1)
        if a <= b:
            lo, hi = min(lo, a), max(hi, b)
    return max(0, hi - lo + 1)


def algo_bytes(w):
    q = w.batch * w.n_h * w.T * w.hd * 2
    kv = w.batch * w.n_kv_h * kv_keys_read(w) * w.hd * 2 * 2
    o = q
    lse = w.batch * w.n_h * w.T * 4
    return q + kv + o + lse


def algo_flops(w):
    pairs = sum(attended_count(w, t) for t in range(w.T))
    return 4.0 * w.hd * w.batch * w.n_h * pairs


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None,
                "measured")
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


# Source files each kernel is built from: a recorded ncu traffic figure is
# only used while these files are unchanged.
KERNEL_SOURCES = {
    "decode_splitkv": ("decode_kernel.cu", "ptx.cuh"),
    "fwd_tc": ("tc_kernel.cu", "tc_common.cuh", "ptx.cuh"),
    "fwd_tc_wide": ("tc_wide_kernel.cu", "tc_common.cuh", "ptx.cuh"),
    "fwd_tc_pair": ("tc_pair_kernel.cu", "tc_common.cuh", "ptx.cuh"),
    "merge_lse": ("merge_kernel.cu", "ptx.cuh"),
}


def kernel_digest(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        h.update(open(os.path.join(CSRC, name), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, or None
    if absent or taken on other kernel sources."""
    path = os.path.join(PROFILE_DIR, "%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"kernel_sources_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_digest(kernel):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0] and parts[0].replace("GPU-", "") not in self.uuid:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1] or rows[-3:]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        mhz = [float(p[1]) for _, p in inside if re.match(r"^[0-9.]+$", p[1])]
        mx = [float(p[2]) for _, p in inside if re.match(r"^[0-9.]+$", p[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in inside:
            for name, val in zip(names, p[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ----------------------------------------------------------------------------
# GPU timing helpers
# ----------------------------------------------------------------------------
def rotating_sets(w, n_bytes_min, seed=0):
    per_set = algo_bytes(w)
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    n = max(1, math.ceil(2 * l2 / max(1, per_set)))
    n = min(n, 64)
    sets = []
    for i in range(n):
        q, k, v = inputs.make_inputs(w, seed=seed + i, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((w.batch, w.n_h, w.T), dtype=torch.float32, device="cuda")
        sets.append((q, k, v, o, lse))
    return sets, l2


def graph_time(step_fn, n_sets, steps, stream, per_graph=None):
    """Time exactly `steps` calls step_fn(i) (i = set index) via CUDA graphs.
    Returns (ms total, launches of the graph)."""
    per_graph = per_graph or max(1, (64 // n_sets)) * n_sets
    per_graph = max(1, min(per_graph, steps))
    full, rem = divmod(steps, per_graph)
    graphs = []
    with torch.cuda.stream(stream):
        for count in ([per_graph] if full else []) + ([rem] if rem else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(count):
                    step_fn(i % n_sets)
            graphs.append((g, count))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        if full:
            g0 = graphs[0][0]
            for _ in range(full):
                g0.replay()
        if rem:
            graphs[-1][0].replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def dist_setup(args, backend="nccl"):
    """(world, rank, local_rank, torch.distributed or None).  One process per
    GPU; ranks are independent replicas (no data-path collective), the process
    group only carries the barrier and the max-over-ranks timing."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
        return ws, rank, local, dist
    return 1, 0, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step, ms_per_step, world):
    """Whole-job throughput: every rank processes its own batch; the slowest
    rank's step time (already maxed over ranks) bounds the job."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------------------
# measurements
# ----------------------------------------------------------------------------
def measure_kernel_only(binding, w, sets, stream, steps):
    """Average duration of each kernel of the plan, timed alone (ms per launch)."""
    n_splits, chunk, kernel = binding.fmha_fwd_plan(w.batch, w.n_h, w.n_kv_h, w.T, w.s_k, w.hd, w.window,
                                                    w.causal, with_kernel=True)
    out = {"n_splits": n_splits, "kv_chunk": chunk, "kernel": kernel}
    if n_splits == 1:
        def fwd(i):
            q, k, v, o, lse = sets[i]
            binding.fmha_fwd(q, k, v, o, lse, scale=w.scale, window=w.window, causal=w.causal, stream=stream)
        out["decode_ms"] = graph_time(fwd, len(sets), steps, stream) / steps
        out["merge_ms"] = 0.0
        return out
    # The same kernels in the same configuration as fmha_fwd: its hd-512
    # tensor-core path keeps fp16 partials (FMHA_PARTS_F16), the others fp32.
    f16 = kernel == "fwd_tc_wide" and w.hd == 512
    out["parts_format"] = "f16" if f16 else "f32"
    parts = []
    for (q, k, v, o, lse) in sets:
        op = torch.empty((n_splits, w.batch, w.n_h, w.T, w.hd), dtype=torch.float16 if f16 else torch.float32,
                         device="cuda")
        lp = torch.empty((n_splits, w.batch, w.n_h, w.T), dtype=torch.float32, device="cuda")
        rp = torch.empty((n_splits, w.batch, w.n_h, w.T, 2), dtype=torch.float32, device="cuda") if f16 else None
        parts.append((op, lp, rp))

    def split(i):
        q, k, v, o, lse = sets[i]
        op, lp, rp = parts[i]
        if f16:
            binding.fmha_fwd_splitkv_f16(q, k, v, chunk, op, lp, rp, scale=w.scale, window=w.window,
                                         causal=w.causal, stream=stream)
        else:
            binding.fmha_fwd_splitkv(q, k, v, chunk, op, lp, scale=w.scale, window=w.window, causal=w.causal,
                                     stream=stream)

    def merge(i):
        q, k, v, o, lse = sets[i]
        op, lp, rp = parts[i]
        if f16:
            binding.fmha_merge_f16(op, lp, rp, o, lse, stream=stream)
        else:
            binding.fmha_merge(op, lp, o, lse, stream=stream)

    split(0)
    merge(0)
    out["decode_ms"] = graph_time(split, len(sets), steps, stream) / steps
    out["merge_ms"] = graph_time(merge, len(sets), steps, stream) / steps
    return out


def run_explicit_split(binding, w, chunk, steps, stream):
    """ms per step of fmha_fwd_splitkv (chunks of `chunk` keys) + fmha_merge,
    graph-replayed over rotating inputs (> 2x L2)."""
    sets, _ = rotating_sets(w, 2)
    _, n = binding.fmha_split_layout(w.T, w.s_k, w.window, chunk)
    parts = []
    for _s in sets:
        op = torch.empty((n, w.batch, w.n_h, w.T, w.hd), dtype=torch.float32, device="cuda")
        lp = torch.empty((n, w.batch, w.n_h, w.T), dtype=torch.float32, device="cuda")
        parts.append((op, lp))

    def step(i):
        q, k, v, o, lse = sets[i]
        binding.fmha_fwd_splitkv(q, k, v, chunk, parts[i][0], parts[i][1], scale=w.scale, window=w.window,
                                 causal=w.causal, stream=stream)
        binding.fmha_merge(parts[i][0], parts[i][1], o, lse, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3):
            step(i % len(sets))
    ms = graph_time(step, len(sets), steps, stream) / steps
    binding.fmha_check_device_status(stream)
    return ms, n


def run_workload(binding, w, steps, warmup, stream, dist=None, sampler=None):
    sets, l2 = rotating_sets(w, 2)

    def fwd(i):
        q, k, v, o, lse = sets[i]
        binding.fmha_fwd(q, k, v, o, lse, scale=w.scale, window=w.window, causal=w.causal, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            fwd(i % len(sets))
    torch.cuda.synchronize()
    binding.fmha_check_device_status(stream)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.time()
    ms = graph_time(fwd, len(sets), steps, stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(dist)
    binding.fmha_check_device_status(stream)
    ms = max_over_ranks(ms, dist)
    kern = measure_kernel_only(binding, w, sets, stream, steps)
    single = kern["n_splits"] == 1
    res = {"ms_total": ms, "ms_per_step": ms / steps, "t0": t0, "t1": t1, "n_sets": len(sets), "l2_bytes": l2,
           "launches_per_step": 1 if single else 2}
    res.update(kern)
    del sets
    torch.cuda.empty_cache()
    return res


def run_e2e(binding, w, steps, stream):
    """The public C ABI with host buffers (fmha_fwd_host): every step copies its
    Q, K and V from page-locked host memory, runs the forward and copies O and
    LSE back.  Steps alternate between two streams, so one step's host-to-device
    copies overlap the previous step's kernels and device-to-host copies; the
    inputs rotate over host sets larger than 256 MB in total, so no step reads
    them from the host's caches."""
    one = sum(t.numel() * t.element_size() for t in inputs.make_inputs(w, seed=99))
    n_sets = max(2, min(16, -(-(256 << 20) // one), (1 << 30) // max(one, 1)))
    host = [tuple(t.pin_memory() for t in inputs.make_inputs(w, seed=99 + i)) for i in range(n_sets)]
    streams = [stream, torch.cuda.Stream()]
    outs = [(torch.empty(host[0][0].shape, dtype=torch.bfloat16).pin_memory(),
             torch.empty((w.batch, w.n_h, w.T), dtype=torch.float32).pin_memory()) for _ in streams]

    def step(i):
        q, k, v = host[i % n_sets]
        o, lse = outs[i % 2]
        binding.fmha_fwd_host(q, k, v, o, lse, scale=w.scale, window=w.window, causal=w.causal,
                              stream=streams[i % 2])

    # Every host set (on both streams) makes its first DMA here, not in the timed region.
    for i in range(2 * n_sets + 2):
        step(i)
    torch.cuda.synchronize()
    e0, e1, e_side = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                      torch.cuda.Event())
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for i in range(steps):
        step(i)
    e_side.record(streams[1])
    streams[0].wait_event(e_side)
    e1.record(streams[0])
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    q, k, v = host[0]
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = outs[0][0].numel() * 2 + outs[0][1].numel() * 4
    return ms, h2d, d2h


def h2d_link_gbs(stream, nbytes):
    """Host-to-device bandwidth of one page-locked copy of `nbytes` (about one
    step's inputs), best of 10, measured in the same run as the e2e figure: the
    ceiling the e2e step time is set against."""
    nbytes = max(1 << 20, int(nbytes))
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = float("inf")
    with torch.cuda.stream(stream):
        dst.copy_(src, non_blocking=True)
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
    return nbytes / (best * 1e-3) / 1e9


def cpu_baseline(w, budget_s=15.0):
    """The fp64 oracle on the host cores over a bounded sample of the workload."""
    import numpy as np
    import oracle
    q, k, v = inputs.make_inputs(w, seed=7)
    qb, kb, vb = inputs.bf16_bits(q), inputs.bf16_bits(k), inputs.bf16_bits(v)
    total_rows = w.batch * w.n_h * w.T
    # calibrate on a small slice of rows, then size the sample to the budget
    probe = inputs.sample_rows(w, min(total_rows, 64), seed=1)
    t = time.time()
    oracle.attention_rows(qb, kb, vb, probe, w.scale, w.window, w.causal)
    per_row = max(1e-7, (time.time() - t) / len(probe))
    n_rows = int(max(1, min(total_rows * 2000, budget_s / per_row)))
    done = 0
    t = time.time()
    while done < n_rows:
        chunk = min(total_rows, n_rows - done)
        rows = np.arange(chunk, dtype=np.int64) if chunk == total_rows else inputs.sample_rows(w, chunk, seed=done)
        oracle.attention_rows(qb, kb, vb, rows, w.scale, w.window, w.causal)
        done += chunk
    el = time.time() - t
    frac = done / total_rows
    gbs = algo_bytes(w) * frac / el / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": "%d query rows (%.3g passes over the %s workload's %d rows) in %.1f s, fp64, OpenMP"
                      % (done, frac, w.name, total_rows, el),
            "seconds": el, "tflops": algo_flops(w) * frac / el / 1e12}


def roofline_obj(bytes_per_launch, ms, hbm_peak, peak_kind, traffic):
    achieved = bytes_per_launch / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": traffic, "peak_source": peak_kind}


def run_sweep():
    """The MHA shape sweep (batch 4, 16 heads, hd x T x s_k, K x 3): GB/s and
    TFLOP/s per point, one JSON line each."""
    from head_attention_forward_fmha_gb300 import binding
    binding.load()
    hbm_peak, bf16_peak, _, peak_kind = peaks()
    stream = torch.cuda.Stream()
    for w in inputs.sweep():
        b, f = algo_bytes(w), algo_flops(w)
        est = b / (hbm_peak * 1e9)
        steps = int(min(200, max(10, 2e-3 / max(est, 1e-7))))
        r = run_workload(binding, w, steps, 3, stream)
        sec = r["ms_per_step"] * 1e-3
        print(json.dumps({
            "workload": w.name, "hd": w.hd, "T": w.T, "s_k": w.s_k, "steps": steps,
            "us_per_step": round(r["ms_per_step"] * 1e3, 2), "GB/s": round(b / sec / 1e9, 1),
            "TFLOP/s": round(f / sec / 1e12, 2), "frac_hbm": round(b / sec / 1e9 / hbm_peak, 4),
            "frac_bf16_peak": round(f / sec / 1e12 / bf16_peak, 4),
            "frac_attainable": round(max(b / (hbm_peak * 1e9), f / (bf16_peak * 1e12)) / sec, 4),
            "kernel": r["kernel"], "n_splits": r["n_splits"], "peak_source": peak_kind}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--sweep", action="store_true",
                    help="time every point of the MHA shape sweep, one JSON line per point (not the bench line)")
    args = ap.parse_args()
    if args.sweep:
        return run_sweep()
    w = inputs.WORKLOADS[args.workload]
    hbm_peak, bf16_peak, bf16_sustained, peak_kind = peaks()
    bytes_step = algo_bytes(w)

    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        cb = None
        times = []
        for _ in range(max(0, args.warmup)):
            cpu_baseline(w, budget_s=0.5)
        for _ in range(args.steps):
            cb = cpu_baseline(w, budget_s=max(0.5, min(args.cpu_budget, 120.0 / max(1, args.steps))))
            times.append(cb)
        value = statistics.median(c["value"] for c in times)
        sec = sum(c["seconds"] for c in times)
        line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * bytes_step / (value * 1e9), 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": w.name, "batch": w.batch, "n_h": w.n_h, "n_kv_h": w.n_kv_h, "T": w.T,
                           "s_k": w.s_k, "hd": w.hd, "window": w.window, "causal": w.causal,
                           "world_size": ws},
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cb["cores"], "kind": "oracle",
                                 "sample": cb["sample"]},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "note": "fp64 CPU oracle timed on the host cores over %.1f s in total" % sec}
        print(json.dumps(line), flush=True)
        return 0

    from head_attention_forward_fmha_gb300 import binding
    binding.load()
    world, rank, local, dist = dist_setup(args)
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    res = run_workload(binding, w, args.steps, args.warmup, stream, dist)
    clocks = sampler.summary(res["t0"], res["t1"])
    e2e_steps = max(200, min(args.steps, 2000))
    e2e_ms, h2d, d2h = run_e2e(binding, w, e2e_steps, stream)
    e2e_ms = max_over_ranks(e2e_ms, dist)
    link_gbs = h2d_link_gbs(stream, h2d)

    secondary = {}
    if not args.no_secondary:
        for name, chunk in (("single_head_decode", 0), ("gqa_swa_decode", 512), ("causal_prefill", 0),
                            ("gqa_prefill", 0)):
            w2 = inputs.WORKLOADS[name]
            st = max(20, min(args.steps, 400))
            r2 = run_workload(binding, w2, st, 3, stream, dist)
            b2, f2 = algo_bytes(w2), algo_flops(w2)
            secondary[name] = {
                "ms_per_step": round(r2["ms_per_step"], 5),
                "GB/s": round(b2 / (r2["ms_per_step"] * 1e-3) / 1e9, 1),
                "TFLOP/s": round(f2 / (r2["ms_per_step"] * 1e-3) / 1e12, 2),
                "frac_hbm": round(b2 / (r2["ms_per_step"] * 1e-3) / 1e9 / hbm_peak, 4),
                "frac_bf16_peak": round(f2 / (r2["ms_per_step"] * 1e-3) / 1e12 / bf16_peak, 4),
                "frac_attainable": round(max(b2 / (hbm_peak * 1e9), f2 / (bf16_peak * 1e12)) /
                                         (r2["ms_per_step"] * 1e-3), 4),
                "n_splits": r2["n_splits"], "kv_chunk": r2["kv_chunk"], "kernel": r2["kernel"],
                "kernel_ms": round(r2["decode_ms"], 5), "merge_kernel_ms": round(r2["merge_ms"], 5),
                "traffic": recorded_traffic(r2["kernel"], name),
                "steps": st,
                "us_per_step": round(r2["ms_per_step"] * 1e3, 3),
            }
            if chunk:
                ms_c, n_c = run_explicit_split(binding, w2, chunk, st, stream)
                secondary[name]["split_%d" % chunk] = {
                    "ms_per_step": round(ms_c, 5), "n_splits": n_c,
                    "GB/s": round(b2 / (ms_c * 1e-3) / 1e9, 1),
                    "frac_hbm": round(b2 / (ms_c * 1e-3) / 1e9 / hbm_peak, 4)}
    sampler.stop()

    n = world
    value = aggregate_gbs(bytes_step, res["ms_per_step"], n)
    traffic = recorded_traffic(res["kernel"], w.name)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_h": w.n_h, "n_kv_h": w.n_kv_h, "T": w.T,
                   "s_k": w.s_k, "hd": w.hd, "window": w.window, "causal": w.causal,
                   "parallelism": "replicas%d" % n,
                   "l2": "inputs rotated over %d copies (%.0f MB > 2x L2 %.0f MB)"
                         % (res["n_sets"], res["n_sets"] * bytes_step / 1e6, res["l2_bytes"] / 1e6),
                   "timing": "CUDA graphs of fmha_fwd calls, CUDA events on the launching stream",
                   "n_splits": res["n_splits"], "kv_chunk": res["kv_chunk"],
                   "partials": res.get("parts_format", "none")},
        "roofline": dict(roofline_obj(bytes_step, res["decode_ms"], hbm_peak, peak_kind, traffic),
                         kernel=res["kernel"]),
        "kernels_ms": {res["kernel"]: round(res["decode_ms"], 6), "merge_lse": round(res["merge_ms"], 6)},
        "tflops": round(algo_flops(w) / (res["ms_per_step"] * 1e-3) / 1e12, 2),
        "e2e": {"value": round(bytes_step / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "h2d_link_gbs": round(link_gbs, 1),
                "h2d_floor_ms": round(h2d / (link_gbs * 1e9) * 1e3, 4)},
        "gpu_launches": args.steps * res["launches_per_step"],
        "clocks": clocks,
        "secondary": secondary,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
        for key in ("seconds", "tflops"):
            line["cpu_baseline"].pop(key, None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
