"""bench.py: the algorithmic units its numbers rest on, and its JSON line.

CPU only.  The byte and FLOP counts of the named workloads are checked against
figures derived independently from the workload definitions (one row of Q and
O per query, the attended keys of K and V, an fp32 LSE; 4 * hd FLOPs per
attended (row, key) pair), the roofline object against its definition, and
the reference arm (the oracle on the host cores) prints one JSON line with
every key of the contract.
"""
import json
import os
import subprocess
import sys

import pytest

import bench
from head_attention_forward_fmha_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# (workload, algorithmic bytes, FLOPs): single-head decode b1 h1 T1 s_k128 hd64;
# MQA decode b16 h128 kv1 s_k512 hd512; GQA window decode b32 h64 kv8 s_k8192
# hd128 with 4096 attended keys; causal prefill b8 h32 T128 after 384 cached
# keys, hd256, rows attending 385..512 keys.
EXPECTED = [
    ("single_head_decode", 64 * 2 + 2 * 128 * 64 * 2 + 64 * 2 + 4, 4 * 64 * 128),
    ("mqa_decode", 16 * 128 * 512 * 2 * 2 + 16 * 512 * 512 * 2 * 2 + 16 * 128 * 4, 4 * 512 * 16 * 128 * 512),
    ("gqa_swa_decode", 32 * 64 * 128 * 2 * 2 + 32 * 8 * 4096 * 128 * 2 * 2 + 32 * 64 * 4,
     4 * 128 * 32 * 64 * 4096),
    ("causal_prefill", 8 * 32 * 128 * 256 * 2 * 2 + 8 * 32 * 512 * 256 * 2 * 2 + 8 * 32 * 128 * 4,
     4 * 256 * 8 * 32 * sum(385 + t for t in range(128))),
]


@pytest.mark.parametrize("name,nbytes,flops", EXPECTED, ids=[e[0] for e in EXPECTED])
def test_algorithmic_units(name, nbytes, flops):
    w = inputs.WORKLOADS[name]
    assert bench.algo_bytes(w) == nbytes
    assert bench.algo_flops(w) == flops


def test_roofline_object():
    r = bench.roofline_obj(20e6, 0.01, 5000.0, "measured", 19e6)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 5000.0
    assert r["achieved"] == pytest.approx(2000.0) and r["frac"] == pytest.approx(0.4)
    assert r["traffic"] == 19e6


def test_aggregate_is_whole_job():
    assert bench.aggregate_gbs(1e9, 1.0, 4) == pytest.approx(4000.0)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "mqa_decode"
    assert d["higher_is_better"] is True and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["e2e"]["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
