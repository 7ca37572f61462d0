"""The bench's host logic on CPU: the algorithmic work it divides by, and the reference arm's
JSON line (the oracle timed on the host cores)."""
import json
import os
import subprocess
import sys

import numpy as np

from paged_kv_cache_apply_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_step_work_counts_each_byte_and_pair_once():
    wl = W.mixed_b256_p4x512()
    w = bench.step_work(wl)
    H, Hk, D, esz = 16, 4, 128, 2
    d = wl.decode
    # decode: K and V of every KV head plus the 4-byte slot per cached token; q in, out
    assert w["decode_bytes"] == float(d.seq_lens.sum()) * (2 * Hk * D * esz + 4) + d.batch * 2 * H * D * esz
    # 2304 tokens: q, k, v read and q_out, k, v written, position + slot, the freqs row
    assert w["rope_bytes"] == 2304 * (2 * (H + 2 * Hk) * D * esz + 8 + 4 * D)
    # 4 chunks of 512 fresh tokens: 512 * 513 / 2 unmasked pairs each, 4 * D * H flops a pair
    assert w["prefill_flops"] == 4.0 * D * H * 4 * (512 * 513 // 2)
    # brute force over the causal mask of one resumed request
    q_len, kv_len = 37, 100
    pairs = sum(1 for i in range(q_len) for j in range(kv_len) if j <= kv_len - q_len + i)
    wl2 = W.make_case("bf16", 8, 2, 64, 16, [kv_len], [q_len])
    assert bench.step_work(wl2)["prefill_flops"] == 4.0 * 64 * 8 * pairs


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    for k in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"]:
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and np.isclose(cb["value"], line["value"])
    e = line["e2e"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0 and e["value"] == line["value"]


def test_clock_summary_keeps_the_timed_region_only():
    cs = bench.ClockSampler(0)
    cs.source = "test"
    cs.mark(10.0, 10.010)
    rows = [(9.99, 1000.0, 2070.0, []), (10.001, 2070.0, 2070.0, []),
            (10.004, 2055.0, 2070.0, ["sw_power_cap"]), (10.009, 2070.0, 2070.0, []),
            (10.02, 900.0, 2070.0, ["hw_slowdown"])]
    r = cs.summarize(rows)
    assert r["in_timed_region"] and r["samples"] == 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    cs.mark(20.0, 20.001)  # no sample inside: all of them count, and the record says so
    r = cs.summarize(rows)
    assert not r["in_timed_region"] and r["samples"] == 5
