#!/usr/bin/env python
"""Benchmark of the paged KV-cache attention path on one GB300 (or N independent replicas).

A step is one pass of the whole path over the mixed continuous batch (256 decode requests with
seq_lens ~ U[128, 8192] plus 4 prefill chunks of 512 tokens; H=16, Hk=4, head_dim 128, bf16,
page 16): the fused RoPE + out_cache_loc cache write over all 2304 new tokens, varlen causal
prefill over the chunks, then split-K decode with its log-sum-exp merge.

value  = algorithmic bytes of the step (decode K/V + index + q/out, the rotate+write traffic,
         prefill q/out and K/V read once) / device time of the step (CUDA events, K steps).
e2e    = the same metric with the step's inputs copied from pinned host memory and its
         outputs read back inside the timed region: one copy each way per step (inputs and
         outputs each sit in one device buffer), double-buffered on two copy streams so that
         the copies of one step overlap the compute of its neighbours.
roofline: the decode call (partial kernel + merge) against the measured HBM copy bandwidth.
Every step reads ~2.2 GB of K/V, far more than the 129 MB L2, so no flush is needed.

--impl reference times the CPU oracle (test infrastructure) on the host cores on a bounded
sample of the same step and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn GB/s (% HBM peak); prefill attn TFLOP/s (% TC peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------------------
# algorithmic work of one step
# ---------------------------------------------------------------------------------------------


def step_work(wl, dec_sel=None, pre_rows=None, rope=True):
    """Bytes / FLOPs the step must move or compute (each counted once).

    decode: per cached token K+V of every KV head plus its 4-byte slot index; per request q
            in and decode_out.
    rope:   per token q,k,v read and q_out,k,v written, position + slot, its freqs row.
    prefill: q in and out, K/V of every key position read once; FLOPs 4*d*H per unmasked
            (query, key) pair (QK^T and PV).
    """
    pool = wl.pool
    esz = 2 if pool.dtype == "bf16" else 4
    H, Hk, D = wl.n_heads, pool.n_kv_heads, pool.head_dim
    out = {"decode_bytes": 0.0, "rope_bytes": 0.0, "prefill_bytes": 0.0, "prefill_flops": 0.0}
    if wl.decode is not None:
        sl = wl.decode.seq_lens if dec_sel is None else wl.decode.seq_lens[dec_sel]
        out["decode_bytes"] = float(sl.sum()) * (2 * Hk * D * esz + 4) + len(sl) * 2 * H * D * esz
    if rope and wl.rope is not None:
        T = wl.rope.n_tokens
        out["rope_bytes"] = T * (2.0 * (H + 2 * Hk) * D * esz + 8 + 4 * D)
    if wl.prefill is not None:
        p = wl.prefill
        q = (p.qo_indptr[1:] - p.qo_indptr[:-1]).astype("int64")
        k = (p.kv_indptr[1:] - p.kv_indptr[:-1]).astype("int64")
        pre = k - q
        if pre_rows is None:
            pairs = float((q * pre + q * (q + 1) // 2).sum())
            nq = float(q.sum())
            nk = float(k.sum())
        else:  # a subset of packed rows: each row attends prefix + its index + 1 keys
            import numpy as np
            b = np.searchsorted(p.qo_indptr, pre_rows, side="right") - 1
            i = pre_rows - p.qo_indptr[b]
            pairs = float((pre[b] + i + 1).sum())
            nq = float(len(pre_rows))
            nk = float(k[np.unique(b)].sum())
        out["prefill_flops"] = 4.0 * D * H * pairs
        out["prefill_bytes"] = nq * 2 * H * D * esz + nk * 2 * Hk * D * esz
    out["total_bytes"] = out["decode_bytes"] + out["rope_bytes"] + out["prefill_bytes"]
    return out


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------


class ClockSampler:
    """SM clocks and clock-event reasons sampled during the timed region.

    A host thread polls NVML (libnvidia-ml.so.1 through ctypes; read-only queries) every
    `interval_s`, so that even a region of a few milliseconds holds several samples. Where NVML
    cannot be loaded, `nvidia-smi -lms 100` runs instead."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReasons bits
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device_index: int, interval_s: float = 0.001):
        self.idx = device_index
        self.interval = interval_s
        self.proc = None
        self.path = None
        self.window = None  # host wall-clock bounds of the timed region
        self.thread = None
        self.rows = []
        self.source = None

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def _nvml_handle(self):
        import ctypes as C
        nv = C.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = C.c_void_p()
        try:  # the CUDA device's own GPU, whatever CUDA_VISIBLE_DEVICES maps it to
            import torch
            uid = "GPU-" + str(torch.cuda.get_device_properties(self.idx).uuid)
            if nv.nvmlDeviceGetHandleByUUID(uid.encode(), C.byref(h)) == 0:
                return nv, h
        except Exception:
            pass
        if nv.nvmlDeviceGetHandleByIndex_v2(self.idx, C.byref(h)) != 0:
            raise OSError("no NVML handle")
        return nv, h

    def _poll(self, nv, h):
        import ctypes as C
        sm, smax, reasons = C.c_uint(), C.c_uint(), C.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        nv.nvmlDeviceGetMaxClockInfo(h, 1, C.byref(smax))  # NVML_CLOCK_SM
        while not self._stop:
            t = time.time()
            if nv.nvmlDeviceGetClockInfo(h, 1, C.byref(sm)) == 0 and \
                    get_reasons(h, C.byref(reasons)) == 0:
                names = [n for n, b in self.REASON_BITS.items() if reasons.value & b]
                self.rows.append((t, float(sm.value), float(smax.value), names))
            time.sleep(self.interval)

    def start(self):
        self._stop = False
        try:
            import threading
            nv, h = self._nvml_handle()
            self.thread = threading.Thread(target=self._poll, args=(nv, h), daemon=True)
            self.thread.start()
            self.source = f"NVML every {self.interval * 1e3:g} ms"
            return
        except Exception:
            self.thread = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi -lms 100"
        except Exception:
            self.proc = None

    def _read_smi(self):
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]),
                                 [n for n, v in zip(names, parts[6:10]) if v.lower().startswith("active")]))
                except ValueError:
                    continue
        os.unlink(self.path)
        return rows

    def stop(self):
        if self.thread is not None:
            time.sleep(0.01)
            self._stop = True
            self.thread.join(timeout=5)
            rows = self.rows
        elif self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()
            rows = self._read_smi()
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        return self.summarize(rows)

    def summarize(self, rows):
        """rows: (host time, SM MHz, max SM MHz, [active reasons]) samples."""
        # only samples taken inside the timed region count; with none there (a region shorter
        # than the sampling interval), the nearest ones do and the record says so
        inside = [r for r in rows if self.window and self.window[0] <= r[0] <= self.window[1]]
        use = inside if inside else rows
        sm = [r[1] for r in use]
        smax = [r[2] for r in use]
        reasons = set(n for r in use for n in r[3])
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use),
                "in_timed_region": bool(inside), "source": self.source}


# ---------------------------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# ---------------------------------------------------------------------------------------------


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# the CPU oracle as a baseline (test infrastructure, timed as it stands)
# ---------------------------------------------------------------------------------------------


def oracle_sample(wl, dec_fraction=1.0, pre_fraction=1.0):
    import numpy as np
    dsel = None
    prows = None
    if wl.decode is not None and dec_fraction < 1.0:
        n = max(1, int(round(wl.decode.batch * dec_fraction)))
        dsel = np.arange(n, dtype=np.int32)
    if wl.prefill is not None and pre_fraction < 1.0:
        tot = wl.prefill.total_q
        n = max(1, int(round(tot * pre_fraction)))
        prows = np.linspace(0, tot - 1, n).astype(np.int32)
    return dsel, prows


def run_oracle_step(wl, kl, vl, dsel, prows):
    import numpy as np
    import oracle
    r = wl.rope
    q = oracle.rope_kv_write(r.q, r.k, r.v, r.freqs_cis, r.position_ids, r.out_cache_loc, kl, vl)
    if wl.prefill is not None:
        p = wl.prefill
        qp = q[p.q_token_offset: p.q_token_offset + p.total_q]
        oracle.prefill(qp, kl, vl, wl.pool.req_to_token, p.req_pool_indices, p.qo_indptr,
                       p.kv_indptr, rows=prows)
    if wl.decode is not None:
        d = wl.decode
        qd = np.ascontiguousarray(q[: d.batch])
        oracle.decode(qd, kl, vl, wl.pool.req_to_token, d.req_pool_indices, d.seq_lens, sel=dsel)


def cpu_baseline(wl, dec_fraction, pre_fraction, repeats=1, min_seconds=10.0):
    import numpy as np
    import oracle
    oracle.build()
    kl = np.ascontiguousarray(wl.pool.k_buffer[0]).copy()
    vl = np.ascontiguousarray(wl.pool.v_buffer[0]).copy()
    dsel, prows = oracle_sample(wl, dec_fraction, pre_fraction)
    work = step_work(wl, dsel, prows)
    t0 = time.perf_counter()
    run_oracle_step(wl, kl, vl, dsel, prows)
    first = time.perf_counter() - t0
    # repeat the sample until about min_seconds of host work have been timed
    repeats = max(repeats, min(30, int(math.ceil(min_seconds / max(first, 1e-3)))))
    t0 = time.perf_counter()
    for _ in range(repeats):
        run_oracle_step(wl, kl, vl, dsel, prows)
    dt = (time.perf_counter() - t0) / repeats
    desc = (f"rope+write of all {wl.rope.n_tokens} tokens, prefill of "
            f"{'all' if prows is None else len(prows)} of {wl.prefill.total_q} rows, decode of "
            f"{'all' if dsel is None else len(dsel)} of {wl.decode.batch} requests")
    out = {"value": work["total_bytes"] / dt / 1e9, "unit": "GB/s",
           "cores": oracle.num_threads(), "kind": "oracle", "sample": desc,
           "seconds_per_sample": round(dt, 4), "repeats": repeats}
    # the same oracle on one host thread, over a 1/16 sample of the decode requests and prefill rows
    threads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        d1, p1 = oracle_sample(wl, dec_fraction / 16, pre_fraction / 16)
        w1 = step_work(wl, d1, p1)
        t0 = time.perf_counter()
        run_oracle_step(wl, kl, vl, d1, p1)
        one = time.perf_counter() - t0
        reps = max(1, min(20, int(math.ceil(min_seconds / 2 / max(one, 1e-3)))))
        t0 = time.perf_counter()
        for _ in range(reps):
            run_oracle_step(wl, kl, vl, d1, p1)
        dt1 = (time.perf_counter() - t0) / reps
        out["single_thread"] = {"value": w1["total_bytes"] / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                                "sample": f"rope+write of all {wl.rope.n_tokens} tokens, prefill of "
                                          f"{len(p1)} rows, decode of {len(d1)} requests",
                                "seconds_per_sample": round(dt1, 4), "repeats": reps}
    finally:
        oracle.set_num_threads(threads)
    return out


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from paged_kv_cache_apply_gb300 import build as B
    if rank == 0:
        B.build()
    barrier(world)
    B.build()
    import paged_kv_cache_apply_gb300 as A
    from paged_kv_cache_apply_gb300 import device as DV
    from paged_kv_cache_apply_gb300 import workloads as W

    wl = W.mixed_b256_p4x512()
    dw = DV.DeviceWorkload.upload(wl)
    work = step_work(wl)
    chunk, n_splits = A.astr_decode_plan(dw.decode["kv"], wl.n_heads)
    launches_per_step = 3 + (1 if n_splits > 1 else 0)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()  # the prefill runs here, concurrently with the decode

    for _ in range(args.warmup):
        dw.run_step(side_stream=side, fused=True)
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    # Per-op times (rows, roofline): K steps with the ops run one after another on one stream
    # and an event between them, so that each kernel is timed on the GPU to itself.
    torch.cuda.synchronize()
    for i in range(K):
        ev[i][0].record(stream)
        dw.run_rope()
        ev[i][1].record(stream)
        dw.run_prefill()
        ev[i][2].record(stream)
        dw.run_decode()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    rope_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    pre_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    dec_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    serial_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in ev)
    # the same ops' marginal costs in a stream (no event between kernels; L2 flushed before each)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rope_mg = marginal_ms(dw.run_rope, flush, stream, K)
    pre_mg = marginal_ms(dw.run_prefill, flush, stream, K)
    dec_mg = marginal_ms(dw.run_decode, flush, stream, min(K, 20))
    del flush

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(K):  # the step: events at the two ends only (an event between kernels costs)
        dw.run_step(side_stream=side, fused=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark(wall0, time.time())
    barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    ms_step = max_over_ranks(total_ms / K, world, torch.device("cuda", local))

    # End to end: every step copies its inputs from pinned host memory and reads its outputs
    # back. Inputs and outputs each sit in one device buffer (one copy each way), and there are
    # two of each, so that step i+1's inputs go up on one copy stream and step i's outputs come
    # down on another while the compute stream runs step i. Events keep a buffer from being
    # overwritten while a step still uses it. The timed region runs from the first step's
    # upload to the last step's read-back.
    import copy as _copy
    arenas_in = [dw.pack(dw.step_inputs())]
    arenas_out = [dw.pack(dw.step_outputs())]
    bind = [(dw.rope, dw.prefill, dw.decode)]
    arenas_in.append(torch.zeros_like(arenas_in[0]))
    arenas_out.append(torch.zeros_like(arenas_out[0]))

    def rebound(d, arenas):  # a copy of step dict `d` whose arena views point at the other buffers
        if d is None:
            return None
        e = dict(d)
        e.pop("c", None)
        if "kv" in e:
            e["kv"] = _copy.copy(e["kv"])
        for src, dst in arenas:
            lo, hi = src.data_ptr(), src.data_ptr() + src.numel()
            def moved(t):
                if isinstance(t, torch.Tensor) and lo <= t.data_ptr() < hi:
                    off = t.data_ptr() - lo
                    return dst[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                return t
            for k in list(e):
                e[k] = moved(e[k])
            if "kv" in e:
                for name, v in list(vars(e["kv"]).items()):
                    setattr(e["kv"], name, moved(v))
        return e

    ref_out = arenas_out[0].to("cpu")  # the outputs of the device-timed steps, for the check below
    pairs = [(arenas_in[0], arenas_in[1]), (arenas_out[0], arenas_out[1])]
    bind.append(tuple(rebound(d, pairs) for d in bind[0]))
    h_in = arenas_in[0].to("cpu").pin_memory()
    h_out = [torch.empty_like(arenas_out[0], device="cpu").pin_memory() for _ in range(2)]
    h2d = arenas_in[0].numel()
    d2h = arenas_out[0].numel()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, step_done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_step(i):
        x = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(step_done[x])  # step i-2 no longer reads these inputs
            arenas_in[x].copy_(h_in, non_blocking=True)
            in_ready[x].record(s_in)
        stream.wait_event(in_ready[x])
        if i >= 2:
            stream.wait_event(out_free[x])  # step i-2's outputs have been read back
        dw.rope, dw.prefill, dw.decode = bind[x]
        dw.run_step(side_stream=side, fused=True)
        step_done[x].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(step_done[x])
            h_out[x].copy_(arenas_out[x], non_blocking=True)
            out_free[x].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(K):
        e2e_step(i)
    e1.record(s_out)  # after the last read-back, which follows every other op of the loop
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, world, torch.device("cuda", local))
    dw.rope, dw.prefill, dw.decode = bind[0]
    # every step recomputes the same outputs: both read-back buffers must hold them byte for byte
    e2e_verified = all(torch.equal(h, ref_out) for h in h_out[:min(K, 2)])

    peaks, peak_kind = read_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    dec_gbs = work["decode_bytes"] / (dec_ms * 1e-3) / 1e9
    rope_gbs = work["rope_bytes"] / (rope_ms * 1e-3) / 1e9
    pre_tflops = work["prefill_flops"] / (pre_ms * 1e-3) / 1e12
    rope_gbs_mg = work["rope_bytes"] / (rope_mg * 1e-3) / 1e9
    pre_tflops_mg = work["prefill_flops"] / (pre_mg * 1e-3) / 1e12
    dec_gbs_mg = work["decode_bytes"] / (dec_mg * 1e-3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as f:
                td = json.load(f)
            if td.get("kernel_source_sha") == _decode_source_sha():
                traffic = td.get("dram_bytes_per_launch_full_size")
        except Exception:
            traffic = None

    if rank != 0:
        return
    out = {
        "metric": METRIC,
        "value": round(world * work["total_bytes"] / (ms_step * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "mixed continuous batch: 256 decode requests seq_lens~U[128,8192] + 4 "
                        "prefill chunks x 512 tokens, fused rope+out_cache_loc write of 2304 "
                        "tokens; n_heads 16, n_kv_heads 4, head_dim 128, bf16, page 16, "
                        "freqs max_len 8192",
            "l2": "no flush: each step reads ~2.2 GB of K/V (> 129 MB L2)",
            "parallelism": f"replicas x{world}",
            "streams": "second stream: rope + write of the 2048 prefill tokens, then the prefill; "
                       "main stream, concurrently: the decode with the rope + write of its 256 "
                       "new tokens folded in (astr_decode_attention_rope); the step ends when "
                       "both are done",
            "timing": "rows: each op's marginal cost in a stream (K pairs of an L2 flush (256 MB "
                      "written, then read) "
                      "and the op between two events, minus K flushes; median of 3), with the "
                      "time between an event on each side of the op as ms_between_events; "
                      "roofline: K steps with the ops serialised and an event between them; "
                      "value: K steps with CUDA events at the ends only",
            "decode_split_chunk": chunk, "decode_splits": n_splits,
        },
        "rows": {
            "rope_kv_write": {"ms": round(rope_mg, 5), "GB/s": round(rope_gbs_mg, 1),
                              "frac_hbm": round(rope_gbs_mg / hbm, 4),
                              "ms_between_events": round(rope_ms, 5),
                              "frac_hbm_between_events": round(rope_gbs / hbm, 4)},
            "prefill": {"ms": round(pre_mg, 5), "TFLOP/s": round(pre_tflops_mg, 2),
                        "frac_tc": round(pre_tflops_mg / tc, 4),
                        "ms_between_events": round(pre_ms, 5),
                        "frac_tc_between_events": round(pre_tflops / tc, 4)},
            "decode": {"ms": round(dec_mg, 5), "GB/s": round(dec_gbs_mg, 1),
                       "frac_hbm": round(dec_gbs_mg / hbm, 4),
                       "ms_between_events": round(dec_ms, 5),
                       "frac_hbm_between_events": round(dec_gbs / hbm, 4)},
            "serialised_step": {"ms": round(serial_ms, 5)},
        },
        "roofline": {"kernel": ("astr_decode_attention call: decode_tc_kernel partials + "
                                "split_merge_kernel (timed together, traffic of both)")
                               if n_splits > 1 else
                               "astr_decode_attention call: decode_tc_kernel, requests unsplit "
                               "(no merge launched)",
                     "bound": "hbm",
                     "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(dec_gbs / hbm, 4), "traffic": traffic,
                     "peak_source": f"{peak_kind} (hbm_gbs)"},
        "e2e": {"value": round(world * work["total_bytes"] / (e2e_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "outputs_verified": bool(e2e_verified),
                "pipelining": "two input and two output buffers; copies on two streams overlap compute"},
        "gpu_launches": int(K * launches_per_step),
        "clocks": clk,
    }
    if world == 1 and not args.no_configs:
        out["configs"] = config_rows(args, peaks, local)
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, 1.0, 1.0)
    print(json.dumps(out), flush=True)


def flush_l2(buf, i):
    """Write `buf` (larger than the 129 MB L2), then read it back: L2 then holds only clean
    lines of `buf`, so the next op reads its inputs from HBM and does not pay for writing the
    flush's dirty lines back."""
    import torch
    buf.fill_(i & 0xFF)
    buf.view(torch.float32).sum()


def marginal_ms(fn, flush, stream, K, rounds=3):
    """The cost of one call of `fn` in a stream of launches: K pairs (an L2 flush, then `fn`)
    between two CUDA events, minus K flushes alone, the median over `rounds` alternations.

    A short kernel timed between its own pair of events also carries the events' cost: on GB300
    an event on each side of a trivial kernel measures 4.4-6 us, most of a 10 us op. Here the
    launches follow one another with no event between them, as in a model's step, and the flush
    (flush_l2: a 256 MB write and read, larger than the 129 MB L2) makes every call read its
    inputs from HBM."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(with_fn):
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(K):
            flush_l2(flush, i)
            if with_fn:
                fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    diffs = []
    for _ in range(rounds):
        diffs.append(timed(True) - timed(False))
    return statistics.median(diffs)


def config_rows(args, peaks, local):
    """The other full-size configurations, one call each per step, timed on the GPU alone.

    decode_b64_page1 (page-size-1 decode) and long_decode_b4 (fixed 4096-token split-K decode
    with its merge) in GB/s of algorithmic bytes against the measured HBM copy bandwidth;
    prefill_b8_varlen (varlen causal prefill, half the requests resumed) in TFLOP/s of unmasked
    (query, key) pairs against the measured bf16 burst peak. Each of `args.steps` calls sits
    between its own pair of CUDA events on the launching stream after `args.warmup` untimed
    calls, and a 256 MB write and read flush L2 before every call (outside the events); that time is
    ms_between_events, and ms is the call's marginal cost in a stream (marginal_ms)."""
    import torch
    from paged_kv_cache_apply_gb300 import device as DV
    from paged_kv_cache_apply_gb300 import workloads as W
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tc = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = {}
    for name, op in (("decode_b64_page1", "decode"), ("prefill_b8_varlen", "prefill"),
                     ("long_decode_b4", "decode")):
        wl = W.make(name)
        dw = DV.DeviceWorkload.upload(wl)
        run = dw.run_decode if op == "decode" else dw.run_prefill
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
        K = args.steps
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        clocks = ClockSampler(local)
        clocks.start()
        wall0 = time.time()
        for i in range(K):
            flush_l2(flush, i)
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        clocks.mark(wall0, time.time())
        clk = clocks.stop()
        ms_ev = statistics.mean(a.elapsed_time(b) for a, b in ev)
        ms = marginal_ms(run, flush, stream, K)
        work = step_work(wl)
        row = {"op": op, "ms": round(ms, 5), "ms_between_events": round(ms_ev, 5),
               "workload": wl.description, "l2": "flushed before every call", "clocks": clk}
        if op == "decode":
            gbs = work["decode_bytes"] / (ms * 1e-3) / 1e9
            gbs_ev = work["decode_bytes"] / (ms_ev * 1e-3) / 1e9
            row.update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                        "frac_hbm_between_events": round(gbs_ev / hbm, 4),
                        "algorithmic_bytes": int(work["decode_bytes"]),
                        "split_chunk": wl.decode.split_chunk})
        else:
            tfs = work["prefill_flops"] / (ms * 1e-3) / 1e12
            tfs_ev = work["prefill_flops"] / (ms_ev * 1e-3) / 1e12
            row.update({"TFLOP/s": round(tfs, 2), "frac_tc": round(tfs / tc, 4),
                        "frac_tc_between_events": round(tfs_ev / tc, 4),
                        "algorithmic_flops": int(work["prefill_flops"])})
        out[name] = row
        del dw, wl
        torch.cuda.empty_cache()
    return out


def _decode_source_sha():
    import hashlib
    h = hashlib.sha256()
    # the partial kernel and its helpers, plus the merge kernel's source
    for f in ["decode_tc.cu", "tc_common.cuh", "astr_internal.cuh", "simt_attention.cu"]:
        with open(os.path.join(ROOT, "paged_kv_cache_apply_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------------------------


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_cache_apply_gb300 import workloads as W
    import numpy as np
    import oracle
    oracle.build()
    wl = W.mixed_b256_p4x512()
    kl = np.ascontiguousarray(wl.pool.k_buffer[0]).copy()
    vl = np.ascontiguousarray(wl.pool.v_buffer[0]).copy()
    dsel, prows = oracle_sample(wl, 1.0 / 16, 1.0 / 16)
    work = step_work(wl, dsel, prows)
    for _ in range(args.warmup):
        run_oracle_step(wl, kl, vl, dsel, prows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_step(wl, kl, vl, dsel, prows)
    dt = (time.perf_counter() - t0) / args.steps
    val = work["total_bytes"] / dt / 1e9
    sample = (f"per step: rope+write of all {wl.rope.n_tokens} tokens, prefill of {len(prows)} of "
              f"{wl.prefill.total_q} rows, decode of {len(dsel)} of {wl.decode.batch} requests")
    out = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "mixed continuous batch (same as the GPU arm), bounded sample",
                      "parallelism": "host cores (OpenMP)"},
           "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2500)  # about a second of timed work
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the rows of the page-1 decode, varlen prefill and long decode")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
