"""Run one call of the path on one of the synthetic workloads, for timing and profiling.

    python -m paged_kv_cache_apply_gb300.run_case --workload mixed_b256_p4x512 --op decode --iters 3 --warmup 1

Uploads the seeded workload (see ``workloads``), runs ``--warmup`` untimed calls of the chosen
op, then ``--iters`` calls timed with CUDA events on the current stream, and prints one JSON
line with the mean time per call. Under a profiler, ``--warmup`` + ``--iters`` is the number of
launches of the op's kernel (decode: of each of its two kernels when it splits).
"""
from __future__ import annotations

import argparse
import json

OPS = ("rope", "prefill", "decode", "step")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="mixed_b256_p4x512",
                    choices=["tiny_chain", "decode_b64_page1", "prefill_b8_varlen", "long_decode_b4",
                             "mixed_b256_p4x512"])
    ap.add_argument("--op", default="step", choices=OPS)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--no-build", action="store_true", help="load the library as built")
    args = ap.parse_args(argv)

    import torch

    from . import build as B
    from . import device as DV
    from . import workloads as W

    if not args.no_build:
        B.build()
    wl = W.make(args.workload)
    dw = DV.DeviceWorkload.upload(wl)
    run = {"rope": dw.run_rope, "prefill": dw.run_prefill, "decode": dw.run_decode,
           "step": dw.run_step}[args.op]
    if args.op == "rope" and dw.rope is None or args.op == "prefill" and dw.prefill is None or \
            args.op == "decode" and dw.decode is None:
        raise SystemExit(f"workload {wl.name} has no {args.op} call")
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.iters):
        run()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    print(json.dumps({"workload": wl.name, "op": args.op, "iters": args.iters,
                      "warmup": args.warmup, "ms_per_call": round(ms, 5)}), flush=True)


if __name__ == "__main__":
    main()
