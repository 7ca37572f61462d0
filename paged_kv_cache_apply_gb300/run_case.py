"""Run one call of the path on one of the synthetic workloads, for timing and profiling.

    python -m paged_kv_cache_apply_gb300.run_case --workload mixed_b256_p4x512 --op decode --iters 3 --warmup 1

Uploads the seeded workload (see ``workloads``), runs ``--warmup`` untimed calls of the chosen
op, then ``--iters`` calls timed with CUDA events on the current stream, and prints one JSON
line with the mean time per call. Under a profiler, ``--warmup`` + ``--iters`` is the number of
launches of the op's kernel (decode: of each of its two kernels when it splits).

``--op pool`` times the host page pool (no GPU): ``--iters`` request lifecycles of 1024 shared
system-prompt tokens plus 512 tokens of their own, page 16, each a match, an allocation, a
record of its tokens and a release, on a 65536-page pool.

``--op rope_backward`` times astr_rope_backward on the rope step's q and k (the gradients of
the training path have the same shapes). ``--op bind`` times astr_bind_tasks on the workload's prefill lengths (device q_lens / kv_lens
to indptrs and tile maps). ``--graph`` captures one call of the op into a CUDA graph after the
warm-up and times ``--iters`` replays of it instead.
"""
from __future__ import annotations

import argparse
import json

OPS = ("rope", "prefill", "decode", "step", "bind", "rope_backward", "pool")


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
    ap.add_argument("--graph", action="store_true", help="time replays of a captured call")
    args = ap.parse_args(argv)

    import numpy as np

    if args.op == "pool":
        return _time_pool(args)
    import torch

    from . import build as B
    from . import device as DV
    from . import workloads as W

    if not args.no_build:
        B.build()
    wl = W.make(args.workload)
    dw = DV.DeviceWorkload.upload(wl)
    need = {"bind": "prefill", "rope_backward": "rope"}.get(args.op, args.op)
    if need != "step" and getattr(dw, need) is None:
        raise SystemExit(f"workload {wl.name} has no {args.op} call")
    if args.op == "bind":
        from . import astr_bind_tasks
        p = wl.prefill
        ql = torch.from_numpy(np.diff(p.qo_indptr).astype(np.int32)).cuda()
        kl = torch.from_numpy(np.diff(p.kv_indptr).astype(np.int32)).cuda()
        qo, kv = torch.empty(ql.numel() + 1, dtype=torch.int32, device="cuda"), \
            torch.empty(ql.numel() + 1, dtype=torch.int32, device="cuda")
        tb = torch.empty(len(p.q_tile_to_batch), dtype=torch.int32, device="cuda")
        ti = torch.empty_like(tb)

        def run():
            astr_bind_tasks(ql, kl, qo, kv, tb, ti)
    elif args.op == "rope_backward":
        from . import astr_rope_backward
        r = dw.rope
        gq, gk = torch.empty_like(r["q"]), torch.empty_like(r["k"])

        def run():
            astr_rope_backward(r["q"], gq, r["k"], gk, r["freqs"], r["pos"])
    else:
        run = {"rope": dw.run_rope, "prefill": dw.run_prefill, "decode": dw.run_decode,
               "step": dw.run_step}[args.op]
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    call = run
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            run()
        call = g.replay
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.iters):
        call()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    print(json.dumps({"workload": wl.name, "op": args.op, "graph": bool(args.graph),
                      "iters": args.iters, "warmup": args.warmup, "ms_per_call": round(ms, 5)}),
          flush=True)


def _time_pool(args):
    import time

    import numpy as np

    from . import PagePool
    from . import build as B
    if not args.no_build:
        B.build()
    ps, shared, own = 16, 1024, 512
    pool = PagePool(65536, ps)
    rng = np.random.default_rng(7)
    system = rng.integers(0, 32000, shared)
    reqs = [np.concatenate([system, rng.integers(0, 32000, own)]).astype(np.int32)
            for _ in range(args.iters + args.warmup)]
    hits = 0

    def life(toks):
        hit = pool.match(toks[:-1])
        pages = np.concatenate([hit, pool.alloc((len(toks) + ps - 1) // ps - len(hit))])
        pool.record(toks, len(toks), pages)
        pool.release(pages)
        return len(hit)

    for t in reqs[:args.warmup]:
        life(t)
    t0 = time.perf_counter()
    for t in reqs[args.warmup:]:
        hits += life(t)
    us = (time.perf_counter() - t0) / max(args.iters, 1) * 1e6
    print(json.dumps({"op": "pool", "iters": args.iters, "tokens_per_request": shared + own,
                      "page_size": ps, "mean_hit_pages": round(hits / max(args.iters, 1), 1),
                      "us_per_request": round(us, 2), "stats": pool.stats()}), flush=True)


if __name__ == "__main__":
    main()
