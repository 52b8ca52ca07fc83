"""Runs the GEMM on one shape a few times and prints the per-launch device time.

  python -m tensor_core_tiled_gb300.run_case --m 6144 --n 6144 --k 6144 [--launches 3]
      [--warmup 2] [--cta-group 2] [--tile-n 256] [--stages 6] [--group-m 8] [--max-ctas 0]
      [--stream-k 0|1|2] [--flush-l2]

Inputs are N(0,1) FP16 drawn on the device (no host generation), so the command is quick
to start; it is meant for profiling one kernel on a chosen shape and for tuning sweeps.
"""
import argparse
import json

import torch

import tensor_core_tiled_gb300 as tct


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--m", type=int, required=True)
    ap.add_argument("--n", type=int, required=True)
    ap.add_argument("--k", type=int, required=True)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--max-ctas", type=int, default=0)
    ap.add_argument("--cta-group", type=int, default=0)
    ap.add_argument("--stream-k", type=int, default=0, help="1 = whole tiles only, 2 = split the last wave")
    ap.add_argument("--flush-l2", action="store_true", help="write 512 MiB between launches")
    args = ap.parse_args()

    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(args.m, args.k, device="cuda", generator=g).half()
    B = torch.randn(args.k, args.n, device="cuda", generator=g).half()
    C = torch.empty(args.m, args.n, device="cuda")
    flush = torch.empty(128 << 20, device="cuda") if args.flush_l2 else None
    opts = dict(tile_n=args.tile_n, stages=args.stages, group_m=args.group_m, max_ctas=args.max_ctas,
                cta_group=args.cta_group, stream_k=args.stream_k)
    opts = {k: v for k, v in opts.items() if v}
    for _ in range(args.warmup):
        tct.matmul(A, B, C, **opts)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.launches):
        if flush is not None:
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        tct.matmul(A, B, C, **opts)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    st = tct.gemm_f16_f32_get_error()
    flops = 2.0 * args.m * args.n * args.k
    best = min(times)
    plan = tct.gemm_f16_f32_plan(args.m, args.n, args.k, **opts)
    print(json.dumps({"shape": [args.m, args.n, args.k], "opts": opts, "ms": times, "best_ms": best,
                      "tflops_best": flops / best / 1e9, "tflops_mean": flops / (sum(times) / len(times)) / 1e9,
                      "plan": plan, "device_status": st}))
    if st != tct.GEMM_OK:
        raise SystemExit(f"device status {st}")


if __name__ == "__main__":
    main()
