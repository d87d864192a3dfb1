"""Run one routed MoE layer configuration on cuda:0 and report its time per layer.

    python -m mixture_experts_layer_09_gb300.run_case --workload qwen3_30b_decode_t16
    python -m mixture_experts_layer_09_gb300.run_case --shape 2048,1408,60,4,4096,5632 --arm gemm --time

Inputs are the seeded synthetic layers of ``inputs`` (random int4 experts, bf16 router,
bf16 tokens).  Without ``--time`` the layer runs ``--iters`` times and the script exits: the
form to put under a profiler.  With ``--time`` it runs ``--warmup`` untimed steps, then
``--iters`` steps between CUDA events on the launching stream, cycling ``--replicas``
independent weight sets so that L2 holds no weights from one step to the next, and prints
one JSON line with the time per layer and the per-kernel device times.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import inputs as gen

ARMS = {"auto": 0, "gemv": 1, "gemm": 2}


def parse_workload(args) -> gen.Workload:
    if args.shape:
        v = [int(s) for s in args.shape.split(",")]
        if len(v) not in (5, 6):
            raise SystemExit("--shape wants H,I,E,k,T[,I_sh]")
        H, I, E, k, T = v[:5]
        return gen.Workload(f"H{H}_I{I}_E{E}_k{k}_T{T}", T, H, I, E, k, I_sh=v[5] if len(v) > 5 else 0,
                            fmt=args.fmt)
    if args.workload not in gen.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; known: {', '.join(gen.WORKLOADS)}")
    return gen.WORKLOADS[args.workload]


def upload(torch, moe, wl: gen.Workload, seed: int):
    """Draws one seeded layer of the workload's shape and uploads it; returns a MoeLayer."""
    def dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype is not None else t).cuda()

    def q4(m):
        return moe.upload_q4(m.q, m.s, m.fmt)

    ex = gen.draw_experts(seed, wl.E, wl.H, wl.I, wl.fmt)
    W = moe.Experts(wl.E, wl.H, wl.I, q4(ex.gate), q4(ex.up), q4(ex.down))
    del ex
    W_r = dev(gen.draw_router(seed, wl.E, wl.H).view(np.int16), torch.bfloat16)
    sh = None
    if wl.I_sh:
        s = gen.draw_shared(seed, wl.H, wl.I_sh, fmt=wl.sh_fmt)
        sh = moe.Shared(wl.I_sh, q4(s.gate), q4(s.up), q4(s.down), dev(s.g.view(np.int16), torch.bfloat16))
    return moe.MoeLayer(W_r, W, sh, wl.k, wl.T)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="qwen3_30b_decode_t16")
    ap.add_argument("--shape", default="", help="H,I,E,k,T[,I_sh] instead of a named workload")
    ap.add_argument("--fmt", default="int4", choices=("int4", "mxfp4"), help="routed experts' format (--shape)")
    ap.add_argument("--arm", choices=list(ARMS), default="auto")
    ap.add_argument("--iters", type=int, default=4)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--replicas", type=int, default=1)
    ap.add_argument("--inputs", type=int, default=4)
    ap.add_argument("--time", action="store_true")
    args = ap.parse_args(argv)

    import torch

    import mixture_experts_layer_09_gb300 as moe

    wl = parse_workload(args)
    layers = [upload(torch, moe, wl, r) for r in range(max(1, args.replicas))]
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    xs = [to(gen.draw_x(100 + i, wl.T, wl.H)) for i in range(max(1, args.inputs))]
    y = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    arm = ARMS[args.arm]

    def step(i):
        layers[i % len(layers)].forward(xs[i % len(xs)], None, y=y, topk_ids_out=ids, arm=arm)

    if not args.time:
        distinct = []
        for i in range(args.iters):
            step(i)
            distinct.append(int(torch.unique(ids).numel()))
        torch.cuda.synchronize()
        print(json.dumps({"workload": wl.name, "iters": args.iters, "distinct_experts": distinct,
                          "y_mean_abs": float(y.abs().mean())}))
        return
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.iters):
        step(args.warmup + i)
    e1.record()
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / args.iters
    moe.moe_profile_enable(True)
    for i in range(args.iters):
        step(i)
    torch.cuda.synchronize()
    kern = moe.moe_profile_read()
    moe.moe_profile_enable(False)
    print(json.dumps({"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "I_sh": wl.I_sh,
                      "arm": args.arm, "us_per_layer": us, "tokens_per_s": wl.T / (us * 1e-6),
                      "kernels_us": {n: 1e3 * v[0] / args.iters for n, v in kern.items()}}))


if __name__ == "__main__":
    main()
