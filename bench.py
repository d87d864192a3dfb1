#!/usr/bin/env python
"""Benchmark of the routed MoE layer on one GB300: tokens/s and us/layer against the roofline.

Headline workload: the Qwen1.5-MoE-A2.7B-shaped prefill layer with its sigmoid-gated shared
expert (H=2048, routed I=1408, E=60, top-k=4, shared I_sh=5632, int4 nibble-8 experts with fp16
scales per 32 columns), T=4096 tokens -- the largest configuration, where the layer is a
grouped GEMM bound by the tensor cores.  A step = one moe_layer_forward call (router logits,
softmax top-k, dispatch, grouped int4 gate/up + SwiGLU and down GEMMs, combine onto the
residual) on one batch.  Weights stay resident in HBM; L2 reuse between steps is defeated by
cycling 2 independent layer replicas (311 MB of experts each, far above the 129 MB L2) and 4
distinct token batches.  Each step is timed by its own CUDA-event pair on the launching stream
(the median and the 10th / 90th percentiles are reported beside the whole region's mean).

``e2e`` is the same layer called from pinned host buffers (inputs in, y out, every step), the
copies overlapped with the neighbouring steps' layers on their own streams; its ``serial_value``
is the same loop on one stream.

The line also carries, as flat numbers in ``config``, the decode layers (Qwen3-30B-A3B-shaped
T=1/4/16 and GLM-class k=8/32 T=1/8, bound by HBM), the T=512 prefill layer, the router +
dispatch sweep and the skewed tiny layer; the fp64 CPU oracle is timed on the host cores, all
of them and one thread.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle instead, on bounded
token slices of the same workload.  Multi-GPU (torchrun) runs independent replicas, one per
rank: the layer has no cross-GPU exchange, so no collective touches the data path.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from mixture_experts_layer_09_gb300 import inputs as gen  # noqa: E402

METRIC = "MoE-layer tokens/s & us/layer at 1 GB300; % of HBM (decode) / TC (prefill) roof"
HEADLINE = dict(name="qwen15_moe_a2.7b_prefill_layer", H=2048, I=1408, E=60, k=4, I_sh=5632, T=4096)
DECODE = dict(name="qwen3_30b_a3b_decode_moe_layer", H=2048, I=768, E=128, k=8, T=(1, 4, 16))
N_PREFILL_REPLICAS, N_PREFILL_INPUTS = 2, 4
N_DECODE_REPLICAS, N_DECODE_INPUTS = 4, 16
BYTES_PER_EXPERT = lambda H, I: 3 * (H * I // 2) + 3 * (H * I // 32) * 2  # noqa: E731


def peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), \
            "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def prefill_flops(T, H, I, E, k, I_sh):
    """FLOPs of one prefill layer call: the two grouped GEMMs (routed and shared rows) and the
    router logits (E rows plus the shared gate row)."""
    gateup = 2.0 * (T * k * H * 2 * I + T * H * 2 * I_sh)
    down = 2.0 * (T * k * I * H + T * I_sh * H)
    return {"gemm_gateup": gateup, "gemm_down": down, "layer": gateup + down + 2.0 * T * H * (E + 1)}


# ----------------------------------------------------------------------------- clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, path, gpu_index):
        self.path, self.proc, self.gpu = path, None, gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing

def oracle_slices(n_tokens, seconds, threads, wl_dict=HEADLINE, seed=0):
    """The fp64 oracle as it stands, on consecutive token slices of a headline-shaped batch (each
    slice a batch of its own: routing, experts, shared expert and combine of those tokens), until
    about `seconds` of CPU time.  Returns (tokens/s, tokens, seconds, threads used, slices)."""
    import oracle
    oracle.build()
    oracle.set_threads(threads)
    w = wl_dict
    wl = gen.Workload(w["name"], n_tokens, w["H"], w["I"], w["E"], w["k"], I_sh=w.get("I_sh", 0), seed=seed)
    base = gen.draw_layer(wl)
    n_tok, dt, b = 0, 0.0, 0
    while b == 0 or dt < seconds:
        inp = dataclasses.replace(base, x=gen.draw_x(seed + 3000 + b, n_tokens, w["H"])) if b else base
        t0 = time.perf_counter()
        oracle.layer_forward(inp)
        dt += time.perf_counter() - t0
        n_tok += n_tokens
        b += 1
    return n_tok / dt, n_tok, dt, oracle.get_threads(), b


def run_reference(args, rank):
    """The fp64 CPU oracle as it stands, timed on every host core this process may use: each
    step is one slice of 8 tokens of the headline workload, run through the whole layer."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    oracle.set_threads(threads)
    w, n = HEADLINE, 8
    base = gen.draw_layer(gen.Workload(w["name"], n, w["H"], w["I"], w["E"], w["k"], I_sh=w["I_sh"]))
    slices = [dataclasses.replace(base, x=gen.draw_x(3000 + i, n, w["H"]),
                                  residual=gen.draw_residual(3100 + i, n, w["H"])) for i in range(4)]

    def step(i):
        oracle.layer_forward(slices[i % len(slices)])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    tps = n * args.steps / dt
    sample = f"{args.steps} slices of {n} tokens of the T={w['T']}-token workload, {threads} threads"
    line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w['name']} H={w['H']} I={w['I']} E={w['E']} k={w['k']} I_sh={w['I_sh']} "
                                   f"T={w['T']}",
                       "impl_note": f"fp64 C oracle on {threads} host threads"},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- timing

def timed_steps(torch, fn, steps, warmup, dist=None):
    """W untimed warm-up calls, then exactly `steps` calls, each between its own CUDA events on
    the current stream, the region bracketed by a barrier and a synchronize on both sides.
    Returns total seconds (max over ranks) and per-call microseconds."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for i in range(steps):
        fn(warmup + i)
        ev[i + 1].record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    per = [1e3 * ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total = ev[0].elapsed_time(ev[steps]) / 1e3
    return reduce_max(dist, total, "cuda"), per


def pipelined_e2e(torch, layers, xd, rd, T, H, steps, warmup, dist=None):
    """End-to-end step loop through pinned host buffers (x and the residual in, y out, every
    step), copies overlapped with the neighbouring steps' layers: a copy-in stream, the compute
    stream and a copy-out stream, two device buffers of each, events for the hand-offs.  The
    region runs from a synchronized start to the last output copy's completion; returns total
    seconds (max over ranks)."""
    n_in = len(xd)
    xh = [t.cpu().pin_memory() for t in xd]
    rh = [t.cpu().pin_memory() for t in rd]
    yh = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    xin = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    rin = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    yd = [torch.empty((T, H), dtype=torch.float32, device="cuda") for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_cmp = torch.cuda.current_stream()

    def run(n0, n):
        ev_in = {}   # inputs of step i on the device
        ev_cmp = {}  # layer of step i done (its inputs free, its y ready)
        ev_out = {}  # y of step i copied out
        for j in range(n):
            i = n0 + j
            b = i % 2
            with torch.cuda.stream(s_in):
                if j >= 2:
                    s_in.wait_event(ev_cmp[i - 2])  # the buffer's previous layer has read it
                xin[b].copy_(xh[i % n_in], non_blocking=True)
                rin[b].copy_(rh[i % n_in], non_blocking=True)
                ev_in[i] = torch.cuda.Event()
                ev_in[i].record(s_in)
            s_cmp.wait_event(ev_in[i])
            if j >= 2:
                s_cmp.wait_event(ev_out[i - 2])  # the buffer's previous y has been copied out
            layers[i % len(layers)].forward(xin[b], rin[b], y=yd[b])
            ev_cmp[i] = torch.cuda.Event()
            ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                yh[b].copy_(yd[b], non_blocking=True)
                ev_out[i] = torch.cuda.Event()
                ev_out[i].record(s_out)
        s_cmp.wait_stream(s_in)
        s_cmp.wait_stream(s_out)

    run(0, warmup)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_cmp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    run(warmup, steps)
    e1.record(s_cmp)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return reduce_max(dist, e0.elapsed_time(e1) / 1e3, "cuda")


def serial_e2e(torch, layers, xd, rd, T, H, steps, warmup, dist=None):
    """The end-to-end step on one stream: copy x and the residual in, the layer, copy y out."""
    n_in = len(xd)
    xh = [t.cpu().pin_memory() for t in xd]
    rh = [t.cpu().pin_memory() for t in rd]
    yh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    xin = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    rin = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    yd = torch.empty((T, H), dtype=torch.float32, device="cuda")

    def step(i):
        xin.copy_(xh[i % n_in], non_blocking=True)
        rin.copy_(rh[i % n_in], non_blocking=True)
        layers[i % len(layers)].forward(xin, rin, y=yd)
        yh.copy_(yd, non_blocking=True)

    total, _ = timed_steps(torch, step, steps, warmup, dist)
    return total


def summary(per_us):
    a = np.asarray(per_us, dtype=np.float64)
    return {"median_us": float(np.median(a)), "p10_us": float(np.percentile(a, 10)),
            "p90_us": float(np.percentile(a, 90)), "mean_us": float(a.mean()), "calls": int(a.size)}


def graph_steps(torch, step, n_graphs, steps, warmup):
    """The same calls captured as CUDA graphs (one per input index) and replayed."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graphs = []
    for i in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(i)
        graphs.append(g)
    _, per = timed_steps(torch, lambda i: graphs[i % n_graphs].replay(), steps, warmup)
    del graphs
    return per


def kernel_times(torch, moe, step, steps):
    """Per-kernel device time: the library's CUDA-event pairs around each of its launches, on
    the launching stream.  {name: (total ms, launches)}."""
    moe.moe_profile_enable(True)
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    kern = moe.moe_profile_read()
    moe.moe_profile_enable(False)
    return kern


# ----------------------------------------------------------------------------- ncu traffic

# DRAM traffic of a kernel from an ncu capture, valid while the sources it was built from are
# unchanged: profiles/dram_traffic.txt holds lines "kernel bytes_per_unit unit sha256 note", the
# hash taken over KERNEL_SOURCES by source_hash(); unit "expert" scales by the distinct experts a
# launch streamed, unit "launch" is the bench's launch as captured.
KERNEL_SOURCES = {
    "gateup_gemv": ("gemv.cu", "quant.cuh", "async.cuh", "common.cuh", "fp4.cuh", "internal.h"),
    "down_gemv_combine": ("gemv.cu", "quant.cuh", "async.cuh", "common.cuh", "fp4.cuh", "internal.h"),
    "gemm_gateup": ("gemm_sm100.cu", "tcgen05.cuh", "async.cuh", "common.cuh", "fp4.cuh", "internal.h"),
    "gemm_down": ("gemm_sm100.cu", "tcgen05.cuh", "async.cuh", "common.cuh", "fp4.cuh", "internal.h"),
}


def source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, ()):
        with open(os.path.join(ROOT, "mixture_experts_layer_09_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel, units=1.0):
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if kernel not in KERNEL_SOURCES or not os.path.exists(p):
        return None
    for ln in open(p):
        parts = ln.split(None, 4)
        if len(parts) >= 4 and not ln.startswith("#") and parts[0] == kernel and parts[3] == source_hash(kernel):
            per = float(parts[1])
            scale = units if parts[2] == "expert" else 1.0
            return {"bytes": per * scale, "note": (parts[4].strip() if len(parts) > 4 else "")}
    return None


# ----------------------------------------------------------------------------- secondary workloads

def _to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def measure_decode(torch, moe, args, seed0):
    """Qwen3-30B-A3B-shaped decode layers, T = 1, 4, 16: 4 replicas of 340 MB cycled with 16
    input batches; median of per-call CUDA-event times, plain launches and CUDA-graph replay."""
    from mixture_experts_layer_09_gb300.run_case import upload
    hbm = peaks()[0]
    D = DECODE
    H, I, E, k = D["H"], D["I"], D["E"], D["k"]
    layers = [upload(torch, moe, gen.Workload("d", max(D["T"]), H, I, E, k), seed0 + rep)
              for rep in range(N_DECODE_REPLICAS)]
    out, kern16 = {}, None
    for T in D["T"]:
        xs = [_to_dev(torch, gen.draw_x(seed0 + 500 + i, T, H)) for i in range(N_DECODE_INPUTS)]
        rs = [_to_dev(torch, gen.draw_residual(seed0 + 700 + i, T, H)) for i in range(N_DECODE_INPUTS)]
        y = torch.empty((T, H), dtype=torch.float32, device="cuda")
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")

        def step(i):
            layers[i % N_DECODE_REPLICAS].forward(xs[i % N_DECODE_INPUTS], rs[i % N_DECODE_INPUTS], y=y,
                                                  topk_ids_out=ids)

        n = max(50, args.steps)
        _, per = timed_steps(torch, step, n, args.warmup)
        perg = graph_steps(torch, step, N_DECODE_INPUTS, n, args.warmup)
        nd = []
        for i in range(N_DECODE_INPUTS):
            step(i)
            nd.append(int(torch.unique(ids).numel()))
        nd = float(np.mean(nd))
        s, sg = summary(per), summary(perg)
        us = min(s["median_us"], sg["median_us"])
        layer_bytes = nd * BYTES_PER_EXPERT(H, I) + E * H * 2 + T * H * (2 + 2 + 4)
        out[f"T={T}"] = {"us_per_layer": us, "plain_median_us": s["median_us"], "graph_median_us": sg["median_us"],
                         "p10_us": s["p10_us"], "p90_us": s["p90_us"], "tokens_per_s": T / (us * 1e-6),
                         "mean_distinct_experts": nd, "layer_bytes": layer_bytes,
                         "hbm_frac": layer_bytes / (us * 1e-6) / 1e9 / hbm}
        kern = kernel_times(torch, moe, step, n)
        out[f"T={T}"]["kernels_us_per_step"] = {nm: 1e3 * v[0] / n for nm, v in kern.items()}
        if T == 16:
            kern16 = kern
            kb = {"gateup_gemv": nd * (2 * I * H // 2 + 2 * I * (H // 32) * 2) + T * H * 2 + T * (H // 32) * 8
                  + T * k * I * 4,
                  "down_gemv_combine": nd * (H * I // 2 + H * (I // 32) * 2) + T * k * I * 2
                  + T * k * (I // 32) * 8 + T * H * 2 + T * H * 4}
            kf = {}
            for name, b in kb.items():
                if name in kern16:
                    kus = 1e3 * kern16[name][0] / max(kern16[name][1], 1)
                    kf[name] = {"us": kus, "bytes": b, "hbm_frac": b / (kus * 1e-6) / 1e9 / hbm}
            out["T=16"]["kernels"] = kf
    del layers
    torch.cuda.empty_cache()
    return out


def measure_norm(torch, moe, args, seed0):
    """The layer with its RMSNorm output (moe_layer_forward_norm) beside the plain layer call,
    on the T=1 and T=16 decode layers (GEMV arm: the norm is one more launch) and the T=4096
    prefill layer (tensor arm: the combine norms its rows)."""
    from mixture_experts_layer_09_gb300.run_case import upload
    out = {}
    D, P = DECODE, HEADLINE
    cases = [("decode_t1", gen.Workload("d", 1, D["H"], D["I"], D["E"], D["k"]), N_DECODE_REPLICAS,
              N_DECODE_INPUTS, 1500),
             ("decode_t16", gen.Workload("d", 16, D["H"], D["I"], D["E"], D["k"]), N_DECODE_REPLICAS,
              N_DECODE_INPUTS, 1500),
             ("prefill_t4096", gen.Workload("pn", 4096, P["H"], P["I"], P["E"], P["k"], I_sh=P["I_sh"]),
              N_PREFILL_REPLICAS, N_PREFILL_INPUTS, 1700)]
    for name, wl, n_rep, n_in, xseed in cases:
        H, T = wl.H, wl.T
        layers = [upload(torch, moe, wl, seed0 + 80 + rep) for rep in range(n_rep)]
        gamma = torch.from_numpy(gen.bf16_bits(gen.rng(23, H).normal(1.0, 0.1, size=H).astype(np.float32))
                                 .view(np.int16)).view(torch.bfloat16).cuda()
        xs = [_to_dev(torch, gen.draw_x(xseed + i, T, H)) for i in range(n_in)]
        y = torch.empty((T, H), dtype=torch.float32, device="cuda")
        yn = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")

        def step_norm(i):
            layers[i % n_rep].forward(xs[i % n_in], None, y=y, norm_gamma=gamma, eps=1e-6, y_norm=yn)

        def step_plain(i):
            layers[i % n_rep].forward(xs[i % n_in], None, y=y)

        steps = max(50, args.steps)
        _, per_n = timed_steps(torch, step_norm, steps, args.warmup)
        _, per_p = timed_steps(torch, step_plain, steps, args.warmup)
        del layers
        torch.cuda.empty_cache()
        us_n, us_p = summary(per_n)["median_us"], summary(per_p)["median_us"]
        out[name] = {"us_per_layer_with_rmsnorm": us_n, "us_per_layer_plain": us_p,
                     "tokens_per_s_with_rmsnorm": T / (us_n * 1e-6)}
    return out


def measure_glm(torch, moe, args):
    """GLM-class decode layers (H=6144, I=2048, E=256, all experts resident: 5.4 GB, far above
    L2), k=8 and k=32, T=1 and T=8, 8 distinct inputs cycled so that routing changes."""
    from mixture_experts_layer_09_gb300.run_case import upload
    hbm = peaks()[0]
    H, I, E = 6144, 2048, 256
    bpe = BYTES_PER_EXPERT(H, I)
    out = {"workload": f"glm_class_decode_moe_layer H={H} I={I} E={E}", "bytes_per_expert": bpe}
    base = upload(torch, moe, gen.Workload("g", 8, H, I, E, 8), 70)
    for k in (8, 32):
        for T in (1, 8):
            layer = moe.MoeLayer(base.W_r, base.experts, None, k, T)
            xs = [_to_dev(torch, gen.draw_x(1300 + i, T, H)) for i in range(8)]
            ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
            y = torch.empty((T, H), dtype=torch.float32, device="cuda")

            def step(i):
                layer.forward(xs[i % 8], None, y=y, topk_ids_out=ids)

            _, per = timed_steps(torch, step, max(50, args.steps), args.warmup)
            nd = []
            for i in range(8):
                step(i)
                nd.append(int(torch.unique(ids).numel()))
            nd = float(np.mean(nd))
            s = summary(per)
            gbs = (nd * bpe + E * H * 2 + T * H * 8) / (s["median_us"] * 1e-6) / 1e9
            out[f"k={k},T={T}"] = {"us_per_layer": s["median_us"], "p10_us": s["p10_us"], "p90_us": s["p90_us"],
                                   "tokens_per_s": T / (s["median_us"] * 1e-6), "mean_distinct_experts": nd,
                                   "hbm_gbs": gbs, "hbm_frac": gbs / hbm}
    del base
    torch.cuda.empty_cache()
    return out


def measure_router_sweep(torch, moe, args):
    """Router + dispatch sweep: bf16 logits ~N(0,1)*2, k=8, E in {32..256}, T in {1..16384}; each
    timed call (moe_router_topk then moe_dispatch) follows an untimed write of 256 MB, so L2
    holds nothing of it; the split per kernel comes from a second pass with per-launch events.
    Algorithmic bytes: T*E*2 + T*k*8 + T*k*12 + (E+1)*4."""
    hbm = peaks()[0]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    k, iters = 8, 20
    out = {}
    for E in (32, 64, 128, 256):
        for T in (1, 64, 1024, 16384):
            L = torch.from_numpy(gen.draw_logits(5, T, E).view(np.int16)).view(torch.bfloat16).cuda()
            ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
            w = torch.empty((T, k), dtype=torch.float32, device="cuda")
            counts = torch.empty(E, dtype=torch.int32, device="cuda")
            offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
            perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
            inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
            ws = torch.zeros(moe.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

            def call(variant=False):
                if variant:
                    moe.moe_router_topk_v(L, E, k, ids, w, sel_bias=bias, renormalize=False, scale=2.5)
                else:
                    moe.moe_router_topk(L, E, k, ids, w)
                moe.moe_dispatch(ids, E, counts, offsets, perm, inv, ws)

            def timed(variant=False):
                per = []
                for i in range(iters + 3):
                    flush.fill_(i & 0xFF)
                    e0.record()
                    call(variant)
                    e1.record()
                    torch.cuda.synchronize()
                    if i >= 3:
                        per.append(e0.elapsed_time(e1) * 1e3)
                return float(np.median(per))

            bias = None
            us = timed()
            moe.moe_profile_enable(True)
            for i in range(iters):
                flush.fill_(i & 0xFF)
                call()
            torch.cuda.synchronize()
            kern = moe.moe_profile_read()
            moe.moe_profile_enable(False)
            ab = T * E * 2 + T * k * 8 + T * k * 12 + (E + 1) * 4
            gbs = ab / (us * 1e-6) / 1e9
            out[f"E={E},T={T}"] = {"us": us, "gbs": gbs, "hbm_frac": gbs / hbm,
                                   "kernels_us": {n: 1e3 * v[0] / iters for n, v in kern.items()}}
            if E == 256 and T == 16384:
                # the router variant: selection bias, weights not renormalised, scaled
                bias = torch.from_numpy(gen.rng(6, E).normal(0.0, 0.5, size=E).astype(np.float32)).cuda()
                us = timed(True)
                gbs = (ab + E * 4) / (us * 1e-6) / 1e9
                out[f"E={E},T={T},bias,unnormalised,scale=2.5"] = {"us": us, "gbs": gbs, "hbm_frac": gbs / hbm}
    del flush
    return out


def measure_skewed_layer(torch, moe, args):
    """Tiny-layer shape at T=8192 with Zipf(1.1)-skewed expert popularity (bias channel): both
    roofs reported; the weights (8 experts, 0.4 MB) stay in L2 by nature."""
    hbm, tc, _, _ = peaks()
    wl = gen.WORKLOADS["tiny_zipf_t8192"]
    inp = gen.draw_layer(wl)
    layer = upload_inputs(torch, moe, inp)
    x = _to_dev(torch, inp.x)
    y = torch.empty((wl.T, wl.H), dtype=torch.float32, device="cuda")
    _, per = timed_steps(torch, lambda i: layer.forward(x, None, y=y), max(50, args.steps), args.warmup)
    us = summary(per)["median_us"]
    flops = wl.T * (wl.k * 6 * wl.H * wl.I + 2 * wl.E * wl.H)
    act_bytes = wl.T * wl.H * (2 + 4)
    return {"workload": f"tiny_zipf_t8192 H={wl.H} I={wl.I} E={wl.E} k={wl.k} T={wl.T} (Zipf 1.1 popularity)",
            "us_per_layer": us, "tokens_per_s": wl.T / (us * 1e-6),
            "tflops": flops / (us * 1e-6) / 1e12, "tc_frac": flops / (us * 1e-6) / 1e12 / tc,
            "act_gbs": act_bytes / (us * 1e-6) / 1e9, "act_hbm_frac": act_bytes / (us * 1e-6) / 1e9 / hbm}


def measure_mxfp4(torch, moe, args):
    """MXFP4 routed experts (e2m1 codes, expanded ue8m0 scales; the int4 shared expert kept):
    the Qwen3-30B-A3B-shaped decode layer at T=16 (2 replicas of 340 MB cycled with 8 inputs)
    and the Qwen1.5-MoE-A2.7B-shaped prefill layer at T=4096 (2 replicas of 300 MB)."""
    from mixture_experts_layer_09_gb300.run_case import upload
    hbm, tc, _, _ = peaks()
    out = {}
    H, I, E, k, T = 2048, 768, 128, 8, 16
    layers = [upload(torch, moe, gen.Workload("m", T, H, I, E, k, fmt=gen.FMT_MXFP4), 80 + r) for r in range(2)]
    xs = [_to_dev(torch, gen.draw_x(1700 + i, T, H)) for i in range(8)]
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")

    def step(i):
        layers[i % 2].forward(xs[i % 8], None, y=y, topk_ids_out=ids)

    _, per = timed_steps(torch, step, max(50, args.steps), args.warmup)
    nd = []
    for i in range(8):
        step(i)
        nd.append(int(torch.unique(ids).numel()))
    us = summary(per)["median_us"]
    gbs = (np.mean(nd) * BYTES_PER_EXPERT(H, I) + E * H * 2 + T * H * 8) / (us * 1e-6) / 1e9
    out["qwen3_30b_decode_t16_mxfp4"] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
                                         "mean_distinct_experts": float(np.mean(nd)), "hbm_gbs": gbs,
                                         "hbm_frac": gbs / hbm}
    del layers
    P = HEADLINE
    T = P["T"]
    layers = [upload(torch, moe, gen.Workload("mp", T, P["H"], P["I"], P["E"], P["k"], I_sh=P["I_sh"],
                                              fmt=gen.FMT_MXFP4), 90 + r) for r in range(2)]
    xs = [_to_dev(torch, gen.draw_x(1900 + i, T, P["H"])) for i in range(4)]
    y = torch.empty((T, P["H"]), dtype=torch.float32, device="cuda")
    _, per = timed_steps(torch, lambda i: layers[i % 2].forward(xs[i % 4], None, y=y), max(20, args.steps // 2),
                         args.warmup)
    us = summary(per)["median_us"]
    fl = prefill_flops(T, P["H"], P["I"], P["E"], P["k"], P["I_sh"])["layer"]
    out["qwen15_prefill_t4096_mxfp4"] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
                                         "layer_tflops": fl / (us * 1e-6) / 1e12,
                                         "layer_tc_frac": fl / (us * 1e-6) / 1e12 / tc}
    del layers
    torch.cuda.empty_cache()
    return out


def upload_inputs(torch, moe, inp):
    """A MoeLayer from drawn layer inputs (routed experts only)."""
    def q4(m):
        return moe.upload_q4(m.q, m.s, m.fmt)

    ex = inp.experts
    E = moe.Experts(ex.E, ex.H, ex.I, q4(ex.gate), q4(ex.up), q4(ex.down))
    return moe.MoeLayer(_to_dev(torch, inp.W_r), E, None, inp.wl.k, inp.wl.T)


def reduce_max(dist, v: float, device) -> float:
    """The largest of every rank's v: a replicated job takes as long as its slowest rank.  No
    process group (one rank): v itself."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Seed base of a rank's replicas and inputs: every rank holds independent layers."""
    return 1000 * rank


def job_value(world: int, tokens_per_step: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return world * tokens_per_step * steps / seconds


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import torch

    import mixture_experts_layer_09_gb300 as moe
    from mixture_experts_layer_09_gb300.run_case import upload
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    moe.build()
    P = HEADLINE
    H, I, E, k, I_sh, T = P["H"], P["I"], P["E"], P["k"], P["I_sh"], P["T"]
    seed0 = rank_seed(rank)
    hbm, tc, tc_sus, src = peaks()

    # ---- resident weights: independent layer replicas of the headline workload
    layers = [upload(torch, moe, gen.Workload("p", T, H, I, E, k, I_sh=I_sh), seed0 + 50 + r)
              for r in range(N_PREFILL_REPLICAS)]
    xd = [_to_dev(torch, gen.draw_x(seed0 + 900 + i, T, H)) for i in range(N_PREFILL_INPUTS)]
    rd = [_to_dev(torch, gen.draw_residual(seed0 + 950 + i, T, H)) for i in range(N_PREFILL_INPUTS)]
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")

    def step(i):
        layers[i % N_PREFILL_REPLICAS].forward(xd[i % N_PREFILL_INPUTS], rd[i % N_PREFILL_INPUTS], y=y)

    # SM clocks are sampled (nvidia-smi, 200 ms) over the whole measurement phase, which
    # contains the timed region; the samples go to $BENCH_CLOCKS_DIR (default: the temp dir)
    clocks = Clocks(os.path.join(os.environ.get("BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_bench_r{rank}.csv"), local)
    clocks.start()
    n0 = moe.moe_launch_count()
    total_s, per = timed_steps(torch, step, args.steps, args.warmup, dist)
    launches = (moe.moe_launch_count() - n0) * args.steps / (args.steps + args.warmup)
    head = summary(per)
    perg = graph_steps(torch, step, N_PREFILL_INPUTS, args.steps, args.warmup)
    graph = summary(perg)
    kern = kernel_times(torch, moe, step, args.steps)

    # end to end through host buffers: every step copies its x and residual in from pinned host
    # memory, runs the layer and copies y out, as a serving loop would: on three streams, step
    # i + 1's input copies and step i - 1's output copy overlap step i's layer (double-buffered
    # device inputs and outputs, ordered by events)
    e2e_s = pipelined_e2e(torch, layers, xd, rd, T, H, args.steps, args.warmup, dist)
    # the same without the overlap (one stream: copy in, layer, copy out), reported beside it
    e2e_serial_s = serial_e2e(torch, layers, xd, rd, T, H, args.steps, args.warmup, dist)
    del layers, xd, rd
    torch.cuda.empty_cache()

    # ---- the other workloads (reported beside the headline)
    extra = {}
    if not args.no_extra:
        extra["decode"] = measure_decode(torch, moe, args, seed0)
        extra["decode_glm"] = measure_glm(torch, moe, args)
        extra["prefill_t512"] = measure_prefill_t512(torch, moe, args, seed0)
        extra["with_rmsnorm"] = measure_norm(torch, moe, args, seed0)
        extra["router_dispatch_sweep"] = measure_router_sweep(torch, moe, args)
        extra["skewed_layer"] = measure_skewed_layer(torch, moe, args)
        extra["mxfp4"] = measure_mxfp4(torch, moe, args)
    clk = clocks.stop()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    fl = prefill_flops(T, H, I, E, k, I_sh)
    ms_step = 1e3 * total_s / args.steps
    value = job_value(world, T, args.steps, total_s)
    dom = max(kern, key=lambda n: kern[n][0])
    dom_us = 1e3 * kern[dom][0] / max(kern[dom][1], 1)
    if dom in ("gemm_gateup", "gemm_down"):
        ach = fl[dom] / (dom_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": tc, "unit": "TFLOP/s", "frac": ach / tc,
                "peak_source": f"bf16 dense burst, {src} (the MMAs take fp16 operands, same dense rate)",
                "algorithmic_flops": fl[dom], "kernel_us": dom_us}
    else:
        roof = {"bound": "tensor", "kernel": dom, "achieved": None, "peak": tc, "unit": "TFLOP/s", "frac": None,
                "kernel_us": dom_us, "note": "dominant kernel is not a GEMM"}
    tr = dram_traffic(dom)
    roof["traffic"] = tr["bytes"] if tr else None
    roof["traffic_note"] = tr["note"] if tr else "no ncu capture of this kernel's current source"
    kus = {n: 1e3 * v[0] / max(v[1], 1) for n, v in kern.items()}
    cfg = {"workload": f"{P['name']} H={H} I={I} E={E} k={k} I_sh={I_sh} T={T}", "global_batch": T * world,
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
           "l2": f"{N_PREFILL_REPLICAS} layer replicas x {(E * BYTES_PER_EXPERT(H, I) + BYTES_PER_EXPERT(H, I_sh)) / 1e6:.0f}"
                 f" MB of experts cycled with {N_PREFILL_INPUTS} distinct batches (inputs larger than L2)",
           "us_per_layer": ms_step * 1e3, "median_us": head["median_us"], "p10_us": head["p10_us"],
           "p90_us": head["p90_us"], "graph_median_us": graph["median_us"],
           "layer_tflops": fl["layer"] / (head["median_us"] * 1e-6) / 1e12,
           "layer_tc_frac": fl["layer"] / (head["median_us"] * 1e-6) / 1e12 / tc}
    for name in ("gemm_gateup", "gemm_down"):
        if name in kus:
            cfg[f"{name}_us"] = kus[name]
            cfg[f"{name}_tc_frac"] = fl[name] / (kus[name] * 1e-6) / 1e12 / tc
    for name, v in kus.items():
        cfg[f"kernel_us.{name}"] = v
    # flat copies of the other workloads' figures, so that they stay with the line's record
    if "decode" in extra:
        for Tb, d in extra["decode"].items():
            tag = f"decode_qwen3_{Tb.replace('=', '').lower()}"
            cfg[f"{tag}_us"] = d["us_per_layer"]
            cfg[f"{tag}_tok_s"] = d["tokens_per_s"]
            cfg[f"{tag}_hbm_frac"] = d["hbm_frac"]
            for kn, kv in d.get("kernels", {}).items():
                cfg[f"{tag}_{kn}_hbm_frac"] = kv["hbm_frac"]
    if "decode_glm" in extra:
        for key, d in extra["decode_glm"].items():
            if isinstance(d, dict):
                tag = "decode_glm_" + key.replace("=", "").replace(",", "_").lower()
                cfg[f"{tag}_us"] = d["us_per_layer"]
                cfg[f"{tag}_tok_s"] = d["tokens_per_s"]
                cfg[f"{tag}_hbm_frac"] = d["hbm_frac"]
    if "prefill_t512" in extra:
        d = extra["prefill_t512"]
        for key in ("us_per_layer", "tokens_per_s", "layer_tc_frac", "roof_frac"):
            cfg[f"prefill_t512_{key}"] = d[key]
    if "skewed_layer" in extra:
        cfg["skewed_t8192_us"] = extra["skewed_layer"]["us_per_layer"]
    if "router_dispatch_sweep" in extra:
        d = extra["router_dispatch_sweep"].get("E=256,T=16384")
        if d:
            cfg["router_dispatch_e256_t16384_us"] = d["us"]

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32", "data": "synthetic",
        "config": cfg,
        "roofline": roof,
        "gpu_launches": int(round(launches)),
        "clocks": clk,
        "e2e": {"value": job_value(world, T, args.steps, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * T * H * 2, "d2h_bytes_per_step": T * H * 4,
                "copies": "each step's input and output copies overlap the neighbouring steps' layers (3 streams)",
                "serial_value": job_value(world, T, args.steps, e2e_serial_s)},
        **extra,
    }
    if not args.no_cpu_baseline:
        import oracle
        cores = oracle.default_threads()
        v, n_tok, dt, thr, nb = oracle_slices(16, args.cpu_seconds, cores)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": f"{nb} batches of 16 tokens of the headline shape ({n_tok} tokens, "
                                          f"{dt:.1f} s) on {thr} threads"}
        v1, n1, dt1, thr1, nb1 = oracle_slices(4, args.cpu_seconds, 1)
        line["cpu_baseline_single_thread"] = {"value": v1, "unit": "tokens/s", "cores": thr1, "kind": "oracle",
                                              "sample": f"{nb1} batches of 4 tokens ({n1} tokens, {dt1:.1f} s)"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def measure_prefill_t512(torch, moe, args, seed0):
    """The prefill layer at T=512: about 34 rows per routed expert, so its roof is
    max(bytes / HBM, FLOPs / tensor peak); both fractions and that roof's are reported."""
    from mixture_experts_layer_09_gb300.run_case import upload
    P = HEADLINE
    H, I, E, k, I_sh, T = P["H"], P["I"], P["E"], P["k"], P["I_sh"], 512
    hbm, tc, _, _ = peaks()
    layers = [upload(torch, moe, gen.Workload("p5", T, H, I, E, k, I_sh=I_sh), seed0 + 60 + r)
              for r in range(N_PREFILL_REPLICAS)]
    xs = [_to_dev(torch, gen.draw_x(seed0 + 1100 + i, T, H)) for i in range(N_PREFILL_INPUTS)]
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")

    def step(i):
        layers[i % N_PREFILL_REPLICAS].forward(xs[i % N_PREFILL_INPUTS], None, y=y, topk_ids_out=ids)

    _, per = timed_steps(torch, step, max(50, args.steps), args.warmup)
    nd = []
    for i in range(N_PREFILL_INPUTS):
        step(i)
        nd.append(int(torch.unique(ids).numel()))
    kern = kernel_times(torch, moe, step, max(20, args.steps // 2))
    del layers
    torch.cuda.empty_cache()
    us = summary(per)["median_us"]
    fl = prefill_flops(T, H, I, E, k, I_sh)
    byts = float(np.mean(nd)) * BYTES_PER_EXPERT(H, I) + BYTES_PER_EXPERT(H, I_sh) + E * H * 2 + T * H * (2 + 2 + 4)
    roof_us = max(byts / (hbm * 1e9), fl["layer"] / (tc * 1e12)) * 1e6
    n = max(20, args.steps // 2)
    return {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
            "layer_tc_frac": fl["layer"] / (us * 1e-6) / 1e12 / tc,
            "layer_hbm_frac": byts / (us * 1e-6) / 1e9 / hbm, "roof_us": roof_us, "roof_frac": roof_us / us,
            "kernels_us": {nm: 1e3 * v[0] / n for nm, v in kern.items()}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU time of each oracle timing")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode, GLM-class, T=512, router/dispatch sweep, skewed and MXFP4 sections")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
