#!/usr/bin/env python
"""Benchmark of the routed MoE layer on one GB300: tokens/s and us/layer.

Workload: the Qwen3-30B-A3B-shaped decode layer (H=2048, I=768, E=128, top-k=8, no shared
expert, int4 nibble-8 experts with fp16 scales per 32 columns), batch T=16 tokens, synthetic
seeded inputs.  A step = one moe_layer_forward call (router logits, softmax top-k, dispatch,
fused int4 expert MLP with the combine in the down projection) on one batch.  Weights stay
resident in HBM; L2 reuse between steps is defeated by cycling 4 independent layer replicas
(340 MB of experts each, 4 x 340 MB > 4 x L2) and 16 distinct input batches.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle instead, on a
bounded sample of the same workload.  Multi-GPU (torchrun) runs independent replicas, one per
rank: the layer has no cross-GPU exchange, so no collective touches the data path.
"""
from __future__ import annotations

import argparse
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
WORKLOAD = dict(name="qwen3_30b_a3b_decode_moe_layer", H=2048, I=768, E=128, k=8, T=16)
SWEEP_T = (1, 4)
N_REPLICAS = 4
N_INPUTS = 16
BYTES_PER_EXPERT = lambda H, I: 3 * (H * I // 2) + 3 * (H * I // 32) * 2  # noqa: E731


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


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


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank):
    """The fp64 CPU oracle as it stands, timed on the host cores: each step is one token of
    the benchmark batch (routing of the whole batch, then that token's experts and combine)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = gen.Workload(WORKLOAD["name"], WORKLOAD["T"], WORKLOAD["H"], WORKLOAD["I"], WORKLOAD["E"], WORKLOAD["k"])
    inp = gen.draw_layer(wl)
    T = wl.T

    def step(i):
        mask = np.zeros(T, dtype=np.uint8)
        mask[i % T] = 1
        oracle.layer_forward(inp, token_mask=mask)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    tps = args.steps / dt
    line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.name} H={wl.H} I={wl.I} E={wl.E} k={wl.k} T={wl.T}",
                       "impl_note": "fp64 C oracle, single thread"},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} steps of 1 token of the T={T} batch"},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

# DRAM traffic of a kernel from an ncu capture, valid while the sources it was built from are
# unchanged: profiles/dram_traffic.txt holds lines "kernel bytes_per_unit unit sha256 note", the
# hash taken over KERNEL_SOURCES by source_hash(); the GEMV kernels' unit is one distinct expert
# streamed by the launch, so a launch's traffic is bytes_per_unit x its distinct experts.
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


def dram_traffic(kernel, units):
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


def time_layer(torch, layer, xs, steps, warmup, ids):
    """CUDA-event time per layer call over `steps` calls cycling the inputs `xs`, and the mean
    number of distinct experts those calls routed to."""
    T, H = xs[0].shape
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")

    def step(i):
        layer.forward(xs[i % len(xs)], None, y=y, topk_ids_out=ids)

    dt = time_loop(torch, step, steps, warmup)
    nd = []
    for i in range(len(xs)):
        step(i)
        nd.append(int(torch.unique(ids).numel()))
    return 1e6 * dt / steps, float(np.mean(nd))


def measure_norm(torch, moe, args, layers, T, H):
    """The decode layer with its RMSNorm output (moe_layer_forward_norm) over the same cycled
    replicas and inputs as the headline: us/layer with the extra pass."""
    gamma = torch.from_numpy(gen.bf16_bits(gen.rng(23, H).normal(1.0, 0.1, size=H).astype(np.float32))
                             .view(np.int16)).view(torch.bfloat16).cuda()
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    xs = [to(gen.draw_x(1500 + i, T, H)) for i in range(N_INPUTS)]
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    yn = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")

    def step(i):
        layers[i % len(layers)].forward(xs[i % N_INPUTS], None, y=y, norm_gamma=gamma, eps=1e-6, y_norm=yn)

    steps = max(10, args.steps // 2)
    dt = time_loop(torch, step, steps, args.warmup)
    return {"us_per_layer_with_rmsnorm": 1e6 * dt / steps, "tokens_per_s": T * steps / dt}


def measure_glm(torch, moe, args):
    """GLM-class decode layers (H=6144, I=2048, E=256, all experts resident: 5.4 GB, far above
    L2), k=8 and k=32, T=1 and T=8, 8 distinct inputs cycled so that routing changes."""
    from mixture_experts_layer_09_gb300.run_case import upload
    hbm, _, _ = peaks()
    H, I, E = 6144, 2048, 256
    bpe = BYTES_PER_EXPERT(H, I)
    out = {"workload": f"glm_class_decode_moe_layer H={H} I={I} E={E}", "bytes_per_expert": bpe}
    base = upload(torch, moe, gen.Workload("g", 8, H, I, E, 8), 70)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    for k in (8, 32):
        for T in (1, 8):
            layer = moe.MoeLayer(base.W_r, base.experts, None, k, T)
            xs = [to(gen.draw_x(1300 + i, T, H)) for i in range(8)]
            ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
            us, nd = time_layer(torch, layer, xs, max(10, args.steps // 2), args.warmup, ids)
            gbs = (nd * bpe + E * H * 2 + T * H * 8) / (us * 1e-6) / 1e9
            out[f"k={k},T={T}"] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6), "mean_distinct_experts": nd,
                                   "hbm_gbs": gbs, "hbm_frac": gbs / hbm}
    del base
    torch.cuda.empty_cache()
    return out


def measure_router_sweep(torch, moe, args):
    """Router + dispatch sweep: bf16 logits ~N(0,1)*2, k=8, E in {32..256}, T in {1..16384}; each
    timed call (moe_router_topk then moe_dispatch) follows an untimed write of 256 MB, so L2
    holds nothing of it.  Algorithmic bytes: T*E*2 + T*k*8 + T*k*12 + (E+1)*4."""
    hbm, _, _ = peaks()
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
            tot = 0.0
            for i in range(iters + 3):
                flush.fill_(i & 0xFF)
                e0.record()
                moe.moe_router_topk(L, E, k, ids, w)
                moe.moe_dispatch(ids, E, counts, offsets, perm, inv, ws)
                e1.record()
                torch.cuda.synchronize()
                if i >= 3:
                    tot += e0.elapsed_time(e1) * 1e3
            us = tot / iters
            gbs = (T * E * 2 + T * k * 8 + T * k * 12 + (E + 1) * 4) / (us * 1e-6) / 1e9
            out[f"E={E},T={T}"] = {"us": us, "gbs": gbs, "hbm_frac": gbs / hbm}
            if E == 256 and T == 16384:
                # the router variant: selection bias, weights not renormalised, scaled
                bias = torch.from_numpy(gen.rng(6, E).normal(0.0, 0.5, size=E).astype(np.float32)).cuda()
                tot = 0.0
                for i in range(iters + 3):
                    flush.fill_(i & 0xFF)
                    e0.record()
                    moe.moe_router_topk_v(L, E, k, ids, w, sel_bias=bias, renormalize=False, scale=2.5)
                    moe.moe_dispatch(ids, E, counts, offsets, perm, inv, ws)
                    e1.record()
                    torch.cuda.synchronize()
                    if i >= 3:
                        tot += e0.elapsed_time(e1) * 1e3
                us = tot / iters
                gbs = (T * E * 2 + E * 4 + T * k * 8 + T * k * 12 + (E + 1) * 4) / (us * 1e-6) / 1e9
                out[f"E={E},T={T},bias,unnormalised,scale=2.5"] = {"us": us, "gbs": gbs, "hbm_frac": gbs / hbm}
    del flush
    return out


def measure_skewed_layer(torch, moe, args):
    """Tiny-layer shape at T=8192 with Zipf(1.1)-skewed expert popularity (bias channel): both
    roofs reported; the weights (8 experts, 0.4 MB) stay in L2 by nature."""
    hbm, tc, _ = peaks()
    wl = gen.WORKLOADS["tiny_zipf_t8192"]
    inp = gen.draw_layer(wl)
    W_r, Ed = upload_layer(torch, moe, inp)
    layer = moe.MoeLayer(W_r, Ed, None, wl.k, wl.T)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    us, _ = time_layer(torch, layer, [x], max(10, args.steps // 2), args.warmup, ids)
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
    hbm, tc, _ = peaks()
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    out = {}
    H, I, E, k, T = 2048, 768, 128, 8, 16
    layers = [upload(torch, moe, gen.Workload("m", T, H, I, E, k, fmt=gen.FMT_MXFP4), 80 + r) for r in range(2)]
    xs = [to(gen.draw_x(1700 + i, T, H)) for i in range(8)]
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")

    def step(i):
        layers[i % 2].forward(xs[i % 8], None, y=y, topk_ids_out=ids)

    steps = max(10, args.steps // 2)
    dt = time_loop(torch, step, steps, args.warmup)
    nd = []
    for i in range(8):
        step(i)
        nd.append(int(torch.unique(ids).numel()))
    us = 1e6 * dt / steps
    gbs = (np.mean(nd) * BYTES_PER_EXPERT(H, I) + E * H * 2 + T * H * 8) / (us * 1e-6) / 1e9
    out["qwen3_30b_decode_t16_mxfp4"] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
                                         "mean_distinct_experts": float(np.mean(nd)), "hbm_gbs": gbs,
                                         "hbm_frac": gbs / hbm}
    del layers
    P = PREFILL
    T = 4096
    layers = [upload(torch, moe, gen.Workload("mp", T, P["H"], P["I"], P["E"], P["k"], I_sh=P["I_sh"],
                                              fmt=gen.FMT_MXFP4), 90 + r) for r in range(2)]
    xs = [to(gen.draw_x(1900 + i, T, P["H"])) for i in range(4)]
    y = torch.empty((T, P["H"]), dtype=torch.float32, device="cuda")

    def pstep(i):
        layers[i % 2].forward(xs[i % 4], None, y=y)

    dt = time_loop(torch, pstep, steps, args.warmup)
    us = 1e6 * dt / steps
    Hh, Ii, kk, Ish = P["H"], P["I"], P["k"], P["I_sh"]
    flops = 2.0 * T * (kk * 3 * Hh * Ii + 3 * Hh * Ish + Hh * (P["E"] + 1))
    out["qwen15_prefill_t4096_mxfp4"] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
                                         "layer_tflops": flops / (us * 1e-6) / 1e12,
                                         "layer_tc_frac": flops / (us * 1e-6) / 1e12 / tc}
    del layers
    torch.cuda.empty_cache()
    return out


PREFILL = dict(name="qwen15_moe_a2.7b_prefill_layer", H=2048, I=1408, E=60, k=4, I_sh=5632, T=(4096, 512))


def measure_prefill(torch, moe, args):
    """Prefill layer (grouped GEMM arm, tensor-core bound): us/layer, tokens/s and the fraction
    of the bf16 dense peak that the layer and its two GEMMs reach."""
    from mixture_experts_layer_09_gb300.run_case import upload
    P = PREFILL
    _, tc, src = peaks()
    res = {"workload": f"{P['name']} H={P['H']} I={P['I']} E={P['E']} k={P['k']} I_sh={P['I_sh']}"}
    reps = 2  # 2 x 300 MB of int4 weights cycled: more than L2
    layers = [upload(torch, moe, gen.Workload("p", max(P["T"]), P["H"], P["I"], P["E"], P["k"], I_sh=P["I_sh"]),
                     50 + r) for r in range(reps)]
    H, I, k, I_sh = P["H"], P["I"], P["k"], P["I_sh"]
    for T in P["T"]:
        to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
        xs = [to(gen.draw_x(900 + i, T, H)) for i in range(4)]
        y = torch.empty((T, H), dtype=torch.float32, device="cuda")

        def step(i):
            layers[i % reps].forward(xs[i % 4], None, y=y)

        steps = max(10, args.steps // 2)
        dt = time_loop(torch, step, steps, args.warmup)
        moe.moe_profile_enable(True)
        time_loop(torch, step, steps, 0)
        kern = moe.moe_profile_read()
        moe.moe_profile_enable(False)
        us = 1e6 * dt / steps
        fl = {"gemm_gateup": 2.0 * (T * k * H * 2 * I + T * H * 2 * I_sh),
              "gemm_down": 2.0 * (T * k * I * H + T * I_sh * H)}
        layer_flops = sum(fl.values()) + 2.0 * T * H * (P["E"] + 1)
        kus = {n: 1e3 * v[0] / steps for n, v in kern.items()}
        gem = {n: {"us": kus[n], "tflops": fl[n] / (kus[n] * 1e-6) / 1e12,
                   "frac": fl[n] / (kus[n] * 1e-6) / 1e12 / tc} for n in fl if n in kus}
        res[f"T={T}"] = {"us_per_layer": us, "tokens_per_s": T / (us * 1e-6),
                         "layer_tflops": layer_flops / (us * 1e-6) / 1e12,
                         "layer_tc_frac": layer_flops / (us * 1e-6) / 1e12 / tc,
                         "gemm": gem, "kernels_us": kus}
    res["peak_tflops"] = tc
    res["peak_source"] = f"bf16 dense burst, {src} (the MMAs take fp16 operands: same dense rate)"
    del layers
    torch.cuda.empty_cache()
    return res


def upload_layer(torch, moe, inp):
    def dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dtype) if dtype is not None else t).cuda()

    def q4(m):
        return moe.upload_q4(m.q, m.s, m.fmt)

    ex = inp.experts
    E = moe.Experts(ex.E, ex.H, ex.I, q4(ex.gate), q4(ex.up), q4(ex.down))
    return dev(inp.W_r.view(np.int16), torch.bfloat16), E


def time_loop(torch, fn, steps, warmup):
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        fn(warmup + i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


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


def run_ours(args, rank, world):
    import torch

    import mixture_experts_layer_09_gb300 as moe
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    moe.build()
    H, I, E, k, T = WORKLOAD["H"], WORKLOAD["I"], WORKLOAD["E"], WORKLOAD["k"], WORKLOAD["T"]
    seed0 = rank_seed(rank)

    # ---- resident weights: independent layer replicas
    layers = []
    for rep in range(N_REPLICAS):
        ex = gen.draw_experts(seed0 + rep, E, H, I)
        Wr = gen.draw_router(seed0 + rep, E, H)
        inp = gen.LayerInputs(gen.Workload("b", T, H, I, E, k), None, None, Wr, ex, None)
        W_r, Ed = upload_layer(torch, moe, inp)
        layers.append(moe.MoeLayer(W_r, Ed, None, k, max_T=T))
        del ex, inp

    def inputs(Tb):
        xs = [gen.draw_x(seed0 + 500 + i, Tb, H) for i in range(N_INPUTS)]
        rs = [gen.draw_residual(seed0 + 700 + i, Tb, H) for i in range(N_INPUTS)]
        to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
        return [to(x).cuda() for x in xs], [to(r).cuda() for r in rs], [to(x).pin_memory() for x in xs], \
            [to(r).pin_memory() for r in rs]

    def measure(Tb, steps, warmup, full=False):
        xd, rd, xh, rh = inputs(Tb)
        y = torch.empty((Tb, H), dtype=torch.float32, device="cuda")
        ids = torch.empty((Tb, k), dtype=torch.int32, device="cuda")

        def step(i):
            layers[i % N_REPLICAS].forward(xd[i % N_INPUTS], rd[i % N_INPUTS], y=y, topk_ids_out=ids)

        out = {}
        if dist is not None:
            dist.barrier()
        n0 = moe.moe_launch_count()
        dt = time_loop(torch, step, steps, warmup)
        out["launches_per_step"] = (moe.moe_launch_count() - n0) / (steps + warmup)
        out["plain_s"] = reduce_max(dist, dt, "cuda")
        # CUDA-graph replay of the same steps (one graph per (replica, input) pair)
        graphs = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step(0)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for i in range(N_INPUTS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(i)
            graphs.append(g)
        dtg = time_loop(torch, lambda i: graphs[i % N_INPUTS].replay(), steps, warmup)
        out["graph_s"] = reduce_max(dist, dtg, "cuda")
        # distinct experts per step (routing is the GPU's own output)
        nd = []
        for i in range(N_INPUTS):
            step(i)
            torch.cuda.synchronize()
            nd.append(len(np.unique(ids.cpu().numpy())))
        out["n_distinct"] = nd
        if full:
            # per-kernel device time over a timed pass, CUDA events on the launching stream
            moe.moe_profile_enable(True)
            time_loop(torch, step, steps, 0)
            out["kernels"] = moe.moe_profile_read()
            moe.moe_profile_enable(False)
            # end to end through host buffers: H2D of x and residual, D2H of y, every step
            yh = torch.empty((Tb, H), dtype=torch.float32).pin_memory()
            xin = torch.empty((Tb, H), dtype=torch.bfloat16, device="cuda")
            rin = torch.empty((Tb, H), dtype=torch.bfloat16, device="cuda")

            def e2e_step(i):
                xin.copy_(xh[i % N_INPUTS], non_blocking=True)
                rin.copy_(rh[i % N_INPUTS], non_blocking=True)
                layers[i % N_REPLICAS].forward(xin, rin, y=y)
                yh.copy_(y, non_blocking=True)

            dte = time_loop(torch, e2e_step, steps, warmup)
            out["e2e_s"] = reduce_max(dist, dte, "cuda")
            out["h2d"] = 2 * Tb * H * 2
            out["d2h"] = Tb * H * 4
        return out

    # SM clocks are sampled (nvidia-smi, 200 ms) over the whole measurement phase, which
    # contains the timed region: a region of a few ms alone would fall between two samples.
    # the samples go to $BENCH_CLOCKS_DIR (default: the temporary directory)
    clocks = Clocks(os.path.join(os.environ.get("BENCH_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"clocks_bench_r{rank}.csv"), local)
    clocks.start()
    main = measure(T, args.steps, args.warmup, full=True)
    sweep = {}
    for Tb in SWEEP_T:
        r = measure(Tb, max(10, args.steps // 2), args.warmup)
        best = min(r["plain_s"], r["graph_s"])
        us = 1e6 * best / max(10, args.steps // 2)
        sweep[f"T={Tb}"] = {"us_per_layer": us, "tokens_per_s": Tb / (us * 1e-6),
                            "plain_us": 1e6 * r["plain_s"] / max(10, args.steps // 2),
                            "graph_us": 1e6 * r["graph_s"] / max(10, args.steps // 2)}

    prefill = measure_prefill(torch, moe, args) if not args.no_prefill else None
    extra = {}
    if not args.no_extra:
        extra = {"decode_with_rmsnorm": measure_norm(torch, moe, args, layers, T, H),
                 "decode_glm": measure_glm(torch, moe, args),
                 "router_dispatch_sweep": measure_router_sweep(torch, moe, args),
                 "skewed_layer": measure_skewed_layer(torch, moe, args),
                 "mxfp4": measure_mxfp4(torch, moe, args)}
    main["clocks"] = clocks.stop()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    steps = args.steps
    best_s = min(main["plain_s"], main["graph_s"])
    ms_step = 1e3 * best_s / steps
    value = job_value(world, T, steps, best_s)
    hbm, tc, src = peaks()
    # roofline of the dominant kernel (by device time)
    kern = main["kernels"]
    dom = max(kern, key=lambda n: kern[n][0])
    dom_ms = kern[dom][0] / max(kern[dom][1], 1)
    nd = float(np.mean(main["n_distinct"]))
    bpe = BYTES_PER_EXPERT(H, I)
    per_kernel_bytes = {
        "gateup_gemv": nd * (2 * I * H // 2 + 2 * I * (H // 32) * 2) + T * H * 2 + T * (H // 32) * 8 + T * k * I * 4,
        "down_gemv_combine": nd * (H * I // 2 + H * (I // 32) * 2) + T * k * I * 2 + T * k * (I // 32) * 8
        + T * H * 2 + T * H * 4,
    }
    ach = per_kernel_bytes.get(dom, float("nan")) / (dom_ms * 1e-3) / 1e9
    traffic = dram_traffic(dom, nd)
    layer_bytes = nd * bpe + E * H * 2 + T * H * (2 + 2 + 4)
    layer_gbs = layer_bytes / (ms_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4xbf16->fp32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD['name']} H={H} I={I} E={E} k={k} T={T}", "global_batch": T * world,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"{N_REPLICAS} layer replicas x {E * bpe / 1e6:.0f} MB of experts cycled with "
                         f"{N_INPUTS} distinct batches (inputs larger than L2)",
                   "us_per_layer": ms_step * 1e3,
                   "plain_us_per_layer": 1e6 * main["plain_s"] / steps,
                   "graph_us_per_layer": 1e6 * main["graph_s"] / steps,
                   "mean_distinct_experts": nd,
                   "layer_hbm_gbs": layer_gbs, "layer_hbm_frac": layer_gbs / hbm,
                   "sweep": sweep},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                     "frac": ach / hbm, "peak_source": src,
                     "traffic": traffic["bytes"] if traffic else None,
                     "traffic_note": traffic["note"] if traffic else "no ncu capture of this kernel's current source",
                     "algorithmic_bytes": per_kernel_bytes.get(dom), "kernel_us": dom_ms * 1e3},
        "kernels_us_per_step": {n: 1e3 * v[0] / steps for n, v in kern.items()},
        "gpu_launches": int(round(main["launches_per_step"] * steps)),
        "prefill": prefill,
        **extra,
        "clocks": main.get("clocks"),
        "e2e": {"value": job_value(world, T, steps, main["e2e_s"]), "unit": "tokens/s",
                "h2d_bytes_per_step": main["h2d"], "d2h_bytes_per_step": main["d2h"]},
    }
    if not args.no_cpu_baseline:
        # the oracle as it stands, one host thread, on whole batches of the same workload (one
        # drawn layer, a fresh token batch each time) until about 10 s of CPU work is done
        import dataclasses

        import oracle
        oracle.build()
        base = gen.draw_layer(gen.Workload(WORKLOAD["name"], T, H, I, E, k))
        n_tok, dt, b = 0, 0.0, 0
        while b == 0 or dt < 10.0:
            inp = dataclasses.replace(base, x=gen.draw_x(500 + b, T, H)) if b else base
            t0 = time.perf_counter()
            oracle.layer_forward(inp)
            dt += time.perf_counter() - t0
            n_tok += T
            b += 1
        line["cpu_baseline"] = {"value": n_tok / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{b} batches of T={T} tokens ({n_tok} tokens, {dt:.1f} s)"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill-layer section")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the GLM-class decode, router/dispatch sweep and skewed-layer sections")
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
