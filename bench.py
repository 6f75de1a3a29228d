#!/usr/bin/env python
"""Throughput of the MoE expert-FFN hot path on GB300 (MegaMoE at
ep_world_size = 1: routing -> permute + MX quant -> grouped GEMM1 + swiglu +
MX requant -> grouped GEMM2 -> top-K combine), one mm_mega_moe call per step.

Workload (one GPU): DeepSeek-V3-shaped prefill, N=8192 tokens, hidden 7168,
intermediate 2048, 256 experts, top-8 with Zipf(s=1) routing, MXFP8 E5M2
dispatch, MXFP8 E4M3 weights with E8M0 scales (prepared once, like a load-time
weight format), bf16 gating weights.  Inputs are seeded and synthetic and are
resident in HBM before timing; the 11.6 GB of weights exceed L2, so no flush
is needed between steps.

Printed: one JSON line (rank 0).  Secondary measurements in the same line:
the routing/permute workload (N=16384, H=7168, E=256, K=8; HBM GB/s of the
permute kernel), the Qwen3-30B-A3B-shaped and the decode (N=128 + one shared
expert) workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (under torchrun) each rank runs its own replica of the workload
(token sharding, no collective on the data path); value = all ranks' tokens
divided by the slowest rank's time.  --impl reference times the CPU oracle
(the only reference implementation of this method) on a bounded sample of
the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE FFN tokens/s + MXFP8 TFLOP/s (% peak); permute HBM GB/s (% peak)"
NOMINAL_FP8_OVER_BF16 = 2.0   # 4.5 / 2.25 PFLOP/s dense
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3_prefill")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-peak", action="store_true",
                    help="skip measuring the dense MXFP8 rate (profiling runs); the tensor roof is then the nominal "
                         "FP8/bf16 ratio times the measured bf16 peak")
    ap.add_argument("--tokens", type=int, default=0, help="override N (profiling on a smaller case)")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiling on a smaller case)")
    ap.add_argument("--weights", choices=["fp8", "fp4", "a4w4"], default="fp8",
                    help="fp4: the A8W4-FP variant of the workload (MXFP4 weights, MXFP8 E4M3 activations); "
                         "a4w4: the A4W4-FP variant (MXFP4 tokens and weights, MXFP8 E4M3 activation for GEMM2)")
    return ap.parse_args()


def workload(args):
    import synth
    cfg = synth.CONFIGS[args.workload]
    if args.tokens:
        cfg = cfg.scaled(n=args.tokens)
    if args.experts:
        cfg = cfg.scaled(e=args.experts)
    if args.weights == "fp4":
        cfg = cfg.scaled(name=cfg.name + "_a8w4", weight_fmt=296, dispatch_fmt=24)
    if args.weights == "a4w4":
        cfg = cfg.scaled(name=cfg.name + "_a4w4", weight_fmt=296, dispatch_fmt=296)
    return cfg


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [s for s, p in zip(sm, power) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ----------------------------------------------------------------------------- helpers
def kernel_source_hash(name):
    return hashlib.sha256(open(os.path.join(ROOT, "routing_permute_mxfp8_gb300", "csrc", name), "rb").read()
                          ).hexdigest()[:16]


def profiled_traffic(profile_file, kernel_src):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (its sha256 prefix is recorded there)."""
    p = os.path.join(ROOT, "profiles", profile_file)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_src = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_hash(kernel_src):
        return None
    return float(m_tr.group(1))


class Dist:
    """One process per GPU (torchrun env).  The data path has no collective:
    the process group only provides the barrier around the timed region and
    the maximum of the ranks' times.  backend "nccl" on GPUs, "gloo" on CPU."""

    def __init__(self, backend="nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cpu"
        if self.world > 1:
            import torch
            import torch.distributed as tdist
            if backend == "nccl":
                torch.cuda.set_device(self.local)
                tdist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
                self.device = "cuda"
            else:
                tdist.init_process_group(backend)
            self.pg = tdist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------- inputs on the GPU
def gpu_inputs(cfg, mm, torch, seed_offset=0, weights=None, shared=None):
    """x, ids, gates from the seeded generator; fp32 N(0, 0.02) weights drawn on
    the GPU (seeded torch generator) and MX-quantised by the library (or the
    given routed / shared weights, reused)."""
    import synth
    dev = torch.device("cuda")
    x = torch.from_numpy(synth.tokens_bf16(cfg).view(np.int16)).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(synth.topk_ids(cfg)).to(dev)
    g = synth.topk_weights(cfg)
    gate = (torch.from_numpy(g.view(np.int16)).to(dev).view(torch.bfloat16) if g.dtype == np.uint16
            else torch.from_numpy(g).to(dev))
    if weights is None:
        weights = gpu_weights(cfg, mm, torch, cfg.e, seed=1000 + seed_offset)
    if cfg.shared and shared is None:
        shared = gpu_weights(cfg, mm, torch, cfg.shared, seed=2000 + seed_offset)
    return x, ids, gate, weights, shared if cfg.shared else None


def gpu_weights(cfg, mm, torch, n_exp, seed):
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    out = []
    for n_out, k_red in ((2 * cfg.inter, cfg.h), (cfg.h, cfg.inter)):
        kq = k_red // 2 if cfg.weight_fmt == mm.DT_FP4_E2M1 else k_red   # FP4: two codes per byte
        q = torch.empty((n_exp, n_out, kq), dtype=torch.uint8, device=dev)
        s = torch.empty((n_exp, n_out, k_red // 32), dtype=torch.uint8, device=dev)
        chunk = max(1, (1 << 28) // (n_out * k_red))
        for e0 in range(0, n_exp, chunk):
            e1 = min(n_exp, e0 + chunk)
            w = torch.randn(((e1 - e0) * n_out, k_red), generator=gen, device=dev, dtype=torch.float32) * 0.02
            qq, ss = mm.mm_mx_quantize(w, cfg.weight_fmt, scale_cols=k_red // 32)
            q[e0:e1] = qq.view(e1 - e0, n_out, kq)
            s[e0:e1] = ss.view(e1 - e0, n_out, k_red // 32)
            del w, qq, ss
        out += [q, s]
    w1, s1, w2, s2 = out
    p1 = mm.mm_prepare_weight_scales(s1, cfg.h, 1)
    p2 = mm.mm_prepare_weight_scales(s2, cfg.inter, 2)
    return {"w1": w1, "s1": s1, "w2": w2, "s2": s2, "p1": p1, "p2": p2}


def e2e_measure(args, mm, torch, cfg, x, ids, gate, W, S, ws, y, dist):
    """MegaMoE steps from pinned host inputs to a pinned host result.

    Every timed step copies its inputs (x, topk_ids, topk_weights) host ->
    device, runs mm_mega_moe and copies y device -> host.  Pipelined (the
    reported value): the input copies run on one copy stream and the result
    copies on another, with the device inputs and y double-buffered, so step
    i+1's inputs arrive and step i-1's result leaves while step i computes.
    Serial: all three on the compute stream, one after the other.
    """
    xh = x.cpu().pin_memory()
    idh = ids.cpu().pin_memory()
    gh = gate.cpu().pin_memory()
    yh = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    idd = [torch.empty_like(ids) for _ in range(2)]
    gd = [torch.empty_like(gate) for _ in range(2)]
    yd = [y, torch.empty_like(y)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    h2d_done, comp_done, d2h_done = ev(), ev(), ev()
    state = {"i": 0}

    def piped():
        i = state["i"]
        b = i % 2
        cur = torch.cuda.current_stream()
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[b])  # step i-2 has read buffer b
            xd[b].copy_(xh, non_blocking=True)
            idd[b].copy_(idh, non_blocking=True)
            gd[b].copy_(gh, non_blocking=True)
            h2d_done[b].record(s_in)
        cur.wait_event(h2d_done[b])
        if i >= 2:
            cur.wait_event(d2h_done[b])  # y buffer b has left for the host
        mega_call(mm, cfg, xd[b], idd[b], gd[b], W, S, ws, yd[b])
        comp_done[b].record(cur)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            yh[b].copy_(yd[b], non_blocking=True)
            d2h_done[b].record(s_out)
        state["i"] = i + 1

    def serial():
        xd[0].copy_(xh, non_blocking=True)
        idd[0].copy_(idh, non_blocking=True)
        gd[0].copy_(gh, non_blocking=True)
        mega_call(mm, cfg, xd[0], idd[0], gd[0], W, S, ws, yd[0])
        yh[0].copy_(yd[0], non_blocking=True)

    def drain():
        cur = torch.cuda.current_stream()
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    e_steps = max(1, min(args.steps, 50))
    # three timed runs, the median reported: the host-to-device copies share
    # the host's memory with whatever else runs on it, which moves single runs
    runs = [time_steps(torch, piped, e_steps, min(args.warmup, 3), dist, finish=drain) for _ in range(3)]
    runs.sort(key=lambda r: r[0])
    ems, est, _ = runs[1]
    ems = dist.max(ems)
    sms, _, _ = time_steps(torch, serial, e_steps, min(args.warmup, 3), dist)
    sms = dist.max(sms)
    h2d = x.numel() * 2 + ids.numel() * 4 + gate.numel() * gate.element_size()
    return {"value": whole_job_rate(cfg.n, e_steps, dist.world, ems), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(y.numel() * 2),
            "ms_per_step": ems / e_steps,
            "copies": "overlapped with the neighbouring steps' kernels (two copy streams, double-buffered)",
            "runs_ms_per_step": [r[0] / e_steps for r in runs], "reported": "median of three timed runs",
            "stage_ms_per_step": {k: v[0] / e_steps for k, v in est.items() if v[1]},
            "serial": {"value": whole_job_rate(cfg.n, e_steps, dist.world, sms), "ms_per_step": sms / e_steps}}


def mega_call(mm, cfg, x, ids, gate, W, S, ws, y):
    kw = {}
    if S is not None:
        kw = dict(shared_weight1=S["w1"], shared_weight2=S["w2"], shared_weight_scales1=S["p1"],
                  shared_weight_scales2=S["p2"], shared_weight_dtype=cfg.weight_fmt)
    return mm.mm_mega_moe(x, ids, gate, W["w1"], W["w2"], W["p1"], W["p2"], cfg.e, weight_dtype=cfg.weight_fmt,
                          weight_scale_layout=mm.WSCALE_PREPARED, dispatch_quant_out_dtype=cfg.dispatch_fmt,
                          workspace=ws, out=y, **kw)


def stage_rooflines(cfg, ms, hbm_peak, fp8_peak):
    """Each stage of the step against the roofline that bounds it, from its
    algorithmic work (inputs read once, outputs written once; FLOPs without
    the padding rows) and its device time per step."""
    rows = cfg.n * cfg.k + cfg.n * cfg.shared          # expanded rows, shared experts included
    gate_b = 2 if cfg.gate_dtype == "bf16" else 4
    out = {}

    def hbm(name, nbytes):
        if ms.get(name):
            gbs = nbytes / (ms[name] / 1e3) / 1e9
            out[name] = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "algorithmic_bytes": nbytes, "ms": ms[name]}

    # dispatch: x and the row indices read; FP8 (packed FP4) rows and E8M0 scales written
    xb = 0.5 if cfg.dispatch_fmt == 296 else 1.0
    hbm("dispatch", cfg.n * cfg.h * 2 + cfg.n * cfg.k * 4 + rows * cfg.h * xb + rows * (cfg.h // 32))
    # combine: O rows, gating weights and indices read; Y written
    hbm("combine", rows * cfg.h * 2 + cfg.n * cfg.k * (gate_b + 4) + cfg.n * cfg.h * 2)
    if ms.get("gemm2"):
        # the bound by arithmetic intensity against the ridge, as for GEMM1;
        # compulsory bytes: W2 and its scales of every expert, A_hat and its
        # scales read, bf16 O written
        sec = ms["gemm2"] / 1e3
        flops = 2.0 * rows * cfg.h * cfg.act_width
        wb = 0.5 if cfg.weight_fmt == 296 else 1.0
        nbytes = ((cfg.e + cfg.shared) * cfg.h * cfg.act_width * (wb + 1 / 32) +
                  rows * cfg.act_width * (1 + 1 / 32) + rows * cfg.h * 2)
        tf, gbs = flops / sec / 1e12, nbytes / sec / 1e9
        hbm_bound = flops / nbytes < fp8_peak * 1e12 / (hbm_peak * 1e9)
        out["gemm2"] = {"bound": "hbm" if hbm_bound else "tensor",
                        "achieved": gbs if hbm_bound else tf, "peak": hbm_peak if hbm_bound else fp8_peak,
                        "unit": "GB/s" if hbm_bound else "TFLOP/s",
                        "frac": gbs / hbm_peak if hbm_bound else tf / fp8_peak,
                        "frac_hbm": gbs / hbm_peak, "frac_tensor": tf / fp8_peak, "achieved_tflops": tf,
                        "achieved_gbs": gbs, "algorithmic_bytes": nbytes,
                        "arithmetic_intensity_flop_per_byte": flops / nbytes, "ms": ms["gemm2"]}
    if ms.get("route"):
        out["route"] = {"bound": "latency", "us": ms["route"] * 1e3}
    return out


def fp8_dense_peak(mm, torch, sustain_s=2.0):
    """Dense MXFP8 rate of this library's own block-scaled GEMM (k_gemm_mx
    GEMM1: E4M3 x E4M3 with E8M0 scales, fp32 accumulation in TMEM, swiglu +
    MX requantisation epilogue) on one square problem: one expert, one choice
    per token, M = N = K = 8192 (8192 tokens, hidden 8192, 2I = 8192).  The
    GEMM1 stage time of mm_mega_moe calls gives the rate: burst = the best of
    20 single calls, sustained = the mean over calls looped for sustain_s
    seconds (power-capped clocks).  Returns TFLOP/s figures and the shape."""
    import synth
    dev = torch.device("cuda")
    n = h = 8192
    inter = 4096
    cfg = synth.CONFIGS["tiny"].scaled(name="dense_8192", n=n, h=h, inter=inter, e=1, k=1, dispatch_fmt=24,
                                       weight_fmt=24, gate_dtype="fp32")
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    x = torch.randn((n, h), generator=gen, device=dev).to(torch.bfloat16)
    ids = torch.zeros((n, 1), dtype=torch.int32, device=dev)
    gate = torch.ones((n, 1), dtype=torch.float32, device=dev)
    W = gpu_weights(cfg, mm, torch, 1, seed=77)
    ws = torch.empty(mm.mm_mega_moe_workspace_size(n, h, 1, 1, inter, 0, mm.WSCALE_PREPARED), dtype=torch.uint8,
                     device=dev)
    y = torch.empty((n, h), dtype=torch.bfloat16, device=dev)
    call = lambda: mega_call(mm, cfg, x, ids, gate, W, None, ws, y)
    flops1 = 2.0 * n * (2 * inter) * h
    flops2 = 2.0 * n * h * inter
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    mm.timing_read()
    mm.timing_enable(True)
    best1 = best2 = 1e9
    for _ in range(20):
        call()
        st = mm.timing_read()
        best1 = min(best1, st["gemm1"][0])
        best2 = min(best2, st["gemm2"][0])
    t0 = time.perf_counter()
    calls = 0
    while time.perf_counter() - t0 < sustain_s:
        for _ in range(50):
            call()
        calls += 50
        torch.cuda.synchronize()
    st = mm.timing_read()
    mm.timing_enable(False)
    sus1 = st["gemm1"][0] / calls
    del x, W, ws, y
    return {"kernel": "k_gemm_mx<1> (MXFP8 E4M3 x E4M3, E8M0 block scales)", "m": n, "n": 2 * inter, "k": h,
            "burst_tflops": flops1 / (best1 / 1e3) / 1e12, "sustained_tflops": flops1 / (sus1 / 1e3) / 1e12,
            "gemm2_burst_tflops": flops2 / (best2 / 1e3) / 1e12, "sustained_calls": calls,
            "burst_ms": best1, "sustained_ms": sus1}


def library_mxfp8_peak(torch, sustain_s=2.0):
    """Dense MXFP8 rate of the vendor library on the same square shape:
    torch._scaled_mm (cuBLASLt) with float8_e4m3fn operands and one
    float8_e8m0fnu scale per 32 elements of every row of A and of B, bf16
    output, M = N = K = 8192.  A reference point for the tensor roofline only
    (nothing on the hot path calls it).  Returns None where this torch build
    has no block-scaled FP8 matmul."""
    e8 = getattr(torch, "float8_e8m0fnu", None)
    if e8 is None or not hasattr(torch, "_scaled_mm"):
        return None
    m = n = k = 8192
    dev = torch.device("cuda")
    try:
        a = torch.randn(m, k, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, k, device=dev).to(torch.float8_e4m3fn)
        sa = torch.full((m * (k // 32),), 127, dtype=torch.uint8, device=dev).view(e8)
        sb = torch.full((n * (k // 32),), 127, dtype=torch.uint8, device=dev).view(e8)
        fn = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
    except Exception as ex:  # this PyTorch has no block-scaled _scaled_mm
        return {"error": str(ex)[:200]}
    best = 1e9
    for _ in range(20):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    calls = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    while time.perf_counter() - t0 < sustain_s:
        for _ in range(50):
            fn()
        calls += 50
        torch.cuda.synchronize()
    e1.record()
    e1.synchronize()
    sus = e0.elapsed_time(e1) / calls
    fl = 2.0 * m * n * k
    del a, b, sa, sb
    return {"kernel": "torch._scaled_mm (cuBLASLt) MXFP8 E4M3, E8M0 scales per 32", "m": m, "n": n, "k": k,
            "burst_tflops": fl / (best / 1e3) / 1e12, "sustained_tflops": fl / (sus / 1e3) / 1e12,
            "sustained_calls": calls}


def gemm1_algorithmic_bytes(cfg, rows):
    """Compulsory bytes of one GEMM1 launch: the weights of the experts that
    receive rows (FP8 1 byte or FP4 half a byte per element, plus one E8M0
    byte per 32), X_hat (FP8, or packed FP4 under A4W4-FP) and its scales
    read, A_hat (FP8) and its scales written."""
    wb = 0.5 if cfg.weight_fmt == 296 else 1.0
    xb = 0.5 if cfg.dispatch_fmt == 296 else 1.0
    per_expert = 2 * cfg.inter * cfg.h * (wb + 1 / 32)
    experts = cfg.e + cfg.shared
    return experts * per_expert + rows * cfg.h * (xb + 1 / 32) + rows * cfg.act_width * (1 + 1 / 32)


def ffn_flops(cfg, tokens=None):
    n = cfg.n if tokens is None else tokens
    rows = n * cfg.k + n * cfg.shared
    return 2.0 * rows * (2 * cfg.inter) * cfg.h + 2.0 * rows * cfg.h * cfg.inter


def whole_job_rate(units_per_rank_step, steps, world, max_ms):
    """Units processed by all ranks per second of the slowest rank's time."""
    return units_per_rank_step * steps * world / (max_ms / 1e3)


def time_steps(torch, fn, steps, warmup, dist, sampler_gpu=None, finish=None):
    """Times `steps` calls of fn (CUDA events on the launching stream, barrier
    and synchronize on both sides).  Inside the timed region the library
    records one event pair per step, around GEMM1 (the dominant kernel, for
    its roofline); an event record between two kernels costs the stream a few
    microseconds, so the per-stage breakdown comes from a second pass of the
    same steps with every stage's pair.  Returns the timed ms, {stage:
    (device ms summed over the steps, kernel launches in the timed region)}
    and the clocks sampled during the timed region."""
    import routing_permute_mxfp8_gb300 as mm
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    mm.timing_read()
    mm.timing_select(["gemm1"])
    mm.timing_enable(True)
    st = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks = None
    if sampler_gpu is not None:
        sampler = ClockSampler(sampler_gpu)
        sampler.__enter__()
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(steps):
        fn()
    if finish is not None:
        finish()  # work of the timed steps on other streams, before the end event
    e1.record(st)
    e1.synchronize()
    if sampler_gpu is not None:
        sampler.__exit__(None, None, None)
        clocks = sampler.summary()
    mm.timing_enable(False)
    live = mm.timing_read()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    # breakdown pass: every stage's event pair
    mm.timing_select(None)
    mm.timing_enable(True)
    for _ in range(steps):
        fn()
    if finish is not None:
        finish()
    torch.cuda.synchronize()
    mm.timing_enable(False)
    full = mm.timing_read()
    stages = {k: (live[k][0] if k == "gemm1" else full[k][0], live[k][1]) for k in live}
    dist.barrier()
    return ms, stages, clocks


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_leg(cfg, rows_per_step, steps, warmup, max_experts=16):
    """Times the CPU oracle as it stands on a bounded sample of the workload.

    One step = the oracle's routing of the whole batch (keyValueSort, inverse,
    histogram of all N*K ids) plus, for `rows_per_step` sampled expanded rows
    (token i, choice k), the oracle's Q_MX of the token and its expert FFN
    (GEMM1 + swiglu + Q_MX + GEMM2), rows spread over the host cores (ctypes
    drops the GIL).  Rows are drawn among the experts touched first so that
    only `max_experts` experts' weights need building.  Returns token
    equivalents per second (rows / K per second) and details.
    """
    import concurrent.futures as cf
    import oracle
    import synth
    x = synth.tokens_bf16(cfg)
    ids = synth.topk_ids(cfg)
    chosen = []
    for e in ids.reshape(-1):
        if e not in chosen:
            chosen.append(int(e))
        if len(chosen) == max_experts:
            break
    cand = np.nonzero(np.isin(ids.reshape(-1), chosen))[0]
    rng = np.random.default_rng(123)
    total_rows = rows_per_step * (steps + warmup)
    pick = rng.choice(cand, size=total_rows, replace=cand.size < total_rows)
    s1c, s2c = 2 * ((cfg.h + 63) // 64), 2 * ((cfg.inter + 63) // 64)
    W = {}
    for e in chosen:
        w1, s1 = oracle.mx_quantize(synth.weight_f32(cfg, 1, e), oracle.DT_F32, cfg.weight_fmt, s1c)
        w2, s2 = oracle.mx_quantize(synth.weight_f32(cfg, 2, e), oracle.DT_F32, cfg.weight_fmt, s2c)
        W[e] = (w1, s1, w2, s2)
    flat = ids.reshape(-1)

    def one_row(j):
        i = j // cfg.k
        xq, xs = oracle.mx_quantize(x[i:i + 1], oracle.DT_BF16, cfg.dispatch_fmt)
        w1, s1, w2, s2 = W[int(flat[j])]
        return oracle.expert_row(xq[0], xs[0], cfg.dispatch_fmt, w1, s1, w2, s2, cfg.weight_fmt, cfg.dispatch_fmt)

    threads = min(rows_per_step, os.cpu_count() or 1)
    times = []
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for st in range(steps + warmup):
            rows = pick[st * rows_per_step:(st + 1) * rows_per_step]
            t0 = time.perf_counter()
            oracle.route(ids, cfg.e)
            list(ex.map(one_row, rows))
            dt = time.perf_counter() - t0
            if st >= warmup:
                times.append(dt)
    total = sum(times)
    tok_per_s = rows_per_step * len(times) / cfg.k / total
    return tok_per_s, {
        "cores": threads, "seconds": total,
        "sample": (f"{len(times)} step(s) x [routing of all {cfg.n * cfg.k} ids of {cfg.name} + Q_MX and expert "
                   f"FFN of {rows_per_step} sampled expanded rows]; value = rows / top-K per second; double "
                   f"precision on {threads} host threads")}


# ----------------------------------------------------------------------------- main arms
def run_reference(args):
    import synth
    dist_rank = int(os.environ.get("RANK", "0"))
    if dist_rank != 0:
        return 0
    cfg = workload(args)
    k_eff = max(1, args.steps)
    w_eff = max(0, args.warmup)
    # about one row per host core per step keeps the whole run within a few minutes
    per_step = max(1, min(os.cpu_count() or 1, 16))
    val, info = oracle_leg(cfg, per_step, k_eff, w_eff)
    ms_step = info["seconds"] / k_eff * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": k_eff, "warmup": w_eff, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "tokens": cfg.n, "hidden": cfg.h, "intermediate": cfg.inter,
                   "experts": cfg.e, "topk": cfg.k, "routing": cfg.routing},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": info["cores"], "kind": "oracle",
                         "sample": info["sample"]},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import synth
    import routing_permute_mxfp8_gb300 as mm

    dist = Dist("nccl")
    torch.cuda.set_device(dist.local)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    gpu_index = vis.split(",")[dist.local].strip() if vis else str(dist.local)
    mm.load()
    peaks, peak_src = load_peaks()
    hbm_peak = peaks["hbm_gbs"]
    # the dense MXFP8 rate, measured on this GPU with the library's own
    # block-scaled GEMM (no FP8 figure in the peaks file); the nominal
    # FP8/bf16 ratio times the bf16 peaks is reported beside it
    if args.no_peak:
        dense = {"burst_tflops": peaks["bf16_tflops"] * NOMINAL_FP8_OVER_BF16,
                 "sustained_tflops": peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * NOMINAL_FP8_OVER_BF16,
                 "kernel": "not measured (--no-peak): nominal FP8/bf16 ratio x measured bf16"}
        lib_dense = None
    else:
        dense = fp8_dense_peak(mm, torch)
        lib_dense = library_mxfp8_peak(torch)
    # the higher of the two measured rates is the roof
    fp8_peak_burst = max(dense["burst_tflops"], (lib_dense or {}).get("burst_tflops", 0.0))
    fp8_peak_sus = max(dense["sustained_tflops"], (lib_dense or {}).get("sustained_tflops", 0.0))
    fp8_nominal = {"burst": peaks["bf16_tflops"] * NOMINAL_FP8_OVER_BF16,
                   "sustained": peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * NOMINAL_FP8_OVER_BF16}

    cfg = workload(args)
    x, ids, gate, W, S = gpu_inputs(cfg, mm, torch, seed_offset=dist.rank)
    need = mm.mm_mega_moe_workspace_size(cfg.n, cfg.h, cfg.k, cfg.e, cfg.inter, cfg.shared, mm.WSCALE_PREPARED)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = torch.empty((cfg.n, cfg.h), dtype=torch.bfloat16, device="cuda")
    fn = lambda: mega_call(mm, cfg, x, ids, gate, W, S, ws, y)
    ms, stages, clocks = time_steps(torch, fn, args.steps, args.warmup, dist, sampler_gpu=gpu_index)
    ms = dist.max(ms)
    ms_step = ms / args.steps
    value = whole_job_rate(cfg.n, args.steps, dist.world, ms)
    flops = ffn_flops(cfg)
    launches = sum(c for _, c in stages.values())
    g1_ms = stages["gemm1"][0] / max(1, stages["gemm1"][1])
    g2_ms = stages["gemm2"][0] / max(1, stages["gemm2"][1])
    rows = cfg.n * cfg.k + cfg.n * cfg.shared
    g1_flops = 2.0 * rows * 2 * cfg.inter * cfg.h
    g1_tflops = g1_flops / (g1_ms / 1e3) / 1e12
    g1_bytes = gemm1_algorithmic_bytes(cfg, rows)
    g1_gbs = g1_bytes / (g1_ms / 1e3) / 1e9
    traffic = profiled_traffic(f"gemm1_{cfg.name}.md", "gemm.cu")
    # the timed region decides which tensor peak applies: a burst figure for
    # a region under a second, the power-capped sustained one otherwise
    burst = ms < 1000.0
    fp8_peak = fp8_peak_burst if burst else fp8_peak_sus
    ridge = fp8_peak * 1e12 / (hbm_peak * 1e9)          # FLOP per byte where the two roofs meet
    intensity = g1_flops / g1_bytes
    bound = "tensor" if intensity > ridge else "hbm"
    # the tensor cores work on 128-row tiles: rows the MMAs compute, padding
    # of every expert's (and shared expert's) rows to a multiple of 128 included
    counts = np.bincount(ids.reshape(-1).cpu().numpy(), minlength=cfg.e)
    padded_rows = 128 * (int(np.sum((counts + 127) // 128)) + cfg.shared * ((cfg.n + 127) // 128))
    g1_exec_tflops = 2.0 * padded_rows * 2 * cfg.inter * cfg.h / (g1_ms / 1e3) / 1e12
    roofline = {"bound": bound, "kernel": "k_gemm_mx<1> (GEMM1 + swiglu + MX requant)",
                "achieved": g1_tflops if bound == "tensor" else g1_gbs,
                "peak": fp8_peak if bound == "tensor" else hbm_peak,
                "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                "frac": g1_tflops / fp8_peak if bound == "tensor" else g1_gbs / hbm_peak,
                "traffic": traffic,
                "frac_hbm": g1_gbs / hbm_peak, "frac_tensor": g1_tflops / fp8_peak,
                "achieved_tflops": g1_tflops, "achieved_gbs": g1_gbs,
                "arithmetic_intensity_flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                "algorithmic_flops_per_launch": g1_flops, "algorithmic_bytes_per_launch": g1_bytes,
                "avg_launch_ms": g1_ms,
                "mma_rows": padded_rows, "padding_frac": 1.0 - rows / padded_rows,
                "frac_tensor_mma_rows": g1_exec_tflops / fp8_peak,
                "peak_source": (f"hbm: {peak_src} copy bandwidth; tensor: {'burst' if burst else 'sustained'} dense "
                                f"MXFP8 rate measured in this run at 8192^3, the higher of cuBLASLt's block-scaled "
                                f"GEMM and k_gemm_mx; the timed region being {ms / 1e3:.2f} s"),
                "frac_tensor_of_nominal_ratio": g1_tflops / fp8_nominal["burst" if burst else "sustained"]}
    stage_ms = {k: (v[0] / max(1, v[1]) if v[1] else 0.0) for k, v in stages.items() if v[1]}
    per_step_stage_ms = {k: v[0] / args.steps for k, v in stages.items() if v[1]}
    stage_roofline = stage_rooflines(cfg, per_step_stage_ms, hbm_peak, fp8_peak_burst if ms < 1000.0 else fp8_peak_sus)

    # end to end through the public call with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = e2e_measure(args, mm, torch, cfg, x, ids, gate, W, S, ws, y, dist)

    secondary = {}
    if not args.no_secondary:
        secondary = secondary_measurements(args, mm, torch, synth, dist, hbm_peak, fp8_peak_burst, W, cfg)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"fp8": "mxfp8", "fp4": "mxfp8 x mxfp4", "a4w4": "mxfp4 (GEMM1), mxfp8 x mxfp4 (GEMM2)"}[args.weights],
        "data": "synthetic (seeded generator; random-init weights)",
        "config": {"workload": cfg.name, "tokens": cfg.n, "hidden": cfg.h, "intermediate": cfg.inter,
                   "experts": cfg.e, "topk": cfg.k, "routing": f"{cfg.routing}" + (" s=1.0" if cfg.routing == "zipf" else ""),
                   "dispatch": {23: "mxfp8_e5m2", 24: "mxfp8_e4m3", 296: "mxfp4_e2m1"}[cfg.dispatch_fmt],
                   "weights": {24: "mxfp8_e4m3", 23: "mxfp8_e5m2", 296: "mxfp4_e2m1"}[cfg.weight_fmt],
                   "gate": cfg.gate_dtype, "shared_experts": cfg.shared,
                   "weight_scale_layout": "prepared once (mm_prepare_weight_scales)",
                   "l2": "inputs larger than L2 (weights streamed from HBM every step)",
                   "parallelism": f"replica per GPU x{dist.world} (token sharding, no collective)"},
        "tflops": flops / (ms_step / 1e3) / 1e12,
        "tflops_frac_of_fp8_peak": flops / (ms_step / 1e3) / 1e12 / fp8_peak,
        "ffn_gemms_tflops": (g1_flops + 2.0 * rows * cfg.h * cfg.act_width) / ((g1_ms + g2_ms) / 1e3) / 1e12,
        "ffn_gemms_frac_of_fp8_peak": (g1_flops + 2.0 * rows * cfg.h * cfg.act_width) / ((g1_ms + g2_ms) / 1e3)
        / 1e12 / fp8_peak,
        "roofline": roofline,
        "stage_roofline": stage_roofline,
        "stage_ms_per_launch": stage_ms,
        "stage_ms_per_step": per_step_stage_ms,
        "stage_timing": ("GEMM1: CUDA events around each launch inside the timed region; the other stages: "
                         "their event pairs in a second pass of the same steps (an event record between two "
                         "kernels costs the stream a few microseconds, so the timed region carries one pair)"),
        "gemm2_tflops": 2.0 * (cfg.n * cfg.k + cfg.n * cfg.shared) * cfg.h * cfg.inter / (g2_ms / 1e3) / 1e12,
        "gpu_launches": launches,
        "gpu_launches_per_step": launches / args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "peaks": {"hbm_gbs": hbm_peak, "hbm_source": peak_src, "fp8_dense_measured": dense,
                  "fp8_dense_library": lib_dense,
                  "fp8_nominal_ratio_tflops": fp8_nominal,
                  "fp8_peak_used": fp8_peak, "fp8_peak_used_kind": "burst" if burst else "sustained"},
    }
    line.update(secondary)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        # about 10 s of host time: two steps of 12 sampled rows per host thread
        val, info = oracle_leg(cfg, 12 * max(1, min(os.cpu_count() or 1, 16)), 2, 0)
        line["cpu_baseline"] = {"value": val, "unit": "tokens/s", "cores": info["cores"], "kind": "oracle",
                                "sample": info["sample"]}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def secondary_measurements(args, mm, torch, synth, dist, hbm_peak, fp8_peak, W_prefill, cfg_prefill):
    out = {}
    steps = max(10, min(args.steps, 50))
    # routing / permute workload: HBM bandwidth of the permute kernel
    rc = synth.CONFIGS["routing"]
    xr = torch.from_numpy(synth.tokens_bf16(rc).view(np.int16)).cuda().view(torch.bfloat16)
    idr = torch.from_numpy(synth.topk_ids(rc)).cuda()
    rows = rc.n * rc.k
    perm = {}
    for name, q in (("mxfp8_e4m3", mm.QUANT_MXFP8_E4M3FN), ("bf16", mm.QUANT_NONE)):
        need = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
        fn = lambda: mm.mm_moe_init_routing(xr, idr, rc.e, q, 1, workspace=need)
        ms, st, _ = time_steps(torch, fn, steps, 3, dist)
        d_ms = st["dispatch"][0] / max(1, st["dispatch"][1])
        r_ms = st["route"][0] / max(1, st["route"][1])
        out_b = rows * rc.h * (1 if q != mm.QUANT_NONE else 2) + (rows * (rc.h // 32) if q != mm.QUANT_NONE else 0)
        dispatch_bytes = rc.n * rc.h * 2 + rows * 4 + out_b           # read x + dest idx, write rows (+scales)
        call_bytes = dispatch_bytes + rows * 4 * 3 + rc.e * 8          # + ids read, idx writes, counts
        perm[name] = {"dispatch_us": d_ms * 1e3, "dispatch_gbs": dispatch_bytes / (d_ms / 1e3) / 1e9,
                      "dispatch_frac": dispatch_bytes / (d_ms / 1e3) / 1e9 / hbm_peak,
                      "route_us": r_ms * 1e3, "call_us": ms / steps * 1e3,
                      "call_gbs": call_bytes / (ms / steps / 1e3) / 1e9,
                      "dispatch_bytes": dispatch_bytes}
    out["permute"] = {"workload": "routing N=16384 H=7168 E=256 K=8 uniform", "unit": "GB/s",
                      "peak_gbs": hbm_peak, **perm}
    del xr
    # Qwen3-30B-A3B-shaped FFN
    qc = synth.CONFIGS["qwen3"]
    x, ids, gate, W, S = gpu_inputs(qc, mm, torch, seed_offset=10 + dist.rank)
    ws = torch.empty(mm.mm_mega_moe_workspace_size(qc.n, qc.h, qc.k, qc.e, qc.inter, 0, 1), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty((qc.n, qc.h), dtype=torch.bfloat16, device="cuda")
    ms, st, _ = time_steps(torch, lambda: mega_call(mm, qc, x, ids, gate, W, S, ws, y), steps, 3, dist)
    t = ms / steps / 1e3
    out["qwen3"] = {"tokens_per_s": qc.n / t, "ms_per_step": t * 1e3, "tflops": ffn_flops(qc) / t / 1e12,
                    "tflops_frac": ffn_flops(qc) / t / 1e12 / fp8_peak,
                    "stage_ms_per_step": {k: v[0] / steps for k, v in st.items() if v[1]}}
    del x, W, ws
    # decode: same expert weights as the prefill workload, plus one shared expert
    # (same weight type as the prefill weights it reuses)
    dc = synth.CONFIGS["dsv3_decode"].scaled(weight_fmt=cfg_prefill.weight_fmt)
    x, ids, gate, _, S = gpu_inputs(dc, mm, torch, seed_offset=20 + dist.rank, weights=W_prefill)
    ws = torch.empty(mm.mm_mega_moe_workspace_size(dc.n, dc.h, dc.k, dc.e, dc.inter, dc.shared, 1),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty((dc.n, dc.h), dtype=torch.bfloat16, device="cuda")
    ms, st, _ = time_steps(torch, lambda: mega_call(mm, dc, x, ids, gate, W_prefill, S, ws, y), steps, 3, dist)
    t = ms / steps / 1e3
    touched = int(torch.unique(ids).numel())
    per_exp = 3 * dc.h * dc.inter * ((0.5 if dc.weight_fmt == mm.DT_FP4_E2M1 else 1.0) + 1 / 32)
    wbytes = (touched + dc.shared) * per_exp
    out["decode"] = {"tokens_per_s": dc.n / t, "ms_per_step": t * 1e3, "experts_touched": touched,
                     "weight_bytes": wbytes, "weight_gbs": wbytes / t / 1e9, "hbm_frac": wbytes / t / 1e9 / hbm_peak,
                     "stage_ms_per_step": {k: v[0] / steps for k, v in st.items() if v[1]}}
    del x, ws, S
    out["ep8"] = ep_local_measurements(mm, torch, synth, dist, hbm_peak, W_prefill, cfg_prefill, steps)
    if cfg_prefill.weight_fmt == mm.DT_FP4_E2M1:
        return out
    # A8W4-FP: the same prefill and decode shapes with MXFP4 E2M1 weights (packed,
    # half the weight bytes) and MXFP8 E4M3 activations; A4W4-FP: the same FP4
    # weights with the tokens dispatched as MXFP4 too (GEMM2 stays A8W4)
    pc4 = cfg_prefill.scaled(weight_fmt=mm.DT_FP4_E2M1, dispatch_fmt=mm.DT_FP8_E4M3FN)
    W4 = None
    S4 = None
    for key, dfmt in (("a8w4", mm.DT_FP8_E4M3FN), ("a4w4", mm.DT_FP4_E2M1)):
        res = {}
        pc = pc4.scaled(dispatch_fmt=dfmt)
        x, ids, gate, W4g, _ = gpu_inputs(pc, mm, torch, seed_offset=30 + dist.rank, weights=W4)
        W4 = W4g if W4 is None else W4
        ws = torch.empty(mm.mm_mega_moe_workspace_size(pc.n, pc.h, pc.k, pc.e, pc.inter, pc.shared, 1),
                         dtype=torch.uint8, device="cuda")
        y = torch.empty((pc.n, pc.h), dtype=torch.bfloat16, device="cuda")
        ms, st, _ = time_steps(torch, lambda: mega_call(mm, pc, x, ids, gate, W4, None, ws, y), steps, 3, dist)
        t = ms / steps / 1e3
        res["prefill"] = {"workload": f"{pc.name} N={pc.n} H={pc.h} I={pc.inter} E={pc.e} K={pc.k}",
                          "tokens_per_s": pc.n / t, "ms_per_step": t * 1e3, "tflops": ffn_flops(pc) / t / 1e12,
                          "tflops_frac": ffn_flops(pc) / t / 1e12 / fp8_peak,
                          "stage_ms_per_step": {k: v[0] / steps for k, v in st.items() if v[1]}}
        del x, ws
        dcf = dc.scaled(weight_fmt=mm.DT_FP4_E2M1, dispatch_fmt=dfmt)
        x, ids, gate, _, S4g = gpu_inputs(dcf, mm, torch, seed_offset=40 + dist.rank, weights=W4, shared=S4)
        S4 = S4g if S4 is None else S4
        ws = torch.empty(mm.mm_mega_moe_workspace_size(dcf.n, dcf.h, dcf.k, dcf.e, dcf.inter, dcf.shared, 1),
                         dtype=torch.uint8, device="cuda")
        y = torch.empty((dcf.n, dcf.h), dtype=torch.bfloat16, device="cuda")
        ms, st, _ = time_steps(torch, lambda: mega_call(mm, dcf, x, ids, gate, W4, S4, ws, y), steps, 3, dist)
        t = ms / steps / 1e3
        touched = int(torch.unique(ids).numel())
        wbytes = (touched + dcf.shared) * 3 * dcf.h * dcf.inter * (0.5 + 1 / 32)
        res["decode"] = {"tokens_per_s": dcf.n / t, "ms_per_step": t * 1e3, "experts_touched": touched,
                         "weight_bytes": wbytes, "weight_gbs": wbytes / t / 1e9,
                         "hbm_frac": wbytes / t / 1e9 / hbm_peak,
                         "stage_ms_per_step": {k: v[0] / steps for k, v in st.items() if v[1]}}
        out[key] = res
        del x, ws
    del W4, S4
    return out


def ep_local_measurements(mm, torch, synth, dist, hbm_peak, W, cfg, steps, world=8):
    """Expert parallelism over `world` ranks (MegaMoE stages 1-4 with
    epWorldSize > 1), the kernels one rank runs, on this GPU: the source
    side's dispatch (rows sorted by destination rank, each token MX-quantised
    once), the expert side of the busiest rank (its E/W experts on the rows
    it receives when every source rank routes like this batch: the rows this
    batch sends it, `world` times), and the source side's combine of the
    returned rows.  The all-to-all exchanges are not measured: one GPU."""
    e_loc = cfg.e // world
    x, ids, gate, _, _ = gpu_inputs(cfg, mm, torch, seed_offset=50 + dist.rank, weights=W)
    sx, ss, se, counts, exp_idx = mm.mm_moe_ep_dispatch(x, ids, cfg.e, world, cfg.dispatch_fmt)
    ms_d, st_d, _ = time_steps(torch, lambda: mm.mm_moe_ep_dispatch(x, ids, cfg.e, world, cfg.dispatch_fmt),
                               steps, 3, dist)
    cnt = counts.cpu().tolist()
    r = int(np.argmax(cnt))
    off = int(sum(cnt[:r]))
    m = world * cnt[r]
    rx = sx[off:off + cnt[r]].repeat(world, 1)
    rs = ss[off:off + cnt[r]].repeat(world, 1)
    re = se[off:off + cnt[r]].repeat(world).contiguous()
    pe1, pe2 = W["p1"].numel() // cfg.e, W["p2"].numel() // cfg.e
    w1, w2 = W["w1"][r * e_loc:(r + 1) * e_loc], W["w2"][r * e_loc:(r + 1) * e_loc]
    p1 = W["p1"][r * e_loc * pe1:(r + 1) * e_loc * pe1]
    p2 = W["p2"][r * e_loc * pe2:(r + 1) * e_loc * pe2]
    ws = torch.empty(mm.mm_mega_moe_workspace_size(m, cfg.h, 1, e_loc, cfg.inter, 0, mm.WSCALE_PREPARED),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty((m, cfg.h), dtype=torch.bfloat16, device="cuda")
    expert = lambda: mm.mm_moe_expert_ffn(rx, rs, re, w1, w2, p1, p2, e_loc, x_dtype=cfg.dispatch_fmt,
                                          weight_dtype=cfg.weight_fmt, weight_scale_layout=mm.WSCALE_PREPARED,
                                          workspace=ws, out=o)
    ms_e, st_e, _ = time_steps(torch, expert, steps, 3, dist)
    del rx, rs, re, ws, o
    back = torch.randn((cfg.n * cfg.k, cfg.h), device="cuda").to(torch.bfloat16)
    y = torch.empty((cfg.n, cfg.h), dtype=torch.bfloat16, device="cuda")
    ms_c, st_c, _ = time_steps(torch, lambda: mm.mm_moe_combine(back, exp_idx, gate, out=y), steps, 3, dist)
    # combine quantisation (combineQuantMode 4): the expert rank's Q_MX of the rows
    # it sends back, and the source rank's combine of MXFP8 rows
    bq, bs = mm.mm_mx_quantize(back, mm.DT_FP8_E4M3FN, scale_cols=cfg.h // 32)
    ms_q, _, _ = time_steps(torch, lambda: mm.mm_mx_quantize(back, mm.DT_FP8_E4M3FN, scale_cols=cfg.h // 32),
                            steps, 3, dist)   # one launch a step, timed with the step's events
    _, st_cq, _ = time_steps(torch, lambda: mm.mm_moe_combine(bq, exp_idx, gate, out=y, expert_scales=bs,
                                                              expert_rows_dtype=mm.DT_FP8_E4M3FN), steps, 3, dist)
    rows = cfg.n * cfg.k
    d_ms = (st_d["route"][0] + st_d["dispatch"][0]) / steps
    c_ms = st_c["combine"][0] / steps
    q_ms = ms_q / steps
    cq_ms = st_cq["combine"][0] / steps
    q_bytes = rows * cfg.h * 2 + rows * (cfg.h + cfg.h // 32)
    cq_bytes = rows * (cfg.h + cfg.h // 32) + rows * (4 + gate.element_size()) + cfg.n * cfg.h * 2
    d_bytes = cfg.n * cfg.h * 2 + rows * (4 + 4 + 4 + cfg.h + cfg.h // 32)
    c_bytes = rows * cfg.h * 2 + rows * (4 + gate.element_size()) + cfg.n * cfg.h * 2
    del x, ids, gate, sx, ss, se, back, y, bq, bs
    return {"workload": f"{cfg.name}, ep_world_size {world}, {e_loc} experts per rank",
            "exchange": "not measured (one GPU)",
            "dispatch_ms": d_ms, "dispatch_gbs": d_bytes / (d_ms / 1e3) / 1e9,
            "dispatch_frac": d_bytes / (d_ms / 1e3) / 1e9 / hbm_peak,
            "expert_rank": r, "expert_rows": m, "expert_ms": ms_e / steps,
            "expert_stage_ms": {k: v[0] / steps for k, v in st_e.items() if v[1]},
            "combine_ms": c_ms, "combine_gbs": c_bytes / (c_ms / 1e3) / 1e9,
            "combine_frac": c_bytes / (c_ms / 1e3) / 1e9 / hbm_peak,
            "combine_quant_e4m3": {"quantise_ms": q_ms, "quantise_gbs": q_bytes / (q_ms / 1e3) / 1e9,
                                   "combine_ms": cq_ms, "combine_gbs": cq_bytes / (cq_ms / 1e3) / 1e9,
                                   "combine_frac": cq_bytes / (cq_ms / 1e3) / 1e9 / hbm_peak,
                                   "exchange_bytes_per_row": cfg.h + cfg.h // 32, "bf16_bytes_per_row": 2 * cfg.h},
            "rank_rows_sent": cnt}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
