"""Benchmark of the MXFP8 activation chain on GB300.

One step = one pass of the whole hot path over one batch of T tokens, inputs resident in HBM:
  rmsnorm_dual_out  x [T, 5120] -> y bf16 + y MXFP8 (int32-packed scales)
  mxfp8_quantize    attention output o [T, 8*4096] bf16 -> MXFP8 (F8_128x4 scales)
  o_proj_mxfp8      the _o_proj pair, one call: wo_a einsum o -> z MXFP8 (fused epilogue,
                    F8_128x4 scales), then wo_b z -> out bf16 [T, 5120] (a programmatic
                    dependent launch)
(DeepSeek-V4.1-Flash TP1 shapes from the vLLM page "[Perf][DSv4.1] MegaAttn: wo_a writes
wo_b's MXFP8 input", Validation). L2 is flushed before every step (cold L2, as on that page);
each call is timed with CUDA events on the launching stream and the flush is outside the
events. `value` is tokens/s through the whole chain, summed over ranks (weak scaling: every
rank runs its own replica). Per-call us, GB/s, TFLOP/s and roofline fractions are reported
alongside, and a compact `sweep` object times every configuration of the metric the way the
page does (each call replayed from a CUDA graph, L2 flushed before it): the _o_proj pair fused
and unfused over T = 1..32768, the quantizer and RMSNorm at two sizes each. `--impl reference`
times the CPU oracle on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--tokens T] [--impl reference] [--sweep]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "_o_proj us/call & TFLOP/s at T=1..32768; MXFP8 quant/RMSNorm HBM GB/s"
G, NA, KA, NB, H = 8, 1024, 4096, 5120, 5120
KB = G * NA
FLOP_PER_TOKEN = 2 * G * NA * KA + 2 * NB * KB
WEIGHT_BYTES = G * NA * KA + NB * KB + (G * NA * KA + NB * KB) // 32
NOMINAL_HBM_GBS = 8000.0         # GB300 HBM3e, nominal
NOMINAL_MXFP8_TFLOPS = 4500.0    # GB300 dense fp8 tensor rate, nominal


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---- algorithmic bytes / flops per launch ---------------------------------------------------
def quant_bytes(T, K, layouts=1):
    return T * K * 2 + T * K + layouts * T * K // 32


def rms_bytes(T, H_=H):
    return T * H_ * 2 + T * H_ * 2 + T * H_ + T * H_ // 32 + H_ * 2


def wo_a_bytes(T):
    return G * NA * KA * 33 // 32 + T * G * KA * 33 // 32 + T * KB * 33 // 32


def wo_b_bytes(T):
    return NB * KB * 33 // 32 + T * KB * 33 // 32 + T * NB * 2


def chain_config(T, world):
    """The workload both arms report (the GPU arm's timing conditions included)."""
    return {"workload": f"MXFP8 activation chain, DeepSeek-V4.1-Flash TP1 _o_proj + RMSNorm, T={T}",
            "tokens": T, "wo_a": "8 groups x 4096 -> 1024", "wo_b": "8192 -> 5120", "rmsnorm_hidden": H,
            "l2": "flushed before every step (outside the timed events)", "parallelism": f"replicas x{world}"}


def wo_a_flops(T):
    return 2 * T * G * NA * KA


def wo_b_flops(T):
    return 2 * T * NB * KB


# ---- clocks -----------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- ranks (replicas only: one process per GPU, no collective on the data path) ---------------
def rank_env():
    """(world size, rank, local rank) from the torchrun environment; (1, 0, 0) without it."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, world, device):
    """The largest `value` over all ranks (all-reduce MAX); `value` itself with one rank."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, tokens_per_rank, steps, max_ms):
    """Tokens per second of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


# ---- the GPU arm -------------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import mxfp8_activation_quant_gb300 as mxq
    from mxfp8_activation_quant_gb300 import synth

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    mxq.load()
    T = args.tokens
    seed = 1000 * rank

    # resident inputs and weights (weights quantized once, outside any timing)
    def mx(x):
        q, s = mxq.quantize(x, layouts=(mxq.SF_TILED_128X4,))
        return mxq.MXFP8(q, s[mxq.SF_TILED_128X4])

    WA = mx(synth.wo_a_weight(seed, device=dev))
    WB = mx(synth.wo_b_weight(seed, device=dev))
    x = synth.rmsnorm_input(seed, T, device=dev)
    gamma = synth.rmsnorm_gamma(seed, device=dev)
    o = synth.o_proj_activation(seed, T, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    yq = torch.empty((T, H), dtype=torch.uint8, device=dev)
    ysf = mxq.empty_sf(mxq.SF_PACKED_I32_MN, T, H, dev)
    oq = torch.empty((T, G * KA), dtype=torch.uint8, device=dev)
    osf = mxq.empty_sf(mxq.SF_TILED_128X4, T, G * KA, dev)
    O = mxq.MXFP8(oq, osf)
    zq = torch.empty((T, KB), dtype=torch.uint8, device=dev)
    zsf = mxq.empty_sf(mxq.SF_TILED_128X4, T, KB, dev)
    Z = mxq.MXFP8(zq, zsf)
    out = torch.empty((T, NB), dtype=torch.bfloat16, device=dev)
    status = mxq.new_status(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(4 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        mxq.rmsnorm_dual_out(x, gamma, synth.RMS_EPS, y, yq, sf_packed=ysf)
        if ev is not None:
            ev[1].record(stream)
        mxq.mxfp8_quantize(o, oq, None, None, osf)
        if ev is not None:
            ev[2].record(stream)
        mxq.o_proj_mxfp8(O, WA, WB, T, G, NA, KA, NB, zq, zsf, out, status=status)
        if ev is not None:
            ev[3].record(stream)

    KERNELS_PER_STEP = 4  # rmsnorm_dual_kernel, quantize_kernel, wo_a and wo_b GEMM kernels
    NPARTS = 3
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(NPARTS + 1)] for _ in range(args.steps)]
    # clocks are sampled from the warm-up through the timed region and the compact sweep (the
    # timed steps alone last a few milliseconds, shorter than the sampling period)
    sampler = ClockSampler(dev.index).__enter__()
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_((i + 7) & 0xFF)  # cold L2 before every step, outside the events
        step(evs[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    mxq.check_status(status)

    parts = [[evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)] for j in range(NPARTS)]
    step_ms = [sum(parts[j][i] for j in range(NPARTS)) for i in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    tokens_per_s = whole_job_rate(world, T, args.steps, total_ms)

    # The two GEMMs as separate launches (no programmatic overlap), each between its own events,
    # cold L2: how the pair's time divides (reported beside the step, not part of it).
    sep = [[], []]
    for i in range(max(3, args.steps // 2) + 3):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        flush.fill_(i & 0xFF)
        e[0].record(stream)
        mxq.wo_a_einsum_mxfp8(O, WA, T, G, NA, KA, z_q=zq, z_sf_128x4=zsf, status=status)
        e[1].record(stream)
        mxq.gemm_mxfp8_bf16(Z, WB, out, status=status)
        e[2].record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            sep[0].append(e[0].elapsed_time(e[1]))
            sep[1].append(e[1].elapsed_time(e[2]))
    mxq.check_status(status)

    # end-to-end through the public API: pinned host inputs -> device -> chain -> host result.
    # Two buffer slots and three streams: step i+1's inputs go in (copy stream) while step i
    # computes, and step i's output comes back (read-back stream) while step i+1 computes.
    x_h = x.cpu().pin_memory()
    o_h = o.cpu().pin_memory()
    slots = []
    for _ in range(2):
        slots.append({"x": torch.empty_like(x), "o": torch.empty_like(o),
                      "out": torch.empty((T, NB), dtype=torch.bfloat16, device=dev),
                      "out_h": torch.empty((T, NB), dtype=torch.bfloat16, pin_memory=True),
                      "comp_done": torch.cuda.Event(),
                      "out_done": torch.cuda.Event()})
    # inputs go in as N_IN row chunks on N_IN streams, so that several copy engines share them
    N_IN = args.copy_streams
    s_ins = [torch.cuda.Stream(dev) for _ in range(N_IN)]
    s_out = torch.cuda.Stream(dev)
    for k in slots:
        k["in_done"] = [torch.cuda.Event() for _ in range(N_IN)]

    def chunks(t):
        return t.chunk(N_IN, dim=0)

    def e2e_step(i):
        k = slots[i & 1]
        for j, si in enumerate(s_ins):
            si.wait_event(k["comp_done"])  # the slot's inputs were consumed two steps ago
            with torch.cuda.stream(si):
                chunks(k["x"])[j].copy_(chunks(x_h)[j], non_blocking=True)
                chunks(k["o"])[j].copy_(chunks(o_h)[j], non_blocking=True)
                k["in_done"][j].record(si)
        for ev in k["in_done"]:
            stream.wait_event(ev)
        stream.wait_event(k["out_done"])  # the slot's output has been read back
        mxq.rmsnorm_dual_out(k["x"], gamma, synth.RMS_EPS, y, yq, sf_packed=ysf)
        mxq.mxfp8_quantize(k["o"], oq, None, None, osf)
        mxq.o_proj_mxfp8(O, WA, WB, T, G, NA, KA, NB, zq, zsf, k["out"], status=status)
        k["comp_done"].record(stream)
        s_out.wait_event(k["comp_done"])
        with torch.cuda.stream(s_out):
            k["out_h"].copy_(k["out"], non_blocking=True)
            k["out_done"].record(s_out)

    for i in range(max(1, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(1e3 * (time.perf_counter() - t0), world, dev)
    e2e_tps = whole_job_rate(world, T, args.steps, e2e_ms)
    out_h = slots[0]["out_h"]

    hbm, bf16_tf, peak_kind = load_peaks()
    mx_tf = 2.0 * bf16_tf  # fp8 dense rate = 2x bf16 (nominal 4.5 / 2.25 PFLOP/s)

    def rate(byts, flops, us):
        d = {"us": round(us, 3), "GB/s": round(byts / us / 1e3, 1)}
        roof_us = max(byts / hbm / 1e3, flops / mx_tf / 1e6)
        if flops:
            d["TFLOP/s"] = round(flops / us / 1e6, 1)
        d["roofline_us"] = round(roof_us, 3)
        d["frac"] = round(roof_us / us, 4)
        if flops:
            d["frac_nominal"] = round(max(byts / NOMINAL_HBM_GBS / 1e3, flops / NOMINAL_MXFP8_TFLOPS / 1e6) / us, 4)
        return d

    mean_us = [1e3 * statistics.mean(pj) for pj in parts]
    o_proj_bytes, o_proj_flops = wo_a_bytes(T) + wo_b_bytes(T), FLOP_PER_TOKEN * T
    detail = {"rmsnorm_dual_out": rate(rms_bytes(T), 0, mean_us[0]),
              "mxfp8_quantize": rate(quant_bytes(T, G * KA), 0, mean_us[1]),
              "o_proj_mxfp8": rate(o_proj_bytes, o_proj_flops, mean_us[2]),
              "wo_a_separate_launch": rate(wo_a_bytes(T), wo_a_flops(T), 1e3 * statistics.mean(sep[0])),
              "wo_b_separate_launch": rate(wo_b_bytes(T), wo_b_flops(T), 1e3 * statistics.mean(sep[1]))}
    # the dominant call of the step: the _o_proj pair (its two kernels, one call)
    dom = max(range(NPARTS), key=lambda j: mean_us[j])
    dom_name = ["rmsnorm_dual_out", "mxfp8_quantize", "o_proj_mxfp8"][dom]
    dom_b, dom_f = [(rms_bytes(T), 0), (quant_bytes(T, G * KA), 0), (o_proj_bytes, o_proj_flops)][dom]
    dom_us = mean_us[dom]
    if dom_f and dom_f / mx_tf / 1e6 >= dom_b / hbm / 1e3:
        roof = {"kernel": dom_name + (" (wo_a + wo_b launches of one call)" if dom == 2 else ""),
                "bound": "tensor", "achieved": round(dom_f / dom_us / 1e6, 1),
                "peak": round(mx_tf, 1), "unit": "TFLOP/s",
                "peak_note": f"{peak_kind} bf16 burst x 2 (fp8/bf16 nominal ratio)",
                "peak_nominal": NOMINAL_MXFP8_TFLOPS}
        roof["frac_nominal"] = round(roof["achieved"] / NOMINAL_MXFP8_TFLOPS, 4)
    else:
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": round(dom_b / dom_us / 1e3, 1),
                "peak": hbm, "unit": "GB/s", "peak_note": f"{peak_kind} copy bandwidth",
                "peak_nominal": NOMINAL_HBM_GBS}
        roof["frac_nominal"] = round(roof["achieved"] / NOMINAL_HBM_GBS, 4)
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = traffic_for(dom_name, T)

    sweep_res = compact_sweep(mxq, synth, torch, dev, WA, WB) if rank == 0 and not args.no_sweep else None
    sampler.__exit__(None, None, None)
    clocks = sampler.summary()
    clocks["window"] = "warm-up, timed steps and the compact sweep"
    res = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/ue8m0 (fp32 accum)",
        "data": "synthetic (seeded SplitMix64 + Box-Muller, shapes of the pages' workloads)",
        "config": chain_config(T, world),
        "parts": detail,
        "roofline": roof,
        "e2e": {"value": round(e2e_tps, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": x_h.numel() * 2 + o_h.numel() * 2, "d2h_bytes_per_step": out_h.numel() * 2},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clocks,
        "wall_ms_per_step_incl_l2_flush": round(1e3 * wall / args.steps, 4),
    }
    if sweep_res is not None:
        res["sweep"] = sweep_res
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args, T, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
        if args.sweep:
            sweep(args, mxq, synth, torch, dev, WA, WB)
    if world > 1:
        dist.destroy_process_group()


# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) from the committed ncu
# captures (profiles/), keyed by (kernel, tokens), with the sources the capture was taken on and
# their SHA-1: once those sources change the figure no longer describes the kernel and reads null.
_GEMM_SRC = ("mxfp8_activation_quant_gb300/csrc/gemm_mxf8.cu", "mxfp8_activation_quant_gb300/csrc/mxq_device.cuh")
TRAFFIC = {
    ("o_proj_mxfp8", 4096): (173_101_312 + 24_235_520 + 127_094_016 + 37_409_792, _GEMM_SRC, "dd6c97c2802a395a"),
}


def traffic_for(kernel, T):
    entry = TRAFFIC.get((kernel, T))
    if entry is None:
        return None
    nbytes, srcs, sha = entry
    blob = b"".join(open(os.path.join(ROOT, f), "rb").read() for f in srcs)
    return nbytes if hashlib.sha1(blob).hexdigest()[:16] == sha else None


class GraphTimer:
    """us per call, the way the pages time _o_proj: the calls replayed from a CUDA graph with an
    L2 flush before each, minus the same graph holding only the flushes (median of 5 replays)."""

    def __init__(self, torch, dev):
        self.torch = torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = torch.empty(max(4 * l2, 256 << 20), dtype=torch.uint8, device=dev)
        self.cap = torch.cuda.Stream(dev)

    def __call__(self, fn, reps=20):
        torch, flush, cap = self.torch, self.flush, self.cap
        with torch.cuda.stream(cap):
            fn()
            flush.fill_(0)
        torch.cuda.synchronize()
        g1, g0 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=cap):
            for i in range(reps):
                flush.fill_(i & 0xFF)
                fn()
        with torch.cuda.graph(g0, stream=cap):
            for i in range(reps):
                flush.fill_(i & 0xFF)
        per = []
        for g in (g1, g0):
            g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3 / reps)
            per.append(statistics.median(ts))
        del g1, g0
        return per[0] - per[1]


def o_proj_roofline_us(T, hbm, mx_tf):
    """max(bytes at the HBM peak, FLOPs at the MXFP8 peak) for the _o_proj pair at T tokens."""
    byts = WEIGHT_BYTES + T * (G * KA * 33 // 32 + 2 * KB * 33 // 32 + NB * 2)
    return max(byts / hbm / 1e3, FLOP_PER_TOKEN * T / mx_tf / 1e6)


def _o_proj_case(mxq, synth, torch, dev, T):
    o = synth.o_proj_activation(0, T, device=dev)
    oq, osf = mxq.quantize(o, layouts=(2,))
    c = {"o": o, "O": mxq.MXFP8(oq, osf[2]), "oq": oq, "osf": osf[2],
         "zq": torch.empty((T, KB), dtype=torch.uint8, device=dev), "zsf": mxq.empty_sf(2, T, KB, dev),
         "zb": torch.empty((T, KB), dtype=torch.bfloat16, device=dev),
         "out": torch.empty((T, NB), dtype=torch.bfloat16, device=dev)}
    c["Z"] = mxq.MXFP8(c["zq"], c["zsf"])
    return c


def _o_proj_fused_unfused(mxq, timer, c, T, WA, WB):
    fused = timer(lambda: mxq.o_proj_mxfp8(c["O"], WA, WB, T, G, NA, KA, NB, c["zq"], c["zsf"], c["out"]))

    def unfused():  # wo_a writes bf16 z, the standalone quantizer, wo_b
        mxq.wo_a_einsum_mxfp8(c["O"], WA, T, G, NA, KA, z_bf16=c["zb"])
        mxq.mxfp8_quantize(c["zb"], c["zq"], None, None, c["zsf"])
        mxq.gemm_mxfp8_bf16(c["Z"], WB, c["out"])

    return fused, timer(unfused)


SWEEP_O_PROJ_T = [1, 16, 64, 128, 256, 384, 512, 4096, 32768]
SWEEP_QUANT_T = [4096, 32768]
SWEEP_RMS_T = [1024, 4096, 8192]
SWEEP_F2_T = [64, 1024, 8192]


def compact_sweep(mxq, synth, torch, dev, WA, WB):
    """Every configuration of the metric in one object, timed as the pages time _o_proj (a CUDA
    graph per call, cold L2): the _o_proj pair fused and unfused, the quantizer, RMSNorm, and
    this library's own MXFP8 GEMM on a square 8192^3 problem (a measured dense MXFP8 rate)."""
    hbm, bf16_tf, kind = load_peaks()
    mx_tf = 2 * bf16_tf
    timer = GraphTimer(torch, dev)
    res = {"timing": "CUDA graph per call, L2 flushed before each (graph of flushes alone subtracted), "
                     "median of 5 replays of 20 calls",
           "peaks": {"hbm_GB/s": hbm, "mxfp8_TFLOP/s": mx_tf, "kind": kind + " (mxfp8 = 2 x bf16 burst)",
                     "nominal_hbm_GB/s": NOMINAL_HBM_GBS, "nominal_mxfp8_TFLOP/s": NOMINAL_MXFP8_TFLOPS}}
    rows = []
    for T in SWEEP_O_PROJ_T:
        c = _o_proj_case(mxq, synth, torch, dev, T)
        fused, unf = _o_proj_fused_unfused(mxq, timer, c, T, WA, WB)
        r = {"T": T, "fused_us": round(fused, 2), "unfused_us": round(unf, 2), "saving_us": round(unf - fused, 2),
             "TFLOP/s": round(FLOP_PER_TOKEN * T / fused / 1e6, 1),
             "roofline_us": round(o_proj_roofline_us(T, hbm, mx_tf), 2),
             "frac": round(o_proj_roofline_us(T, hbm, mx_tf) / fused, 4),
             "frac_nominal": round(o_proj_roofline_us(T, NOMINAL_HBM_GBS, NOMINAL_MXFP8_TFLOPS) / fused, 4)}
        # bf16 o quantized inside wo_a (no quantize launch for o either), against the standalone
        # quantize launch followed by the fused pair
        r["from_bf16_us"] = round(timer(lambda: mxq.o_proj_mxfp8_from_bf16(
            c["o"], WA, WB, T, G, NA, KA, NB, c["zq"], c["zsf"], c["out"])), 2)
        r["quantize_then_fused_us"] = round(timer(lambda: (
            mxq.mxfp8_quantize(c["o"], c["oq"], None, None, c["osf"]),
            mxq.o_proj_mxfp8(c["O"], WA, WB, T, G, NA, KA, NB, c["zq"], c["zsf"], c["out"]))), 2)
        rows.append(r)
        del c
    res["o_proj"] = rows
    q = []
    for T in SWEEP_QUANT_T:
        xq = synth.quantizer_input(0, T, device=dev)
        qq = torch.empty((T, KB), dtype=torch.uint8, device=dev)
        sf = mxq.empty_sf(2, T, KB, dev)
        us = timer(lambda: mxq.mxfp8_quantize(xq, qq, None, None, sf))
        b = quant_bytes(T, KB)
        q.append({"shape": [T, KB], "us": round(us, 2), "GB/s": round(b / us / 1e3, 1),
                  "frac_hbm": round(b / us / 1e3 / hbm, 4), "frac_nominal": round(b / us / 1e3 / NOMINAL_HBM_GBS, 4)})
        del xq, qq, sf
    res["mxfp8_quantize"] = q
    rm = []
    for T in SWEEP_RMS_T:
        xr = synth.rmsnorm_input(0, T, device=dev)
        gm = synth.rmsnorm_gamma(0, device=dev)
        yr = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        yrq = torch.empty((T, H), dtype=torch.uint8, device=dev)
        sf = mxq.empty_sf(1, T, H, dev)
        us = timer(lambda: mxq.rmsnorm_dual_out(xr, gm, synth.RMS_EPS, yr, yrq, sf_packed=sf))
        b = rms_bytes(T)
        rm.append({"shape": [T, H], "us": round(us, 2), "GB/s": round(b / us / 1e3, 1),
                   "frac_hbm": round(b / us / 1e3 / hbm, 4), "frac_nominal": round(b / us / 1e3 / NOMINAL_HBM_GBS, 4)})
        del xr, yr, yrq, sf
    res["rmsnorm_dual_out"] = rm
    # the second producer -> consumer pair: RMSNorm's MXFP8 y fed straight into the MXFP8 GEMM
    # (fused_wqa_wkv stand-in, 5120 -> synth.WQKV_N), against quantizing RMSNorm's bf16 y with a
    # standalone launch before the same GEMM
    wqq, wqs = mxq.quantize(synth.wqa_wkv_weight(0, device=dev), layouts=(2,))
    wq = mxq.MXFP8(wqq, wqs[2])
    f2 = []
    for T in SWEEP_F2_T:
        xr = synth.rmsnorm_input(0, T, device=dev)
        gm = synth.rmsnorm_gamma(0, device=dev)
        yr = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        yrq = torch.empty((T, H), dtype=torch.uint8, device=dev)
        sf = mxq.empty_sf(2, T, H, dev)
        yq2 = torch.empty_like(yrq)
        sf2 = mxq.empty_sf(2, T, H, dev)
        out = torch.empty((T, synth.WQKV_N), dtype=torch.bfloat16, device=dev)
        chain = timer(lambda: (mxq.rmsnorm_dual_out(xr, gm, synth.RMS_EPS, yr, yrq, sf_128x4=sf),
                               mxq.gemm_mxfp8_bf16(mxq.MXFP8(yrq, sf), wq, out)))
        quant = timer(lambda: mxq.mxfp8_quantize(yr, yq2, None, None, sf2))
        f2.append({"T": T, "rmsnorm_then_gemm_us": round(chain, 2), "standalone_quantize_of_y_us": round(quant, 2)})
        del xr, yr, yrq, sf, yq2, sf2, out
    res["rmsnorm_to_mxfp8_gemm"] = {"gemm": f"{H} -> {synth.WQKV_N}", "rows": f2}
    n = 8192
    A = mxq.MXFP8(*_rand_mx(mxq, synth, n, n, synth.TID_SQ_A, dev))
    B = mxq.MXFP8(*_rand_mx(mxq, synth, n, n, synth.TID_SQ_B, dev))
    cc = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
    us = timer(lambda: mxq.gemm_mxfp8_bf16(A, B, cc), reps=5)
    tf = 2 * n ** 3 / us / 1e6
    res["mxfp8_gemm_8192^3"] = {"us": round(us, 2), "TFLOP/s": round(tf, 1), "frac": round(tf / mx_tf, 4),
                                "frac_nominal": round(tf / NOMINAL_MXFP8_TFLOPS, 4)}
    # every _o_proj fraction once more against this library's own dense MXFP8 rate
    for r in rows:
        r["frac_own_gemm_peak"] = round(o_proj_roofline_us(r["T"], hbm, tf) / r["fused_us"], 4)
    return res


def sweep(args, mxq, synth, torch, dev, WA, WB):
    """Per-config lines for the design tables (more token counts than the compact object):
    quantizer, RMSNorm, and the _o_proj pair fused vs unfused with each GEMM alone."""
    hbm, bf16_tf, _ = load_peaks()
    mx_tf = 2 * bf16_tf
    timer = GraphTimer(torch, dev)
    for T in [1, 16, 256, 4096, 32768]:
        x = synth.quantizer_input(0, T, device=dev)
        q = torch.empty((T, KB), dtype=torch.uint8, device=dev)
        sf = mxq.empty_sf(2, T, KB, dev)
        us = timer(lambda: mxq.mxfp8_quantize(x, q, None, None, sf))
        b = quant_bytes(T, KB)
        print(json.dumps({"sweep": "mxfp8_quantize", "T": T, "us": round(us, 3), "GB/s": round(b / us / 1e3, 1),
                          "frac_hbm": round(b / us / 1e3 / hbm, 4)}), flush=True)
        del x, q
    for T in [1, 64, 1024, 4096, 8192]:
        x = synth.rmsnorm_input(0, T, device=dev)
        g = synth.rmsnorm_gamma(0, device=dev)
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        yq = torch.empty((T, H), dtype=torch.uint8, device=dev)
        sf = mxq.empty_sf(1, T, H, dev)
        us = timer(lambda: mxq.rmsnorm_dual_out(x, g, synth.RMS_EPS, y, yq, sf_packed=sf))
        b = rms_bytes(T)
        print(json.dumps({"sweep": "rmsnorm_dual_out", "T": T, "us": round(us, 3), "GB/s": round(b / us / 1e3, 1),
                          "frac_hbm": round(b / us / 1e3 / hbm, 4)}), flush=True)
    for T in [1, 2, 4, 8, 16, 64, 128, 256, 384, 512, 1024, 2048, 4096, 8192, 16384, 32768]:
        c = _o_proj_case(mxq, synth, torch, dev, T)
        fused, unf = _o_proj_fused_unfused(mxq, timer, c, T, WA, WB)
        extra = {}
        # bf16 o quantized inside wo_a, against the quantize launch + the fused pair
        extra["from_bf16_us"] = round(timer(lambda: mxq.o_proj_mxfp8_from_bf16(
            c["o"], WA, WB, T, G, NA, KA, NB, c["zq"], c["zsf"], c["out"])), 3)
        extra["quantize_then_fused_us"] = round(timer(lambda: (
            mxq.mxfp8_quantize(c["o"], c["oq"], None, None, c["osf"]),
            mxq.o_proj_mxfp8(c["O"], WA, WB, T, G, NA, KA, NB, c["zq"], c["zsf"], c["out"]))), 3)
        wa_us = timer(lambda: mxq.wo_a_einsum_mxfp8(c["O"], WA, T, G, NA, KA, z_q=c["zq"], z_sf_128x4=c["zsf"]))
        wb_us = timer(lambda: mxq.gemm_mxfp8_bf16(c["Z"], WB, c["out"]))
        roof = o_proj_roofline_us(T, hbm, mx_tf)
        print(json.dumps({"sweep": "o_proj", "T": T, "fused_us": round(fused, 3), "unfused_us": round(unf, 3),
                          "saving_us": round(unf - fused, 3), "wo_a_us": round(wa_us, 3), "wo_b_us": round(wb_us, 3),
                          "TFLOP/s": round(FLOP_PER_TOKEN * T / fused / 1e6, 1), "roofline_us": round(roof, 3),
                          "frac": round(roof / fused, 4),
                          "weight_GB/s": round(WEIGHT_BYTES / fused / 1e3, 1), **extra}), flush=True)
        del c


def _rand_mx(mxq, synth, rows, cols, tid, dev):
    """MXFP8 (bytes, F8_128x4 scales) of a seeded normal bf16 matrix, quantized by the library."""
    x = synth.normal_bf16(0, tid, rows, cols, 1.0, device=dev)
    q, sfs = mxq.quantize(x, layouts=(2,))
    return q, sfs[2]


# ---- the CPU oracle (cpu_baseline and the reference arm) -----------------------------------
_ORACLE_STATE = {}


def _oracle_setup(T_sample):
    import numpy as np
    import torch

    import oracle
    from mxfp8_activation_quant_gb300 import synth

    if "wa_d" not in _ORACLE_STATE:
        def bits(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        waq, wasf = oracle.quantize_bf16(bits(synth.wo_a_weight(0)))
        wbq, wbsf = oracle.quantize_bf16(bits(synth.wo_b_weight(0)))
        _ORACLE_STATE["wa_d"] = oracle.dequant(waq, wasf)
        _ORACLE_STATE["wb_d"] = oracle.dequant(wbq, wbsf)
        _ORACLE_STATE["bits"] = bits
    bits = _ORACLE_STATE["bits"]
    rows = torch.arange(T_sample)
    return (bits(synth.rmsnorm_input(0, T_sample)), bits(synth.rmsnorm_gamma(0)),
            bits(synth.o_proj_activation(0, T_sample, rows=rows)))


def _oracle_step(xb, gb, ob):
    import oracle
    from mxfp8_activation_quant_gb300 import synth

    y = oracle.bf16_round(oracle.rmsnorm(xb, gb, synth.RMS_EPS))
    oracle.quantize_bf16(y)
    oq, osf = oracle.quantize_bf16(ob)
    z = oracle.einsum_wo_a(oracle.dequant(oq, osf), _ORACLE_STATE["wa_d"], G)
    zq, zsf = oracle.quantize_bf16(oracle.bf16_round(z))
    return oracle.gemm_nt(oracle.dequant(zq, zsf), _ORACLE_STATE["wb_d"])


def cpu_baseline(args, T, budget_s=15.0):
    """The oracle as it stands, on the host cores, over a bounded token sample of the same
    workload (RMSNorm + quantize + _o_proj for the first `n` tokens); tokens/s."""
    import oracle

    oracle.build()
    n = 2
    xb, gb, ob = _oracle_setup(n)
    t0 = time.perf_counter()
    _oracle_step(xb, gb, ob)
    dt = time.perf_counter() - t0
    n = max(2, min(T, int(n * budget_s / max(dt, 1e-3) / 2)))
    xb, gb, ob = _oracle_setup(n)
    t0 = time.perf_counter()
    _oracle_step(xb, gb, ob)
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {n} of the {T} tokens: fp64 RMSNorm + quantize + o quantize + wo_a + z quantize + wo_b"}


def run_reference(args):
    """The reference arm: the CPU oracle timed on this machine's host cores, rank 0 only (the other
    ranks return at once, without work)."""
    world, rank, _ = rank_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    T = args.tokens
    n = max(1, args.ref_tokens)
    xb, gb, ob = _oracle_setup(n)
    for _ in range(args.warmup):
        _oracle_step(xb, gb, ob)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(xb, gb, ob)
    dt = time.perf_counter() - t0
    tps = n * args.steps / dt
    sample = f"{n} of the {T} tokens per step: fp64 RMSNorm + quantize + o quantize + wo_a + z quantize + wo_b"
    res = {"impl": "reference", "metric": METRIC, "value": round(tps, 3), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": chain_config(T, world),
           "cpu_baseline": {"value": round(tps, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(tps, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true", help="also print the per-config design-table lines")
    ap.add_argument("--no-sweep", action="store_true", help="leave the compact sweep out of the line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-tokens", type=int, default=4)
    ap.add_argument("--copy-streams", type=int, default=1, help="streams for the end-to-end input copies")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
