#!/usr/bin/env python3
"""Benchmark of the MXFP8 block-scaled fused-MoE expert forward on GB300.

One step = one pass of the whole layer hot path through the C ABI
(moe_forward_mxfp8: top-k routing + fused MX activation quant + permutation,
grouped GEMM1 + SwiGLU + MXFP8 requant, grouped GEMM2, finalize) on the
Qwen3-30B-A3B-shaped 16K-token prefill layer (T=16384, H=2048, E=128, top-8,
I=768).  Expert weights are MX-quantized at load (outside the timed region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM, each step timed with CUDA events on the launching stream and
L2 flushed (a 256 MB write, then a 256 MB read) between steps; `e2e` is the same metric through the
same public call with pinned host buffers, the host<->device copies inside
the timed region.  Multi-GPU (torchrun): independent replicas, weak scaling.
`--impl reference` times the CPU oracle (the only reference on this path) on
a bounded sample of the same workload, on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and MXFP8 TFLOP/s (frac of peak); route/quant GB/s vs HBM"
WORKLOAD = "qwen3_30b_prefill"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0   # nominal dense ratio (4.5 / 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0   # nominal dense ratio (13.5 / 2.25 PFLOP/s): e2m1 x e2m1 MMAs

# DRAM traffic of one grouped GEMM1 launch on the bench workload: ncu's
# dram__bytes_read.sum + dram__bytes_write.sum from a one-pass capture of the
# profile_case layer run, keyed by the hash of the GEMM sources it was taken
# on (a changed kernel reports no traffic until it is captured again)
NCU_TRAFFIC = {"a9ec3d6a1d8bbad4": 786553600, "64d58b0d55536f8c": 786384128,
               "f21fe81032a4b103": 786399488, "afe529db44d76b76": 787179008,
               "318d8521ea941ed5": 786471936, "7ede47c7a46a5cfc": 787526144,
               "1c20b020eb8a1633": 787512064, "cc23eb524901ee20": 787625984,
               "5238fc07798b52b4": 787269376, "16b1bf2dc0156978": 787060736,
               "0fd02ef804c608ce": 787518976}


def max_over_ranks(torch, dist, ms, world, device):
    """The slowest rank's time (MAX all-reduce over the job; the local time
    when world == 1)."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, tokens_per_rank, steps, max_ms):
    """Whole-job tokens/s: every replica processes its tokens in every step;
    the job takes as long as its slowest rank."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-linear", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        def pick(*keys):
            for k in keys:
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k])
            return None
        hbm = pick("hbm_gbs", "hbm_GBs")
        bf16 = pick("bf16_tflops", "bf16_TFLOPs")
        bf16s = pick("bf16_tflops_sustained")
        if hbm and bf16:
            return dict(hbm_gbs=hbm, bf16_tflops=bf16, bf16_tflops_sustained=bf16s or bf16,
                        source="measured")
    return dict(FALLBACK_PEAKS, source="fallback")


GEMM_SOURCES = ("gemm.cu", "gemm2sm.cu", "gemm_common.cuh", "tiled_scales.h", "common.cuh",
                "api.cu")


def gemm_src_hash():
    """Hash of the sources the grouped GEMM kernels and their 1-SM / 2-SM
    choice (api.cu) are compiled from; the stored ncu traffic is only
    reported while it matches."""
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "mxfp8_block_scaled_moe_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks/throttle sampling (every 20 ms) around the timed
    region; `mark_start` / `mark_end` bracket the region and `summary` keeps
    the samples that arrived inside it."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.gpu_index = gpu_index
        self.proc = None
        self.enabled = enabled
        self.samples = []          # (arrival time, line)
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.samples.append((time.time(), line))

    def __enter__(self):
        if self.enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
            if self.proc is not None:
                self.thread = threading.Thread(target=self._reader, daemon=True)
                self.thread.start()
                t_wait = time.time() + 3.0   # let the sampler start before the region
                while not self.samples and time.time() < t_wait:
                    time.sleep(0.01)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.thread.join(timeout=5)

    def summary(self):
        inside = [l for t, l in self.samples
                  if self.t0 is not None and self.t1 is not None and self.t0 <= t <= self.t1]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in inside:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "interval_ms": 20,
                "region_s": round(self.t1 - self.t0, 3)}


def library_gemm_rates(torch, dev, n=8192, reps=10):
    """Dense n^3 GEMM rates of the vendor library on this GPU (context for the
    MXFP8 peak): bf16, and MXFP8 through torch._scaled_mm with e4m3 operands
    and e8m0 block-32 scales.  Best of `reps`; None where unsupported."""
    def best(fn):
        fn()
        torch.cuda.synchronize()
        t = []
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            t.append(a.elapsed_time(b))
        return 2.0 * n ** 3 / min(t) / 1e9
    out = {"n": n}
    try:
        x = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
        w = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
        out["bf16_tflops"] = round(best(lambda: x @ w.t()), 1)
        del x, w
    except Exception:
        out["bf16_tflops"] = None
    try:
        a8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        sc = torch.full((n * (n // 32),), 127, dtype=torch.uint8, device=dev).view(
            torch.float8_e8m0fnu)
        out["mxfp8_tflops"] = round(best(lambda: torch._scaled_mm(
            a8, b8.t(), scale_a=sc, scale_b=sc, out_dtype=torch.bfloat16)), 1)
        del a8, b8, sc
    except Exception:
        out["mxfp8_tflops"] = None
    torch.cuda.empty_cache()
    return out


LINEAR_BENCH = ("qwen3vl_vision_fc2", "qwen3vl_vision_fc1", "qwen3_8b_down_prefill",
                "qwen3_8b_gate_up_prefill", "qwen3_8b_down_decode")


def dense_linear_bench(torch, mm, workloads, dev, flush, stream, peak, hbm, fp4=False):
    """The dense MXFP8 (or, fp4, W4A4) linear on the pages' dense shapes: per
    call (L2 flushed), the activation quant and the GEMM from the library's
    event profiler, GEMM TFLOP/s against the MXFP8 (MXFP4) peak `peak` (weight
    GB/s against HBM for the 32-token decode), and the vendor library's MXFP8
    GEMM on the same shape with unit scales (GEMM only; None where it rejects
    the shape)."""
    out = {}
    for name in LINEAR_BENCH:
        shape = workloads.LINEAR_CONFIGS[name]
        M, N, K = shape.M, shape.N, shape.K
        if fp4 and K % 128:
            continue
        x, w = workloads.make_linear(shape, dev)
        lin = (mm.MXFP4Linear if fp4 else mm.MXFP8Linear).from_bf16(w)
        del w
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            lin(x, out=y)
        torch.cuda.synchronize()
        reps = 50 if M <= 128 else 20
        mm.api.layer_profile_enable(True)
        tot, q, g = [], [], []
        for _ in range(reps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            lin(x, out=y)
            b.record(stream)
            b.synchronize()
            tot.append(a.elapsed_time(b))
            pr = mm.api.linear_profile_read()
            q.append(pr["act_quant"])
            g.append(pr["gemm"])
        mm.api.layer_profile_enable(False)
        t_ms, q_ms, g_ms = (statistics.mean(v) for v in (tot, q, g))
        flops = 2.0 * M * N * K
        wbytes = N * K * ((0.5 if fp4 else 1) + 1 / 32)
        ent = {"M": M, "N": N, "K": K, "scales_per_row": -(-K // 32),
               "ms": round(t_ms, 4), "act_quant_ms": round(q_ms, 4), "gemm_ms": round(g_ms, 4),
               "gemm_TFLOP/s": round(flops / (g_ms / 1e3) / 1e12, 1),
               ("gemm_frac_fp4_peak" if fp4 else "gemm_frac_fp8_peak"):
                   round(flops / (g_ms / 1e3) / 1e12 / peak, 3),
               "call_TFLOP/s": round(flops / (t_ms / 1e3) / 1e12, 1)}
        if M <= 128:
            ent["gemm_weight_GB/s"] = round(wbytes / (g_ms / 1e3) / 1e9, 1)
            ent["gemm_frac_hbm"] = round(wbytes / (g_ms / 1e3) / 1e9 / hbm, 3)
        ent["vendor_mxfp8_gemm_ms"] = None
        if K % 32 == 0 and not fp4:
            try:
                a8 = torch.randn(M, K, device=dev).to(torch.float8_e4m3fn)
                b8 = torch.randn(N, K, device=dev).to(torch.float8_e4m3fn)
                sa = torch.full((M * K // 32,), 127, dtype=torch.uint8, device=dev).view(
                    torch.float8_e8m0fnu)
                sb = torch.full((N * K // 32,), 127, dtype=torch.uint8, device=dev).view(
                    torch.float8_e8m0fnu)
                fn = lambda: torch._scaled_mm(a8, b8.t(), scale_a=sa, scale_b=sb,  # noqa: E731
                                              out_dtype=torch.bfloat16)
                fn()
                vt = time_fn(torch, fn, reps, flush, torch.cuda.current_stream())
                ent["vendor_mxfp8_gemm_ms"] = round(statistics.mean(vt), 4)
                del a8, b8, sa, sb
            except Exception:
                pass
        out[name] = ent
        del x, y, lin
        torch.cuda.empty_cache()
    return out


def gemm_algorithmic(T, H, E_touched, k, I):
    """Flops and bytes of the two grouped GEMMs of one layer call: every
    expanded row read once, every touched expert's weights (payload + e8m0
    scales) read once, the outputs written once."""
    M = T * k
    sc = 1 + 1 / 32
    g1 = dict(flops=2.0 * M * 2 * I * H,
              bytes=M * H * sc + E_touched * 2 * I * H * sc + M * I * sc)
    g2 = dict(flops=2.0 * M * H * I,
              bytes=M * I * sc + E_touched * H * I * sc + 2.0 * M * H)
    return g1, g2


def kernel_roofline(ms, flops, nbytes, fp8_peak, hbm):
    """TFLOP/s and GB/s of one launch, their fractions of the MXFP8 tensor
    peak and of HBM, and the fraction of the launch's own roofline (the
    larger of its tensor-bound and HBM-bound times over the measured one)."""
    tf = flops / (ms / 1e3) / 1e12
    gb = nbytes / (ms / 1e3) / 1e9
    t_tensor = flops / (fp8_peak * 1e12) * 1e3
    t_hbm = nbytes / (hbm * 1e9) * 1e3
    return {"ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_fp8_peak": round(tf / fp8_peak, 4),
            "GB/s": round(gb, 1), "frac_hbm": round(gb / hbm, 4),
            "bound": "tensor" if t_tensor >= t_hbm else "hbm",
            "frac_roofline": round(max(t_tensor, t_hbm) / ms, 4)}


CONFIG_BENCH = (("qwen3_30b_decode", None), ("qwen3_235b_prefill", None)) + tuple(
    ("qwen3_30b_skewed", t) for t in (1, 8, 128, 1024, 4096, 16384))


def layer_config_bench(torch, mm, workloads, dev, flush, stream, name, T, fp8_peak, hbm,
                       steps=20):
    """One layer configuration, timed like the headline step (L2 flushed,
    CUDA events on the stream) with the library's per-kernel events: tokens/s
    and each kernel against its roofline."""
    shape = workloads.CONFIGS[name] if T is None else workloads.CONFIGS[name].with_tokens(T)
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    inp = workloads.make_layer(shape, dev)
    if shape.offline:
        layer = mm.MXFP8MoELayer.from_quantized(inp["w13q"], inp["w13s"], inp["w2q"], inp["w2s"],
                                                k)
    else:
        layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], k)
    for key in ("w13", "w2", "w13q", "w13s", "w2q", "w2s"):
        inp.pop(key, None)
    x, logits = inp["x"], inp["logits"]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    counts = mm.moe_route_quant_mxfp8(x, logits, k)["expert_counts"].cpu()
    e_touched = int((counts > 0).sum())
    for _ in range(3):
        layer(x, logits, out=out)
    torch.cuda.synchronize()
    # eager calls (no instrumentation), then a pass with events at every
    # kernel boundary for the per-kernel times
    step_ms = statistics.mean(time_fn(torch, lambda: layer(x, logits, out=out), steps, flush,
                                      stream))
    mm.api.layer_profile_enable(True)
    prof = []
    for _ in range(steps):
        flush()
        layer(x, logits, out=out)
        prof.append(mm.api.layer_profile_read())
    mm.api.layer_profile_enable(False)
    # the same call replayed from a CUDA graph (no host launch cost)
    graph_ms = None
    try:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            layer(x, logits, out=out)
        stream.wait_stream(gs)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer(x, logits, out=out)
        g.replay()
        torch.cuda.synchronize()
        graph_ms = statistics.mean(time_fn(torch, g.replay, steps, flush, stream))
        del g
    except Exception as exc:  # graph capture unavailable: report the eager time only
        graph_ms = f"unavailable: {exc}"
    if mm.device_status() != 0:
        raise RuntimeError(f"device status error in the {shape.name} layer")

    def km(key):
        return statistics.mean(p_[key] for p_ in prof)
    ab = algorithmic_bytes(T, H, E, k, I)
    g1, g2 = gemm_algorithmic(T, H, e_touched, k, I)
    r_ms, f_ms = km("route_quant"), km("finalize")
    ent = {"T": T, "H": H, "E": E, "k": k, "I": I, "experts_touched": e_touched,
           "max_expert_rows": int(counts.max()), "empty_experts": int((counts == 0).sum()),
           "ms_per_step": round(step_ms, 4), "tokens_per_s": round(T / (step_ms / 1e3), 1),
           "graph_ms_per_step": round(graph_ms, 4) if isinstance(graph_ms, float) else graph_ms,
           "graph_tokens_per_s": (round(T / (graph_ms / 1e3), 1)
                                  if isinstance(graph_ms, float) else None),
           "route_quant": {"ms": round(r_ms, 4), "GB/s": round(ab["route"] / r_ms / 1e6, 1),
                           "frac_hbm": round(ab["route"] / r_ms / 1e6 / hbm, 4)},
           "gemm1_swiglu_quant": kernel_roofline(km("gemm1_swiglu_quant"), g1["flops"],
                                                 g1["bytes"], fp8_peak, hbm),
           "gemm2": kernel_roofline(km("gemm2"), g2["flops"], g2["bytes"], fp8_peak, hbm),
           "finalize": {"ms": round(f_ms, 4), "GB/s": round(ab["finalize"] / f_ms / 1e6, 1),
                        "frac_hbm": round(ab["finalize"] / f_ms / 1e6 / hbm, 4)},
           "steps": steps}
    if T <= 32 and H % 256 == 0 and I % 128 == 0:
        # the library runs both grouped GEMMs as one kernel here (its profile
        # gives the pair's time as gmm1's): one roofline over both GEMMs' work
        pair_ms = km("gemm1_swiglu_quant") + km("gemm2")
        ent["gemms_one_kernel"] = kernel_roofline(pair_ms, g1["flops"] + g2["flops"],
                                                  g1["bytes"] + g2["bytes"], fp8_peak, hbm)
        ent["gemm1_swiglu_quant"] = ent["gemm2"] = "in gemms_one_kernel"
    del layer, inp, x, logits, out
    torch.cuda.empty_cache()
    return shape.name, ent


def algorithmic_bytes(T, H, E, k, I):
    M = T * k
    route = 2 * T * H + M * H + M * H // 32 + 4 * T * E + M * 4 * 4
    twostep = (2 * T * H + 2 * M * H) + (2 * M * H + M * H + M * H // 32) + 4 * T * E + M * 16
    fin = 2 * M * H + 2 * T * H + M * 8
    wq = (E * 2 * I * H + E * H * I) * (2 + 1 + 1 / 32)
    return dict(route=route, twostep=twostep, finalize=fin, weight_quant=wq)


class L2Flush:
    """Evicts the L2 (129 MB) before a timed step: a 256 MB write, then a 256 MB
    read of a second buffer.  The read writes the first buffer's dirty lines
    back to HBM before the step starts; without it the step itself pays for
    that write-back (~129 MB: 12 us of a 32-token decode layer, 4 us of the
    16K-token prefill, measured)."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def time_fn(torch, fn, iters, flush_buf, stream):
    """Per-call CUDA-event times (ms) on `stream`, L2 flushed before each call."""
    ts = []
    for _ in range(iters):
        flush_buf()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return ts


def cpu_baseline_run(shape, inp_host, weights_host, n_tokens):
    """Time the CPU oracle on the first n_tokens tokens of the same workload."""
    import numpy as np
    from oracle import moe as omoe
    xb, logits = inp_host
    w13q, w13s, w2q, w2s = weights_host
    t0 = time.perf_counter()
    omoe.moe_forward(xb[:n_tokens], logits[:n_tokens], w13q, w13s, w2q, w2s, shape.k, shape.I)
    dt = time.perf_counter() - t0
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    return dict(value=n_tokens / dt, unit="tokens/s", cores=cores, kind="oracle",
                sample=f"first {n_tokens} of {shape.T} tokens of the {shape.name} layer through the "
                       f"fp64 NumPy oracle (all {shape.E} experts' weights dequantized per call), "
                       f"{dt:.1f} s wall")


def _oracle_quant_expert(w_bits):
    """Load-time weight quant of one expert by the oracle (process-pool worker)."""
    from oracle import mx as omx
    return omx.mx_quantize(omx.bf16_bits_to_f64(w_bits))


def _oracle_quant_weights(w):
    """Quantize bf16 [E, N, K] weights with the oracle, one expert per task."""
    import multiprocessing as mp
    import numpy as np
    import torch
    bits = w.view(torch.int16).numpy().view(np.uint16)
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(32, os.cpu_count() or 1)) as pool:
        res = pool.map(_oracle_quant_expert, [bits[e] for e in range(bits.shape[0])])
    return np.stack([r[0] for r in res]), np.stack([r[1] for r in res])


def run_reference(args):
    """The oracle as the reference arm: rank 0 only, bounded sample per step.

    Each step runs the oracle's whole layer (routing, fused quant, both grouped
    GEMMs with their per-expert weight dequant, finalize) on a fixed sample of
    the workload's tokens; the weights are quantized once, by the oracle, at
    load time (outside the timed steps, as on the GPU arm)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch
    from mxfp8_block_scaled_moe_gb300 import workloads
    from oracle import moe as omoe
    shape = workloads.CONFIGS[args.config]
    n_tok = 8
    inp = workloads.make_layer(shape, "cpu", weights=False)
    xb = inp["x"].view(torch.int16).numpy().view(np.uint16)
    logits = inp["logits"].numpy()
    if shape.offline:
        w13q, w13s, w2q, w2s = (t.numpy() for t in workloads.make_weights_offline(shape, "cpu"))
    else:
        w13, w2 = workloads.make_weights_bf16(shape, "cpu")
        w13q, w13s = _oracle_quant_weights(w13)
        w2q, w2s = _oracle_quant_weights(w2)
        del w13, w2
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        omoe.moe_forward(xb[:n_tok], logits[:n_tok], w13q, w13s, w2q, w2s, shape.k, shape.I)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = n_tok * len(times) / total
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    cb = dict(value=value, unit="tokens/s", cores=cores, kind="oracle",
              sample=f"first {n_tok} of {shape.T} tokens of the {shape.name} layer per step "
                     f"through the fp64 NumPy oracle (every touched expert's weights "
                     f"dequantized per call)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{shape.name}: T={shape.T} H={shape.H} E={shape.E} "
                                   f"top-{shape.k} I={shape.I}",
                       "sample_tokens_per_step": n_tok},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_moe_gb300 as mm
    from mxfp8_block_scaled_moe_gb300 import workloads

    shape = workloads.CONFIGS[args.config]
    T, H, E, k, I = shape.T, shape.H, shape.E, shape.k, shape.I
    M = T * k
    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16

    inp = workloads.make_layer(shape, dev)
    stream = torch.cuda.current_stream()
    # ---- load time: weight MX quant (timed separately, not part of the step)
    if shape.offline:
        layer = mm.MXFP8MoELayer.from_quantized(inp["w13q"], inp["w13s"], inp["w2q"], inp["w2s"], k)
        wq_ms = None
        layer4 = layer44 = None
    else:
        flush = L2Flush(torch, dev)
        mm.mx_quantize_3d(inp["w13"])  # warm
        torch.cuda.synchronize()
        wq_t = time_fn(torch, lambda: (mm.mx_quantize_3d(inp["w13"]), mm.mx_quantize_3d(inp["w2"])),
                       3, flush, stream)
        wq_ms = min(wq_t)
        layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], k)
        # the W4A8 variant (MXFP4 weights) from the same bf16 weights, and its
        # load-time quantizer rate
        wq4_ms = min(time_fn(torch, lambda: (mm.mx_quantize_fp4_3d(inp["w13"]),
                                             mm.mx_quantize_fp4_3d(inp["w2"])), 3, flush, stream))
        layer4 = mm.W4A8MoELayer.from_bf16(inp["w13"], inp["w2"], k)
        # W4A4: the same MXFP4 weights, MXFP4 expert inputs
        layer44 = mm.W4A4MoELayer.from_quantized(layer4.w13p, layer4.w13s, layer4.w2p, layer4.w2s,
                                                 k)
        del inp["w13"], inp["w2"]
    x, logits = inp["x"], inp["logits"]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = layer.workspace(T, dev)
    flush = L2Flush(torch, dev)

    def step():
        layer(x, logits, out=out)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if mm.device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    # ---- timed region: exactly K steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # CUDA events around gmm1 only (the roofline's kernel); the other kernel
    # boundaries keep their overlapped launches
    mm.api.layer_profile_enable("gemm1")
    step_ms, prof = [], []
    with ClockSampler(local_rank, enabled=not args.no_clocks) as clk:
        clk.mark_start()
        for _ in range(args.steps):
            flush()
            ev_a = torch.cuda.Event(enable_timing=True)
            ev_b = torch.cuda.Event(enable_timing=True)
            ev_a.record(stream)
            step()
            ev_b.record(stream)
            ev_b.synchronize()
            step_ms.append(ev_a.elapsed_time(ev_b))
            prof.append(mm.api.layer_profile_read())
        torch.cuda.synchronize()
        clk.mark_end()
    mm.api.layer_profile_enable(False)
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(torch, dist, sum(step_ms), world, dev)
    value = whole_job_rate(world, T, args.steps, total_ms)

    # ---- gmm1 inside the timed steps (library events on the stream); the
    # other kernels from a pass with events at every boundary, after the
    # timed region
    gemm1_ms = statistics.mean(p_["gemm1_swiglu_quant"] for p_ in prof)
    reps_b = max(5, min(args.steps, 20))
    mm.api.layer_profile_enable(True)
    prof_all = []
    for _ in range(reps_b):
        flush()
        step()
        prof_all.append(mm.api.layer_profile_read())
    mm.api.layer_profile_enable(False)

    def kmean(key):
        return statistics.mean(p_[key] for p_ in prof_all)
    route_ms, gemm2_ms, fin_ms = kmean("route_quant"), kmean("gemm2"), kmean("finalize")
    # the two-step comparator (bf16 permute, then a separate quant pass)
    reps = max(5, min(args.steps, 20))

    def twostep():
        rr = mm.moe_route_permute_bf16(x, logits, k)
        mm.mx_quantize_3d(rr["xp"])
    twostep_ms = statistics.median(time_fn(torch, twostep, reps, flush, stream))
    torch.cuda.synchronize()
    if mm.device_status() != 0:
        raise RuntimeError("device status error during timing")

    ab = algorithmic_bytes(T, H, E, k, I)
    g1_alg, g2_alg = gemm_algorithmic(T, H, E, k, I)
    gemm1_flops = 2.0 * M * (2 * I) * H
    gemm2_flops = 2.0 * M * H * I
    gemm1_tflops = gemm1_flops / (gemm1_ms * 1e-3) / 1e12
    gemm2_tflops = gemm2_flops / (gemm2_ms * 1e-3) / 1e12
    hbm = peaks["hbm_gbs"]
    src_hash = gemm_src_hash()
    traffic = NCU_TRAFFIC.get(src_hash)
    roofline = {"bound": "tensor", "kernel": "grouped_gemm_swiglu_quant_mxfp8",
                "achieved": round(gemm1_tflops, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                "frac": round(gemm1_tflops / fp8_peak, 4), "traffic": traffic,
                "peak_source": f"{peaks['source']}: bf16 dense burst {peaks['bf16_tflops']} TFLOP/s "
                               f"x {FP8_OVER_BF16} (nominal fp8/bf16 ratio)",
                "flops_per_launch": gemm1_flops, "launch_ms": round(gemm1_ms, 4),
                "timing": "mean over the timed steps, CUDA events recorded by the library "
                          "around this kernel on the launching stream"}
    kernels = {
        "route_quant": {"ms": route_ms, "GB/s": ab["route"] / route_ms / 1e6,
                        "frac_hbm": ab["route"] / route_ms / 1e6 / hbm},
        "two_step_route_then_quant": {"ms": twostep_ms, "GB/s": ab["twostep"] / twostep_ms / 1e6},
        "gemm1_swiglu_quant": kernel_roofline(gemm1_ms, g1_alg["flops"], g1_alg["bytes"],
                                              fp8_peak, peaks["hbm_gbs"]),
        "gemm2": kernel_roofline(gemm2_ms, g2_alg["flops"], g2_alg["bytes"], fp8_peak,
                                 peaks["hbm_gbs"]),
        "finalize": {"ms": fin_ms, "GB/s": ab["finalize"] / fin_ms / 1e6,
                     "frac_hbm": ab["finalize"] / fin_ms / 1e6 / hbm},
    }
    if wq_ms:
        kernels["weight_quant_load_time"] = {"ms": wq_ms, "GB/s": ab["weight_quant"] / wq_ms / 1e6,
                                             "frac_hbm": ab["weight_quant"] / wq_ms / 1e6 / hbm}
    for v in kernels.values():
        for kk in list(v):
            if isinstance(v[kk], float):
                v[kk] = round(v[kk], 4)

    # ---- end to end through the public host-buffer call (copies overlapped with compute)
    x_h = x.cpu().pin_memory()
    l_h = logits.cpu().pin_memory()
    o_h = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        layer.forward_host(x_h, l_h, out_host=o_h)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if not torch.equal(o_h, out.cpu()):
        raise RuntimeError("host-buffer layer output differs from the device layer")
    e2e_t = time_fn(torch, e2e_step, args.steps, flush, stream)
    e2e_max_ms = max_over_ranks(torch, dist, sum(e2e_t), world, dev)
    e2e_value = whole_job_rate(world, T, args.steps, e2e_max_ms)
    h2d = x_h.numel() * 2 + l_h.numel() * 4
    d2h = o_h.numel() * 2
    # vendor-library dense GEMM rates (context for the MXFP8 peak; after the
    # timed work, rank 0)
    lib_rates = library_gemm_rates(torch, dev) if rank == 0 else None
    # the W4A8 variant (MXFP4 expert weights): the same prefill step, and a
    # 32-token decode slice (weight-streaming bound) for both weight formats
    w4a8 = None
    if layer4 is not None:
        def layer_ms(lyr, xx, ll, reps):
            lyr(xx, ll)
            torch.cuda.synchronize()
            mm.api.layer_profile_enable(True)
            ts, pr = [], []
            for _ in range(reps):
                flush()
                a_ = torch.cuda.Event(enable_timing=True)
                b_ = torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                lyr(xx, ll)
                b_.record(stream)
                b_.synchronize()
                ts.append(a_.elapsed_time(b_))
                pr.append(mm.api.layer_profile_read())
            mm.api.layer_profile_enable(False)
            return statistics.mean(ts), statistics.mean(p_["gemm1_swiglu_quant"] for p_ in pr)
        p_ms, p_g1 = layer_ms(layer4, x, logits, 20)
        Td = 32
        d4_ms, _ = layer_ms(layer4, x[:Td], logits[:Td], 50)
        d8_ms, _ = layer_ms(layer, x[:Td], logits[:Td], 50)
        wbytes4 = E * (2 * I * H + H * I) * (0.5 + 1 / 32)
        wbytes8 = E * (2 * I * H + H * I) * (1 + 1 / 32)
        w4a8 = {
            "weights": "MXFP4: packed e2m1 + e8m0 block-32 scales; activations MXFP8",
            "prefill": {"tokens_per_s": round(T / (p_ms / 1e3), 1), "ms_per_step": round(p_ms, 4),
                        "gemm1_TFLOP/s": round(2.0 * T * k * 2 * I * H / (p_g1 / 1e3) / 1e12, 1)},
            "decode_T32": {"w4a8_ms": round(d4_ms, 4), "mxfp8_ms": round(d8_ms, 4),
                           "w4a8_weight_GB/s": round(wbytes4 / (d4_ms / 1e3) / 1e9, 1),
                           "mxfp8_weight_GB/s": round(wbytes8 / (d8_ms / 1e3) / 1e9, 1),
                           "note": "all experts touched: the layer streams every expert's weights"},
            "weight_quant_load_time": {"ms": round(wq4_ms, 4),
                                       "GB/s": round(E * 3 * I * H * (2 + 0.5 + 1 / 32) / (wq4_ms / 1e3) / 1e9, 1)},
            "parity": "tests/test_gpu_w4a8.py (quantizer bit-exact; layer vs oracle; byte-identical to the MXFP8 layer on re-encoded weights)",
        }
    w4a4 = None
    if layer44 is not None:
        p_ms, p_g1 = layer_ms(layer44, x, logits, 20)
        d44_ms, _ = layer_ms(layer44, x[:32], logits[:32], 50)
        w4a4 = {
            "weights": "MXFP4 (packed e2m1 + e8m0 block-32 scales); both grouped GEMMs' inputs "
                       "MXFP4-quantized on the device; e2m1 x e2m1 MMAs of kind::mxf4 on packed "
                       "operands",
            "prefill": {"tokens_per_s": round(T / (p_ms / 1e3), 1), "ms_per_step": round(p_ms, 4),
                        "gemm1_TFLOP/s": round(2.0 * T * k * 2 * I * H / (p_g1 / 1e3) / 1e12, 1),
                        "gemm1_frac_fp4_peak": round(2.0 * T * k * 2 * I * H / (p_g1 / 1e3) / 1e12
                                                     / (fp8_peak / FP8_OVER_BF16 * FP4_OVER_BF16),
                                                     3)},
            "decode_T32": {"ms": round(d44_ms, 4)},
            "dense_linear": (dense_linear_bench(torch, mm, workloads, dev, flush, stream,
                                                fp8_peak / FP8_OVER_BF16 * FP4_OVER_BF16, hbm,
                                                fp4=True) if not args.no_linear else None),
            "fp4_peak": {"TFLOP/s": round(fp8_peak / FP8_OVER_BF16 * FP4_OVER_BF16, 1),
                         "source": f"{peaks['source']}: bf16 dense burst x {FP4_OVER_BF16} "
                                   "(nominal fp4/bf16 ratio)"},
            "parity": "tests/test_gpu_w4a4.py (exact W4A4 GEMM pins; layer vs oracle; sampled "
                      "prefill tokens vs oracle)",
        }

    # the router gate GEMM fused with softmax top-k (the step upstream of the
    # routing), and the layer run from hidden states + gate
    router = None
    if rank == 0 and not shape.offline and shape.zipf_s == 0:
        gate = workloads.make_gate(shape, dev)
        mm.moe_router_gate_topk(x, gate, k)
        torch.cuda.synchronize()
        r_t = time_fn(torch, lambda: mm.moe_router_gate_topk(x, gate, k), 50, flush, stream)
        r_ms = statistics.mean(r_t)
        v_t = time_fn(torch, lambda: torch.matmul(x, gate.t()).float(), 50, flush, stream)
        g_t = time_fn(torch, lambda: layer.forward_gated(x, gate, out=out), 20, flush, stream)
        r_bytes = T * H * 2 + E * H * 2 + T * k * 8
        router = {
            "ms": round(r_ms, 4), "GB/s": round(r_bytes / (r_ms / 1e3) / 1e9, 1),
            "frac_hbm": round(r_bytes / (r_ms / 1e3) / 1e9 / hbm, 3),
            "TFLOP/s": round(2.0 * T * E * H / (r_ms / 1e3) / 1e12, 1),
            "algorithmic_bytes": r_bytes,
            "vendor_bf16_gate_gemm_ms": round(statistics.mean(v_t), 4),
            "gated_layer_ms": round(statistics.mean(g_t), 4),
            "gated_layer_tokens_per_s": round(T / (statistics.mean(g_t) / 1e3), 1),
            "note": "gate GEMM + top-k + weights + in-block ranks in one kernel; the vendor "
                    "figure is the logits GEMM alone (torch.matmul, bf16 -> fp32)",
            "parity": "tests/test_gpu_router.py (exact integer logits with ties; top-k equal to "
                      "the oracle on the device logits and byte-identical to the logits-input "
                      "routing; gated layer byte-identical)",
        }
        del gate

    # the dense MXFP8 linear (partial K blocks, ragged N) on the pages' dense shapes
    dense = None
    if rank == 0 and not args.no_linear:
        dense = dense_linear_bench(torch, mm, workloads, dev, flush, stream, fp8_peak, hbm)
        dense["parity"] = ("tests/test_gpu_linear.py (row quant bit-exact incl. the partial block; "
                           "exact structured GEMM; sampled outputs of every shape vs oracle)")

    # every other layer configuration: decode, the 235B offline prefill and
    # the skewed-load sweep (each against its own roofline)
    configs = None
    if rank == 0 and not args.no_configs:
        configs = {}
        for cname, cT in CONFIG_BENCH:
            key, ent = layer_config_bench(torch, mm, workloads, dev, flush, stream, cname, cT,
                                          fp8_peak, hbm)
            configs[key] = ent

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import mx as omx  # noqa: F401
        xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
        lg = logits.cpu().numpy()
        wh = tuple(t.cpu().numpy() for t in (layer.w13q, layer.w13s, layer.w2q, layer.w2s))
        cpu_base = cpu_baseline_run(shape, (xb, lg), wh, 128)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8 e4m3+e8m0, fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": f"{shape.name}: T={T} H={H} E={E} top-{k} I={I}, seeded "
                                   "N(0,1) hidden with 1% outlier channels x20, N(0,0.02) bf16 "
                                   "weights MX-quantized at load",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed before every timed step by a 256 MB write and then a 256 MB "
                             "read (the flush's dirty lines reach HBM before the step)",
                       "timing": "CUDA events per step on the launching stream"},
            "roofline": roofline,
            "kernels": kernels,
            "kernels_timing": "gemm1_swiglu_quant: library CUDA events around it inside the "
                              "timed steps; route_quant, gemm2, finalize: a separate pass of "
                              f"{reps_b} steps with events at every kernel boundary (L2 "
                              "flushed), after the timed region",
            "clocks": clk.summary(),
            "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_max_ms / args.steps, 4)},
            "gpu_launches": 6 * args.steps,
            "e2e_api": "moe_forward_mxfp8_host (pinned host buffers, default chunk plan 3/16 | 5/8 | 3/16 of the tokens, "
                       "H2D / compute / D2H on three streams)",
            "cpu_baseline": cpu_base,
            "w4a8": w4a8,
            "router": router,
            "dense_linear": dense,
            "w4a4": w4a4,
            "configs": configs,
            "peaks": {"hbm_gbs": hbm, "fp8_tflops": fp8_peak, "source": peaks["source"],
                      "library_dense_gemm": lib_rates},
            "gemm_src": src_hash,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
