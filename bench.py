#!/usr/bin/env python
"""Benchmark of the quantized mul_mat hot path on GB300.

Headline (one JSON line on stdout): decode GB/s of the Q4_K x Q8_K GEMV,
M = 1, N = K = 4096. One step = the whole decode path for one token batch:
quantize the fp32 activations to Q8_K (kernel 1) and run the GEMV over the
packed Q4_K weights (kernel 2). Inputs are resident in HBM; 32 copies of the
packed weights are used in rotation (302 MB, above the 129 MB L2), so every
step streams its weights from HBM. Steps are replayed as CUDA graphs of 64
steps so that the host's launch rate does not set the pace.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun each rank runs the same workload on its own GPU (replicas,
weak scaling; the path has no exchange step, so there is no data-path
collective); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "quantized mul_mat GB/s (M=1) and TOPS (M=512) vs GB300 roofline"
GRAPH_STEPS = 64
COPIES = 32
WORKLOAD = ("Q4_K x Q8_K GEMV decode, M=1, N=K=4096 (16 super-blocks of 256 per row, 6-bit "
            "scale/min in 12 bytes, fp16 d/dmin); W ~ N(0,0.02) + per-row offset N(0,0.005); "
            "X ~ N(0,1); seed 0")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ environment
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.uuid = None
        try:
            u = torch.cuda.get_device_properties(device).uuid
            self.uuid = str(u)
        except Exception:
            pass
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            if self.uuid and self.uuid.replace("GPU-", "") not in f[0]:
                continue
            rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


GEMV_SOURCES = ["block_quantized_matmul_q4_gb300/csrc/gemv.cu",
                "block_quantized_matmul_q4_gb300/csrc/qmm_internal.cuh"]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel_key)
    if not rec or rec.get("source_digest") != source_digest(GEMV_SOURCES):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ GPU arm
def step_bytes(q, N, K, M):
    """Algorithmic bytes of one step: weight blocks + Q8_K activations +
    fp32 outputs + the fp32 activations the quantizer reads."""
    w = N * (K // 256) * 144
    xq = M * (K // 256) * 292
    return w, xq, M * N * 4, M * K * 4


def capture(fn, n, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i)
    return g


def run_graphs(big, small, n_big):
    for _ in range(n_big):
        big.replay()
    if small is not None:
        small.replay()


LEAD_SPIN_CYCLES = 2_000_000  # about 1 ms of SM clock: covers the host's enqueue of the replays


def timed(stream, fn, lead_spin=False):
    """Run fn() between CUDA events on `stream`; returns seconds. With
    lead_spin, a spin kernel runs on `stream` just before the start event, so
    that the work fn() enqueues is queued up by the time the start event is
    reached."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if lead_spin:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(LEAD_SPIN_CYCLES)
    a.record(stream)
    with torch.cuda.stream(stream):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / 1e3


def job_rate(t_local: float, units_local: float, world: int, device) -> tuple:
    """Whole-job throughput of a weak-scaling run: every rank processed
    units_local units in t_local seconds; the job took the slowest rank's
    time, and value = (units of all ranks) / that time / 1e9. Collective over
    the default process group when world > 1 (each rank ran the same K steps,
    so the unit counts are equal)."""
    t = t_local
    if world > 1:
        tt = torch.tensor([t_local], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.barrier()
        t = float(tt.item())
    return t, units_local * world / t / 1e9


def gpu_arm(args, rank, world):
    import block_quantized_matmul_q4_gb300 as q
    dev = torch.device("cuda", torch.cuda.current_device())
    L = wl.GEMV_Q4_K_4096
    N, K, M = L.N, L.K, 1
    wt = q.QMM_TYPE_Q4_K

    # inputs resident in HBM
    w = wl.weights(0, N, K, L.wstd, row_offset_std=L.row_offset_std, device=dev)
    Wq = q.empty_blocks(wt, N, K)
    q.qmm_quantize_weights(wt, w, Wq, N, K)
    del w
    Wp0 = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, Wq, Wp0, N, K)
    copies = [Wp0] + [Wp0.clone() for _ in range(COPIES - 1)]
    X = wl.activations(0, M, K, device=dev)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    Y = torch.empty(M, N, device=dev)
    stream = torch.cuda.Stream()

    def step(i):
        q.qmm_mul_mat_ws(wt, copies[i % COPIES], N, K, X, M, Y, ws, ws_bytes, stream)

    def gemv_only(i):
        q.qmm_mul_mat_prepared(wt, copies[i % COPIES], N, K, ws, ws_bytes, M, Y, stream)

    # warm-up outside capture (module load, function attributes), then graphs:
    # the timed region replays g_big n_big times and g_small once, exactly
    # args.steps steps
    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    n0 = q.qmm_kernel_launch_count()
    g_big = capture(step, GRAPH_STEPS, stream)
    launches_per_step = (q.qmm_kernel_launch_count() - n0) // GRAPH_STEPS
    n_big, rem = divmod(args.steps, GRAPH_STEPS)
    g_small = capture(step, rem, stream) if rem else None
    wrem = args.warmup % GRAPH_STEPS
    g_wsmall = capture(step, wrem, stream) if wrem else None
    g_gemv = capture(gemv_only, GRAPH_STEPS, stream)
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)  # the sampler's first rows
    # warm-up (untimed): args.warmup steps, then one replay of every graph the
    # timed region uses (a graph's first launch uploads it), back to back
    with torch.cuda.stream(stream):
        run_graphs(g_big, g_wsmall, args.warmup // GRAPH_STEPS)
        if n_big:
            g_big.replay()
        if g_small is not None:
            g_small.replay()
    torch.cuda.synchronize()

    # timed region: exactly K steps. A spin kernel ahead of the start event
    # keeps the GPU busy while the host enqueues the replays, so the events
    # time the steps and not the host's launch latency.
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t = timed(stream, lambda: run_graphs(g_big, g_small, n_big), lead_spin=True)
    torch.cuda.synchronize()
    bw, bxq, by, bx = step_bytes(q, N, K, M)
    per_step = bw + bxq + by + bx
    t, value = job_rate(t, per_step * args.steps, world, dev)

    # dominant kernel. With M*K this small the activation quantizer runs inside
    # the GEMV (one kernel per step), so the step's event timing is the
    # kernel's. The GEMV on prepared activations is timed too, back to back
    # over the rotating copies: one warm replay, then at least 8 timed.
    reps = max(8, min(2000, args.steps // GRAPH_STEPS))
    with torch.cuda.stream(stream):
        g_gemv.replay()
    t_prep = timed(stream, lambda: run_graphs(g_gemv, None, reps), lead_spin=True) / (reps * GRAPH_STEPS)
    clk = clocks.stop()
    peaks = load_peaks()
    if launches_per_step == 1:
        kname, t_kern, kbytes = "gemv_q4_K_kernel<1, fused>", t / args.steps, per_step
    else:
        kname, t_kern, kbytes = "gemv_q4_K_kernel<1, staged>", t_prep, bw + bxq + by
    achieved = kbytes / t_kern / 1e9
    traffic = profiled_traffic("gemv_q4_K_4096_m1")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "kernel": kname, "kernel_us": round(t_kern * 1e6, 3),
                "algorithmic_bytes": kbytes, "peak_source": peaks["source"],
                "launches_per_step": launches_per_step,
                "prepared_gemv_us": round(t_prep * 1e6, 3)}

    # end to end through the public C-ABI call with host buffers: per step one
    # qmm_mul_mat_host call (pinned, mapped buffers): a kernel pulls X from
    # host memory into device memory, the GEMV quantizes it and stores Y into
    # pinned host memory, all in stream order; eager launches, no graph
    e2e_steps = max(3, min(args.steps, 3000))
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(M, N).pin_memory()
    hbytes = q.qmm_host_call_bytes(wt, M, N, K)
    hbuf = torch.empty(hbytes, dtype=torch.uint8, device=X.device)
    sptr = stream.cuda_stream
    wptrs = [c.data_ptr() for c in copies]
    xp, yp, bp = Xh.data_ptr(), Yh.data_ptr(), hbuf.data_ptr()
    call = q._lib.qmm_mul_mat_host

    def e2e_loop():
        for i in range(e2e_steps):
            st = call(wt, wptrs[i % COPIES], N, K, xp, M, yp, bp, hbytes, q.QMM_HOST_MAPPED, sptr)
            if st:
                q._check("qmm_mul_mat_host", st)

    for i in range(3):
        call(wt, wptrs[i], N, K, xp, M, yp, bp, hbytes, q.QMM_HOST_MAPPED, sptr)
    t_e2e = timed(stream, e2e_loop)
    e2e = {"value": round(per_step * e2e_steps * world / t_e2e / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": Xh.numel() * 4, "d2h_bytes_per_step": Yh.numel() * 4,
           "steps": e2e_steps, "path": "qmm_mul_mat_host with QMM_HOST_MAPPED (C ABI, one call per step: a kernel pulls the pinned host X into device memory, the GEMV stores Y into pinned host memory), eager"}
    q.qmm_check_device_error(stream)

    extras = {}
    if args.extras:
        extras = gpu_extras(q, dev, stream, args)

    return {
        "value": round(value, 2), "ms_per_step": t / args.steps * 1e3, "roofline": roofline,
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clk,
        "extras": extras,
    }


def gemv_rate(q, dev, stream, wt, N, K, M, seed, L=None, steps=6400, copies=None, hot=0.0):
    """GB/s of qmm_mul_mat_ws (quantizer + GEMV) on one projection; weights
    rotate over enough copies to exceed L2."""
    if L is None:
        w = wl.weights(seed, N, K, 0.02, row_offset_std=0.005, device=dev)
    else:
        w = wl.weights(seed, N, K, L.wstd, row_offset_std=L.row_offset_std,
                       outlier_frac=L.outlier_frac, device=dev)
    Wq = q.empty_blocks(wt, N, K)
    q.qmm_quantize_weights(wt, w, Wq, N, K)
    del w
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, Wq, Wp, N, K)
    del Wq
    nbytes = Wp.numel()
    ncopies = copies or max(1, min(32, -(-300_000_000 // nbytes)))
    cps = [Wp] + [Wp.clone() for _ in range(ncopies - 1)]
    X = wl.activations(seed, M, K, hot_frac=hot, device=dev)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    Y = torch.empty(M, N, device=dev)

    def step(i):
        q.qmm_mul_mat_ws(wt, cps[i % ncopies], N, K, X, M, Y, ws, ws_bytes, stream)

    for i in range(3):
        step(i)
    g = capture(step, GRAPH_STEPS, stream)
    reps = max(3, steps // GRAPH_STEPS)
    with torch.cuda.stream(stream):
        g.replay()
    t = timed(stream, lambda: run_graphs(g, None, reps)) / (reps * GRAPH_STEPS)
    qk = 32 if wt == q.QMM_TYPE_Q4_0 else 256
    bq = 34 if wt == q.QMM_TYPE_Q4_0 else 292
    b = nbytes * N // (-(-N // 8) * 8) + M * (K // qk) * bq + M * N * 4 + M * K * 4
    del cps, Wp
    return t, b


def prefill_rate(q, dev, stream, L, M, seed, reps=6, graph_steps=4, wt=None):
    """Prefill mul_mat (prefill quantizer + tcgen05 GEMM) on one shape: us per
    call and TOPS (2 M N K multiply-adds per call), plus the GEMM alone on
    prepared activations."""
    wt = q.QMM_TYPE_Q4_K if wt is None else wt
    N, K = L.N, L.K
    off = L.row_offset_std if wt != q.QMM_TYPE_Q4_0 else 0.0
    w = wl.weights(seed, N, K, L.wstd, row_offset_std=off, device=dev)
    Wq = q.empty_blocks(wt, N, K)
    q.qmm_quantize_weights(wt, w, Wq, N, K)
    del w
    Wp = q.empty_packed(wt, N, K)
    q.qmm_repack_weights(wt, Wq, Wp, N, K)
    del Wq
    X = wl.activations(seed, M, K, device=dev)
    ws_bytes = q.qmm_workspace_bytes(wt, M, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    Y = torch.empty(M, N, device=dev)
    step = lambda i: q.qmm_mul_mat_ws(wt, Wp, N, K, X, M, Y, ws, ws_bytes, stream)
    gemm = lambda i: q.qmm_mul_mat_prepared(wt, Wp, N, K, ws, ws_bytes, M, Y, stream)
    for i in range(2):
        step(i)
        gemm(i)
    g1 = capture(step, graph_steps, stream)
    g2 = capture(gemm, graph_steps, stream)
    with torch.cuda.stream(stream):
        g1.replay()
        g2.replay()
    t1 = timed(stream, lambda: run_graphs(g1, None, reps)) / (reps * graph_steps)
    t2 = timed(stream, lambda: run_graphs(g2, None, reps)) / (reps * graph_steps)
    ops = 2.0 * M * N * K
    return {"us": round(t1 * 1e6, 2), "TOPS": round(ops / t1 / 1e12, 1),
            "gemm_us": round(t2 * 1e6, 2), "gemm_TOPS": round(ops / t2 / 1e12, 1)}


PEAK_KINDS = (("mma_sync_s8_m16n8k32", 0, 4000), ("mma_sync_f16_m16n8k16", 1, 4000),
              ("tcgen05_f16_128x128x16_smem_smem", 2, 20000), ("tcgen05_f16_128x128x16_tmem_smem", 3, 20000),
              ("tcgen05_f16_128x256x16_smem_smem", 4, 10000), ("tcgen05_f16_128x256x16_tmem_smem", 5, 10000))


def peaks_rate(q, dev, stream, reps=3):
    """Tensor throughput microbenchmarks (qmm_debug_peak): TFLOP/s (TOPS for
    s8) of back-to-back MMAs over the whole GPU, best of `reps` launches after
    one warm launch, each timed with CUDA events on `stream`."""
    out = {}
    for name, kind, iters in PEAK_KINDS:
        with torch.cuda.stream(stream):
            q.qmm_debug_peak(kind, iters, stream)
        best = None
        for _ in range(reps):
            ops = [0.0]

            def run():
                ops[0] = q.qmm_debug_peak(kind, iters, stream)
            t = timed(stream, run, lead_spin=True)
            best = t if best is None or t < best else best
        out[name] = {"TFLOP/s": round(ops[0] / best / 1e12, 1), "us": round(best * 1e6, 1)}
    q.qmm_check_device_error(stream)
    out["note"] = ("qmm_debug_peak: nonzero operands, all SMs, best of 3 launches; mma.sync: 32 warps "
                   "per SM x 8 independent accumulators; tcgen05: one CTA per SM, one thread "
                   "issuing K = 64 rounds into one TMEM accumulator")
    return out


def prefill_extras(q, dev, stream, peaks_measured=None):
    peaks = load_peaks()
    pm = peaks_measured or peaks_rate(q, dev, stream)
    s8 = pm["mma_sync_s8_m16n8k32"]["TFLOP/s"]
    tcf = pm["tcgen05_f16_128x128x16_tmem_smem"]["TFLOP/s"]
    out = {}
    for wt, tag in ((q.QMM_TYPE_Q4_K, "q4_K"), (q.QMM_TYPE_Q4_0, "q4_0"), (q.QMM_TYPE_Q6_K, "q6_K")):
        for L in wl.PREFILL_SHAPES:
            for M in wl.PREFILL_M:
                r = prefill_rate(q, dev, stream, L, M, 31, wt=wt)
                r["frac_of_fp16_peak"] = round(r["gemm_TOPS"] / peaks["bf16_tflops"], 4)
                r["frac_of_tcgen05_f16_measured"] = round(r["gemm_TOPS"] / tcf, 4)
                r["frac_of_int8_mma_sync_measured"] = round(r["gemm_TOPS"] / s8, 4)
                out[f"{tag}_{L.name}_M{M}"] = r
                torch.cuda.empty_cache()
    out["peak"] = {"value": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "note": "measured bf16 dense GEMM peak (cuBLAS); kind::f16 with fp16 operands "
                           "has the same nominal rate"}
    out["peaks_measured"] = pm
    return out


def w4a16_extras(q, dev, stream, reps=8, graph_steps=16, ms=None):
    """W4A16 on the 8192 x 8192, G = 128 layer at M in {1, 16, 256}: us per
    call, GB/s of algorithmic bytes (codes + scales + zeros + A + C) and
    TOPS (2 M N K). Rotating weight copies larger than L2 at M <= 16."""
    N = K = wl.W4A16_N
    G = wl.W4A16_G
    qc, s16, z, _ = wl.w4a16_inputs(9, N, K, G, 1, device=dev)
    v = qc.view(N, K // 8, 8).to(torch.int64)
    del qc
    word = torch.zeros(N, K // 8, dtype=torch.int64, device=dev)
    for i in range(8):
        word |= v[:, :, i] << (4 * i)
    del v
    qweight = (word - ((word >> 31) << 32)).to(torch.int32)
    del word
    Wp = torch.empty(q.qmm_packed_bytes(q.QMM_TYPE_W4A16, N, K), dtype=torch.uint8, device=dev)
    q.qmm_repack_weights(q.QMM_TYPE_W4A16, qweight, Wp, N, K)
    del qweight
    ncopies = 5  # 5 x 35 MB > the 129 MB L2
    sets = [(Wp, s16, z)] + [(Wp.clone(), s16.clone(), z.clone()) for _ in range(ncopies - 1)]
    wbytes = Wp.numel() + s16.numel() * 2 + z.numel()
    out = {}
    for M in (ms or wl.W4A16_M):
        A = wl.normal_rows(9, wl.S_A, M, K, device=dev).to(torch.float16)
        C = torch.empty(M, N, dtype=torch.float16, device=dev)
        nset = ncopies if M <= 16 else 1
        step = lambda i: q.qmm_w4a16(*sets[i % nset], G, A, C, M, N, K, stream)
        for i in range(nset):
            step(i)
        g = capture(step, graph_steps, stream)
        with torch.cuda.stream(stream):
            g.replay()
        t = timed(stream, lambda: run_graphs(g, None, reps)) / (reps * graph_steps)
        b = wbytes + 2 * M * K + 2 * M * N
        out[f"M{M}"] = {"us": round(t * 1e6, 3), "GB/s": round(b / t / 1e9, 1),
                        "TOPS": round(2.0 * M * N * K / t / 1e12, 2)}
        # the same codes and scales through a 16-entry code table (NF4-like)
        lut = wl.nf4_like_table().to(dev)
        step = lambda i: q.qmm_w4a16_lut(sets[i % nset][0], sets[i % nset][1], lut, G, A, C, M, N, K,
                                         stream)
        for i in range(nset):
            step(i)
        g = capture(step, graph_steps, stream)
        with torch.cuda.stream(stream):
            g.replay()
        t = timed(stream, lambda: run_graphs(g, None, reps)) / (reps * graph_steps)
        b = Wp.numel() + s16.numel() * 2 + 32 + 2 * M * K + 2 * M * N
        out[f"lut_M{M}"] = {"us": round(t * 1e6, 3), "GB/s": round(b / t / 1e9, 1),
                            "TOPS": round(2.0 * M * N * K / t / 1e12, 2)}
    out["shape"] = {"N": N, "K": K, "G": G}
    return out


def gpu_extras(q, dev, stream, args):
    out = {"peaks": peaks_rate(q, dev, stream)}
    out["prefill"] = prefill_extras(q, dev, stream, out["peaks"])
    out["w4a16_8192"] = w4a16_extras(q, dev, stream)
    torch.cuda.empty_cache()
    out["q6_K"] = q6_K_rate(q, dev, stream)
    out["q4_K_4096_M_sweep"] = sweep_rate(q, dev, stream)
    out["q4_0_q6_K_4096_M_sweep"] = small_m_rate(q, dev, stream)
    # Q4_0 x Q8_0 GEMV, 256 x 1024, M = 1 (L2-resident correctness case)
    Ls = wl.GEMV_Q4_0_SMALL
    t, b = gemv_rate(q, dev, stream, q.QMM_TYPE_Q4_0, Ls.N, Ls.K, 1, 0, Ls, copies=1)
    out["q4_0_256x1024_m1"] = {"us": round(t * 1e6, 3), "GB/s": round(b / t / 1e9, 1),
                               "note": "147 KB of weights stay in L2; latency-bound"}
    # 70B-shaped decode layer
    out["layer_70B_q4_K_m1"] = layer_rate(q, dev, stream)
    torch.cuda.empty_cache()
    per = {}
    for i, Lp in enumerate(wl.LAYER_70B):
        t, b = gemv_rate(q, dev, stream, q.QMM_TYPE_Q4_K, Lp.N, Lp.K, 1, 100 + i, Lp,
                         steps=640, hot=wl.LAYER_70B_HOT_FRAC)
        per[Lp.name] = {"us": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1)}
        torch.cuda.empty_cache()
    out["layer_70B_q4_K_m1"]["per_projection_alone"] = per
    return out


def q6_K_rate(q, dev, stream):
    """Q6_K x Q8_K decode (scalar GEMV, 6.5625 bits per weight): the 4096 x
    4096 shape at M in {1, 4, 16} and the 70B layer's largest projection
    (28672 x 8192) at M = 1; GB/s of algorithmic bytes."""
    out = {}
    L = wl.GEMV_Q4_K_4096
    for M in (1, 4, 16):
        t, b = gemv_rate(q, dev, stream, q.QMM_TYPE_Q6_K, L.N, L.K, M, 0, L)
        out[f"4096x4096_m{M}"] = {"us": round(t * 1e6, 3), "GB/s": round(b / t / 1e9, 1)}
    Lp = [x for x in wl.LAYER_70B if x.name == "gate_proj"][0]
    t, b = gemv_rate(q, dev, stream, q.QMM_TYPE_Q6_K, Lp.N, Lp.K, 1, 7, Lp, steps=640)
    out[f"{Lp.N}x{Lp.K}_m1"] = {"us": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1)}
    torch.cuda.empty_cache()
    return out


def small_m_rate(q, dev, stream):
    """Q4_0 and Q6_K at 4096 x 4096, M in {1, 2, 4, 8, 12, 16} through
    qmm_mul_mat_ws: M = 1 runs the scalar GEMV, M >= 2 the tensor-core one
    (with its activation image written by a quantizer launch ahead of it);
    us per call, weights rotating over 32 copies (302 MB, above L2), GB/s of
    the weight bytes."""
    out = {}
    L = wl.GEMV_Q4_K_4096
    for wt, tag in ((q.QMM_TYPE_Q4_0, "q4_0"), (q.QMM_TYPE_Q6_K, "q6_K")):
        w = wl.weights(0, L.N, L.K, 0.02, row_offset_std=0.0 if wt == q.QMM_TYPE_Q4_0 else 0.005,
                       device=dev)
        Wq = q.empty_blocks(wt, L.N, L.K)
        q.qmm_quantize_weights(wt, w, Wq, L.N, L.K)
        Wp = q.empty_packed(wt, L.N, L.K)
        q.qmm_repack_weights(wt, Wq, Wp, L.N, L.K)
        del w, Wq
        wbytes = Wp.numel()
        cps = [Wp] + [Wp.clone() for _ in range(31)]
        for M in (1, 2, 4, 8, 12, 16):
            X = wl.activations(0, M, L.K, device=dev)
            Y = torch.empty(M, L.N, device=dev)
            ws_bytes = max(q.qmm_workspace_bytes(wt, M, L.K), 16)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
            fn = lambda i: q.qmm_mul_mat_ws(wt, cps[i % 32], L.N, L.K, X, M, Y, ws, ws_bytes, stream)
            for i in range(3):
                fn(i)
            g = capture(fn, GRAPH_STEPS, stream)
            with torch.cuda.stream(stream):
                g.replay()
            t = timed(stream, lambda: run_graphs(g, None, 20)) / (20 * GRAPH_STEPS)
            out[f"{tag}_m{M}"] = {"us": round(t * 1e6, 3), "GB/s": round(wbytes / t / 1e9, 1)}
        del cps, Wp
        torch.cuda.empty_cache()
    return out


def sweep_rate(q, dev, stream, Ms=None):
    """The headline GEMV (Q4_K, N = K = 4096) at M in {1, 2, 4, 8, 16}: M = 1
    runs the scalar GEMV, M >= 2 the tensor-core one."""
    sweep = {}
    L = wl.GEMV_Q4_K_4096
    for M in Ms or wl.GEMV_Q4_K_M_SWEEP:
        t, b = gemv_rate(q, dev, stream, q.QMM_TYPE_Q4_K, L.N, L.K, M, 0, L)
        sweep[str(M)] = {"us": round(t * 1e6, 3), "GB/s": round(b / t / 1e9, 1),
                         "TOPS": round(2 * M * L.N * L.K / t / 1e12, 3)}
    return sweep


def layer_rate(q, dev, stream, reps=20, graph_steps=16):
    """The 70B-shaped decode layer (M = 1) as one step: q, k, v from one input
    (qmm_mul_mat_multi: one quantization, one launch), o, gate and up from one
    input (multi), down; and the same seven projections as seven qmm_mul_mat
    calls. The 481 MB of weights exceed L2, so each step reads them from HBM."""
    wt = q.QMM_TYPE_Q4_K
    Wp, Y = {}, {}
    wbytes = 0
    for i, Lp in enumerate(wl.LAYER_70B):
        w = wl.weights(100 + i, Lp.N, Lp.K, Lp.wstd, outlier_frac=Lp.outlier_frac, device=dev)
        Wq = q.empty_blocks(wt, Lp.N, Lp.K)
        q.qmm_quantize_weights(wt, w, Wq, Lp.N, Lp.K)
        del w
        Wp[Lp.name] = q.empty_packed(wt, Lp.N, Lp.K)
        q.qmm_repack_weights(wt, Wq, Wp[Lp.name], Lp.N, Lp.K)
        del Wq
        wbytes += Lp.N * (Lp.K // 256) * 144
        Y[Lp.name] = torch.empty(Lp.N, device=dev)
    torch.cuda.empty_cache()
    L = {Lp.name: Lp for Lp in wl.LAYER_70B}
    hot = wl.LAYER_70B_HOT_FRAC
    X = {name: wl.activations(100 + i, 1, L[name].K, hot_frac=hot, device=dev)
         for i, name in enumerate(L)}
    ws_bytes = q.qmm_workspace_bytes(wt, 1, L["down_proj"].K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def one(name, x):
        q.qmm_mul_mat_ws(wt, Wp[name], L[name].N, L[name].K, x, 1, Y[name], ws, ws_bytes, stream)

    def multi(names, x):
        q.qmm_mul_mat_multi(wt, [Wp[n] for n in names], [L[n].N for n in names], L[names[0]].K, x, 1,
                            [Y[n] for n in names], stream)

    def shared(i):
        multi(("q_proj", "k_proj", "v_proj"), X["q_proj"])
        one("o_proj", X["o_proj"])
        multi(("gate_proj", "up_proj"), X["gate_proj"])
        one("down_proj", X["down_proj"])

    def separate(i):
        for name in L:
            one(name, X[name])

    res = {"bytes": wbytes}
    for key, fn, launches in (("shared", shared, 4), ("separate", separate, 7)):
        for i in range(3):
            fn(i)
        g = capture(fn, graph_steps, stream)
        with torch.cuda.stream(stream):
            g.replay()
        t = timed(stream, lambda: run_graphs(g, None, reps)) / (reps * graph_steps)
        res[key] = {"us": round(t * 1e6, 2), "GB/s": round(wbytes / t / 1e9, 1),
                    "calls": launches}
    res["us"] = res["shared"]["us"]
    res["GB/s"] = res["shared"]["GB/s"]
    res["note"] = ("one step = the whole layer in a CUDA graph; 'shared': q/k/v and gate/up as "
                   "qmm_mul_mat_multi calls on one input each (one quantization, one launch); "
                   "'separate': seven qmm_mul_mat calls; GB/s counts weight bytes")
    del Wp, Y, X, ws
    return res


# ------------------------------------------------------------------ oracle (CPU)
def cpu_arm(target_s: float, steps: int | None = None, warmup: int = 0):
    """The oracle, as it stands, on the host cores: quantize the activations
    and run the fp32 vec_dot mul_mat over a sample of the weight rows."""
    import oracle
    L = wl.GEMV_Q4_K_4096
    N, K, M = L.N, L.K, 1
    nthreads = oracle.default_threads()
    rows_all = 512
    w = wl.weights(0, N, K, L.wstd, row_offset_std=L.row_offset_std,
                   rows=range(rows_all)).numpy()
    Wc = oracle.quantize(oracle.Q4_K, w, nthreads)
    x = wl.activations(0, M, K).numpy()
    row_b = (K // 256) * 144

    def one(nrows):
        oracle.mul_mat(oracle.Q4_K, Wc[:nrows], nrows, K, x, nthreads=nthreads, want=("y32",))

    one(rows_all)  # warm the thread pool
    t0 = time.perf_counter()
    one(rows_all)
    t_row = max((time.perf_counter() - t0) / rows_all, 1e-9)
    if steps is None:  # baseline leg: about target_s seconds of work
        nrows = rows_all
        reps = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < target_s:
            one(nrows)
            reps += 1
    else:              # reference arm: K steps fit the time budget
        nrows = int(min(rows_all, max(8, target_s / max(steps, 1) / t_row)))
        reps = steps
        for _ in range(warmup):
            one(nrows)
        t0 = time.perf_counter()
        for _ in range(reps):
            one(nrows)
    t = time.perf_counter() - t0
    b = nrows * row_b + (K // 256) * 292 + nrows * 4 + K * 4
    return {"value": round(b * reps / t / 1e9, 4), "unit": "GB/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{nrows} of {N} weight rows per call (M=1, K={K}), {reps} calls, "
                      f"{t:.1f} s; activation quantization included"}, t / reps


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--case", choices=["decode", "prefill", "w4a16", "layer", "sweep", "q6_K", "small_m",
                                       "peaks"],
                    default="decode",
                    help="prefill / w4a16 / layer / sweep / q6_K: only that measurement (for "
                         "profiler captures)")
    ap.add_argument("--m", type=int, action="append",
                    help="with --case sweep or w4a16: only these token counts")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    config = {"workload": WORKLOAD, "M": 1, "N": 4096, "K": 4096,
              "l2": f"{COPIES} rotating copies of the packed weights (302 MB > 129 MB L2)",
              "timing": f"CUDA events around CUDA-graph replays of {GRAPH_STEPS} steps"}

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 120.0
        res, per = cpu_arm(budget, steps=args.steps, warmup=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": res["value"], "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int8", "data": "synthetic", "config": config,
                "cpu_baseline": res,
                "e2e": {"value": res["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    if args.case != "decode":
        import block_quantized_matmul_q4_gb300 as q
        fn = {"prefill": prefill_extras, "w4a16": lambda q, d, s: w4a16_extras(q, d, s, ms=args.m),
              "layer": layer_rate, "q6_K": q6_K_rate,
              "small_m": small_m_rate, "peaks": peaks_rate,
              "sweep": lambda q, d, s: sweep_rate(q, d, s, args.m)}[args.case]
        print(json.dumps(fn(q, torch.device("cuda", torch.cuda.current_device()),
                            torch.cuda.Stream())), flush=True)
        return
    res = gpu_arm(args, rank, world)
    if rank == 0:
        cpu, _ = cpu_arm(args.cpu_seconds)
        line = {"metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "int8", "data": "synthetic", "config": config,
                "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
                "extras": res["extras"]}
        pf = res["extras"].get("prefill") if res["extras"] else None
        if pf:
            # the metric's TOPS half: the Q4_K prefill GEMM, 11008 x 4096, M = 512,
            # against the measured kind::f16 rate of the MMA form it issues
            # (A in TMEM, B in shared memory), and the int8 mma.sync rate
            r = pf["q4_K_up_11008x4096_M512"]
            tcf = pf["peaks_measured"]["tcgen05_f16_128x128x16_tmem_smem"]["TFLOP/s"]
            s8 = pf["peaks_measured"]["mma_sync_s8_m16n8k32"]["TFLOP/s"]
            line["roofline_prefill"] = {
                "bound": "tensor", "achieved": r["gemm_TOPS"], "peak": tcf, "unit": "TFLOP/s",
                "frac": round(r["gemm_TOPS"] / tcf, 4), "kernel": "gemm_f16_kernel<Q4_K>",
                "config": "Q4_K 11008x4096, M=512", "kernel_us": r["gemm_us"],
                "peak_source": "measured here (qmm_debug_peak, tcgen05 kind::f16 128x128x16, A in TMEM)",
                "frac_of_int8_mma_sync": round(r["gemm_TOPS"] / s8, 4),
                "frac_of_bf16_cublas": r["frac_of_fp16_peak"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
