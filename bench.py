#!/usr/bin/env python
"""Benchmark of the NVFP4 W4A4 MoE expert block on GB300.

One step = one pass of the whole hot path over one batch: top-k routing of the router
logits, then the expert-block forward (grouping, per-token NVFP4 quantisation gathered
to every routed slot, gate/up W4A4 grouped GEMM, SwiGLU + requantisation, down W4A4
grouped GEMM, weighted un-permute).  Weight quantisation is done once before timing
(it runs once per weight update).  Workload: the Qwen3-30B-A3B-shaped block, T = 16384
tokens, H = 2048, I = 768, E = 128 experts, top-8, Zipf(1.1) expert popularity.

Prints one JSON line (rank 0).  Multi-GPU: replicas only -- each rank runs the same
workload on its own GPU with no exchange (weak scaling), timing is the max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S  # noqa: E402

METRIC = "NVFP4 grouped-GEMM TFLOPS (% of 9 PF FP4) and MoE-layer tokens/s on 1 GB300"
UNIT = "tokens/s"
PF_TARGET = 9000.0          # TFLOP/s, the dense FP4 figure the target is quoted against
PF_B300 = 13500.0           # TFLOP/s, dense FP4 per GPU on the pages' B300 row
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio (6)
FLUSH_BYTES = 256 << 20     # > 129 MB L2


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gpu_selector(dev, local_rank):
    """nvidia-smi -i argument for this process's GPU (its UUID when torch reports one)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[local_rank].strip()
    return str(local_rank)


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
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
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def profiled_traffic(profile_md, source):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel source has not
    changed since (the summary stores the source hash next to the figure)."""
    if not os.path.exists(profile_md):
        return None, None
    txt = open(profile_md).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != kernel_source_sha(source):
        return None, txt
    return float(m.group(1)), txt


# --------------------------------------------------------------------------- timing helpers

def time_launches(fn, iters, flush, stream):
    """Average device time (ms) of fn() over iters launches, L2 flushed before each."""
    ts = []
    for _ in range(iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return float(np.mean(ts)), float(np.median(ts))


def capture_graph(fn):
    """fn()'s launches captured once in a CUDA graph (after a warm-up call on a side
    stream, as torch asks before a capture)."""
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_launches_median(fn, iters, flush, stream):
    """Median device time (ms) of fn() over iters launches, L2 flushed before each: the
    per-kernel figures (standalone quantisers, grouped GEMMs) are medians."""
    return time_launches(fn, iters, flush, stream)[1]


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (replicas run side by side; the job takes as long as its
    slowest rank).  One all-reduce on the process group's device (NCCL on GPUs, gloo on CPU)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time (weak scaling:
    each replica runs the full per-GPU workload)."""
    return world * tokens_per_rank * steps / (total_ms / 1e3)


def run_ours(args, rank, world, local_rank):
    import __graft_entry__ as G
    G.build()
    import nvfp4_w4a4_moe_quantize_gb300 as L
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = measured_peaks()

    shape = S.WORKLOADS["forward"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    x_h, logits_h, w13_h, w2_h = S.moe_inputs(shape, seed=0)
    x, logits = x_h.to(dev), logits_h.to(dev)
    t0 = time.time()
    pw = L.moe_prepare_weights(w13_h.to(dev), w2_h.to(dev))
    torch.cuda.synchronize()
    prep_s = time.time() - t0
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    wts = torch.empty(T, k, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = L.moe_forward_workspace(T, k, pw, dev)
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.zero_()

    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_clean():
        # the same write, then a read of the buffer: the flush's own dirty lines are written
        # back to HBM before the timed launch instead of inside it
        flush_buf.zero_()
        torch.sum(flush_buf, dim=0, out=flush_sink)

    def step():
        L.moe_route_topk(logits, k, True, out=(ids, wts))
        L.moe_expert_forward(x, ids, wts, pw, out=out, workspace=ws)

    for _ in range(max(args.warmup, 0)):
        flush()
        step()
    torch.cuda.synchronize()
    if L.nvfp4_status_check() != 0:
        raise RuntimeError("device status set during warm-up")

    sampler = ClockSampler(gpu_selector(dev, local_rank))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms = []
    t_wall = time.time()
    for _ in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()
        step_ms.append(a.elapsed_time(b))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall_s = time.time() - t_wall
    clocks = sampler.stop()
    total_ms = max_over_ranks(float(np.sum(step_ms)), world, dev)
    value = job_tokens_per_s(world, T, args.steps, total_ms)
    ms_per_step = total_ms / args.steps
    assert L.nvfp4_status_check() == 0

    # ---------------------------------------------------------------- stage timings
    lay = L.moe_forward_workspace_layout(T, k, E, H, I)
    mcap = lay[13]

    def view(i, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[lay[i]:lay[i] + nbytes].view(dtype)
    counts, padded = view(0, E, torch.int32), view(2, E + 1, torch.int32)
    inv = view(3, T * k, torch.int32).view(T, k)
    aq, ga = ws[lay[5]:lay[7]], view(7, mcap, torch.float32)
    hbuf = view(8, mcap * I, torch.bfloat16).view(mcap, I)
    hq, gh = ws[lay[9]:lay[11]], view(11, mcap, torch.float32)
    ybuf = view(12, mcap * H, torch.bfloat16).view(mcap, H)
    n_rows = T * k
    iters = max(10, min(50, args.steps))

    def gemm13():
        L.nvfp4_grouped_gemm_tiled(aq, ga, pw.w13, pw.w13_g, padded, counts, mcap, 2 * I, H, E,
                                   epilogue=L.EPILOGUE_SWIGLU, out=hbuf)

    def gemm2():
        L.nvfp4_grouped_gemm_tiled(hq, gh, pw.w2, pw.w2_g, padded, counts, mcap, H, pw.Ip, E, out=ybuf)

    def combine():
        L.load().moe_combine(L._p(ybuf), L._p(inv), L._p(wts), T, k, H, L._p(out), L._stream())

    def route():
        L.moe_route_topk(logits, k, True, out=(ids, wts))

    stages = {}
    for name, fn in (("route_topk", route), ("gateup_gemm_swiglu", gemm13), ("down_gemm", gemm2),
                     ("combine", combine)):
        stages[name] = time_launches(fn, iters, flush, stream)[0]
    stages["grouping_quantise_gather_requant"] = max(ms_per_step - sum(stages.values()), 0.0)
    torch.cuda.synchronize()

    # dominant kernel: the gate/up grouped GEMM with the SwiGLU epilogue
    t13 = stages["gateup_gemm_swiglu"] * 1e-3
    flops13 = 2.0 * n_rows * (2 * I) * H
    bytes13 = (n_rows * H / 2 * 1.125 + n_rows * 4 + E * 2 * I * H / 2 * 1.125 + n_rows * I * 2)
    tflops13 = flops13 / t13 / 1e12
    gbs13 = bytes13 / t13 / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    fp4_peak = float(peaks.get("bf16_tflops", 1900.0)) * FP4_OVER_BF16
    t_hbm = bytes13 / (hbm_peak * 1e9)
    t_tc = flops13 / (fp4_peak * 1e12)
    traffic, _ = profiled_traffic(os.path.join(ROOT, "profiles", "gateup_gemm_forward_T16384.md"),
                                  os.path.join(ROOT, "nvfp4_w4a4_moe_quantize_gb300", "csrc", "gemm_tiled.cu"))
    if t_hbm >= t_tc:
        roofline = {"bound": "hbm", "achieved": round(gbs13, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(gbs13 / hbm_peak, 4), "traffic": traffic}
    else:
        roofline = {"bound": "tensor", "achieved": round(tflops13, 1), "peak": round(fp4_peak, 1),
                    "unit": "TFLOP/s", "frac": round(tflops13 / fp4_peak, 4), "traffic": traffic}
    roofline.update({"kernel": "grouped_gemm_tiled_kernel<SwiGLU> (gate/up projection, forward workload)",
                     "peak_source": peak_src, "algorithmic_bytes": bytes13, "algorithmic_flops": flops13,
                     "launch_ms": round(t13 * 1e3, 4), "tflops": round(tflops13, 1),
                     "frac_of_9pf": round(tflops13 / PF_TARGET, 4)})

    # ---------------------------------------------------------------- grouped-GEMM workload
    gshape = S.WORKLOADS["gateup"]
    gx = S.randn_bf16((gshape.T, H), 1.0, 1).to(dev)
    glog = S.router_logits_zipf(gshape.T, E, gshape.zipf_s, 2).to(dev)
    gids, gw = L.moe_route_topk(glog, k)
    gws = L.moe_forward_workspace(gshape.T, k, pw, dev)
    L.moe_expert_forward(gx, gids, gw, pw, workspace=gws)
    glay = L.moe_forward_workspace_layout(gshape.T, k, E, H, I)
    gm = glay[13]
    gview = lambda i, n, dt: gws[glay[i]:glay[i] + n * torch.empty((), dtype=dt).element_size()].view(dt)  # noqa: E731
    g_aq, g_ga = gws[glay[5]:glay[7]], gview(7, gm, torch.float32)
    g_cnt, g_pad = gview(0, E, torch.int32), gview(2, E + 1, torch.int32)
    g_d = torch.empty(gm, 2 * I, dtype=torch.bfloat16, device=dev)
    gt = time_launches_median(lambda: L.nvfp4_grouped_gemm_tiled(g_aq, g_ga, pw.w13, pw.w13_g, g_pad, g_cnt, gm, 2 * I,
                                                             H, E, out=g_d), iters, flush, stream)
    gflops = 2.0 * gshape.T * k * 2 * I * H
    gemm_tflops = gflops / (gt * 1e-3) / 1e12
    tiles = int(g_pad[-1].item()) // 128
    grouped = {"timing": f"median of {iters} launches, L2 flushed before each",
               "workload": "gate/up grouped GEMM, T=8192 top-8 of 128 experts (65,536 routed rows, Zipf 1.1), "
                           "K=2048, N=1536, BF16 out", "ms": round(gt, 4), "tflops": round(gemm_tflops, 1),
               "frac_of_9pf": round(gemm_tflops / PF_TARGET, 4), "frac_of_13_5pf": round(gemm_tflops / PF_B300, 4),
               "frac_of_fp4_peak_from_measured_bf16": round(gemm_tflops / fp4_peak, 4), "row_tiles": tiles}
    del gws, g_d

    # ---------------------------------------------------------------- quantiser workload
    qx = S.outlier_channels_bf16(*S.QUANTISER_SHAPE, seed=0).to(dev)
    qrows, qcols = S.QUANTISER_SHAPE
    qcodes = torch.empty(qrows, qcols // 2, dtype=torch.uint8, device=dev)
    qsf = torch.empty(L.nvfp4_sf_bytes(qrows, qcols), dtype=torch.uint8, device=dev)
    qg = torch.empty(1, dtype=torch.float32, device=dev)
    qws = torch.empty(4096, dtype=torch.uint8, device=dev)
    qbytes = qrows * qcols * 2 + qrows * qcols // 2 + L.nvfp4_sf_bytes(qrows, qcols)
    quant = {"timing": f"median of {iters} launches, L2 flushed before each",
             "workload": "standalone quantiser 16384x2048 BF16, 1% outlier channels x50, per-tensor scale",
             "algorithmic_bytes": qbytes, "bytes_note": "one read of x + codes + scales (the amax pass re-reads x)"}
    for rnd, name in ((L.ROUND_RNE, "rne"), (L.ROUND_STOCHASTIC, "sr")):
        qt = time_launches_median(lambda: L.nvfp4_quantize(qx, L.SCALE_PER_TENSOR, rnd, 0, 0, out=(qcodes, qsf, qg),
                                                       workspace=qws), iters, flush, stream)
        quant[f"{name}_us"] = round(qt * 1e3, 2)
        quant[f"{name}_gbs"] = round(qbytes / (qt * 1e-3) / 1e9, 1)
        quant[f"{name}_frac_hbm"] = round(qbytes / (qt * 1e-3) / 1e9 / hbm_peak, 4)
    qt_row = time_launches_median(lambda: L.nvfp4_quantize(qx, L.SCALE_PER_ROW, L.ROUND_RNE, 0, 0, out=(qcodes, qsf,
                              torch.empty(qrows, dtype=torch.float32, device=dev)), workspace=qws), iters, flush, stream)
    quant["per_row_rne_gbs"] = round(qbytes / (qt_row * 1e-3) / 1e9, 1)
    quant["per_row_rne_frac_hbm"] = round(qbytes / (qt_row * 1e-3) / 1e9 / hbm_peak, 4)

    # ---------------------------------------------------------------- MXFP8 recipe variant
    # The validation format: E4M3 elements, E8M0 scales per 32 values.  Quantiser and DQ
    # on the standalone quantiser's matrix; the grouped GEMM on the gate/up workload's
    # groups (the same 65,536 routed rows, K=2048, N=1536), operands quantised by
    # mxfp8_quantize from the same random BF16 weights.
    mcodes = torch.empty(qrows, qcols, dtype=torch.uint8, device=dev)
    msf = torch.empty(L.mxfp8_sf_bytes(qrows, qcols), dtype=torch.uint8, device=dev)
    mbytes = qrows * qcols * 2 + qrows * qcols + L.mxfp8_sf_bytes(qrows, qcols)
    mq = time_launches_median(lambda: L.mxfp8_quantize(qx, mcodes, msf), iters, flush, stream)
    mdq_out = torch.empty(qrows, qcols, dtype=torch.bfloat16, device=dev)
    mdq = time_launches_median(lambda: L.mxfp8_dequantize(mcodes, msf, out=mdq_out), iters, flush, stream)
    ma_bf16 = S.randn_bf16((gm, H), 1.0, 3).to(dev)
    ma, msfa = L.mxfp8_quantize(ma_bf16)
    mb, msfb = L.mxfp8_quantize(w13_h.to(dev).reshape(E * 2 * I, H))
    mg_d = torch.empty(gm, 2 * I, dtype=torch.bfloat16, device=dev)
    mgt = time_launches_median(lambda: L.mxfp8_grouped_gemm(ma, msfa, mb, msfb, g_pad, g_cnt, 2 * I, H, E, out=mg_d),
                           iters, flush, stream)
    fp8_peak = float(peaks.get("bf16_tflops", 1900.0)) * 2.0      # nominal FP8 : BF16 ratio 2
    mx_tflops = gflops / (mgt * 1e-3) / 1e12
    mxfp8 = {"timing": f"median of {iters} launches, L2 flushed before each",
             "quantiser": {"workload": "16384x2048 BF16 (the standalone quantiser's matrix)",
                           "algorithmic_bytes": mbytes, "us": round(mq * 1e3, 2),
                           "gbs": round(mbytes / (mq * 1e-3) / 1e9, 1),
                           "frac_hbm": round(mbytes / (mq * 1e-3) / 1e9 / hbm_peak, 4)},
             "dequantize_bf16": {"algorithmic_bytes": qrows * qcols * 3 + L.mxfp8_sf_bytes(qrows, qcols),
                                 "us": round(mdq * 1e3, 2),
                                 "gbs": round((qrows * qcols * 3 + L.mxfp8_sf_bytes(qrows, qcols)) / (mdq * 1e-3) / 1e9,
                                              1)},
             "grouped_gemm": {"workload": "MXFP8 x MXFP8 grouped GEMM on the gate/up groups (65,536 routed rows), "
                                          "K=2048, N=1536, BF16 out", "ms": round(mgt, 4),
                              "tflops": round(mx_tflops, 1), "frac_of_4_5pf": round(mx_tflops / 4500.0, 4),
                              "frac_of_fp8_peak_from_measured_bf16": round(mx_tflops / fp8_peak, 4)}}
    del ma_bf16, ma, msfa, mb, msfb, mg_d, mdq_out, mcodes, msf

    # ---------------------------------------------------------------- dequantised backward
    # The recipe's backward GEMM on the dequantised weights: dgrad of the gate/up
    # projection, dX = dGU . DQ(W13), over the gate/up groups (65,536 routed rows): DQ of
    # all 128 experts' W13 to BF16 (from a per-expert NVFP4 quantisation), transposed to
    # [E, H, 2I], then the BF16 grouped GEMM (N = H = 2048, K = 2I = 1536).
    w13_dev = w13_h.to(dev).reshape(E * 2 * I, H)
    wc, wsf, wg = L.nvfp4_quantize(w13_dev, L.SCALE_PER_GROUP, group_rows=2 * I)
    del w13_dev
    wdq = torch.empty(E * 2 * I, H, dtype=torch.bfloat16, device=dev)
    dq_t = time_launches_median(lambda: L.nvfp4_dequantize(wc, wsf, wg, H, L.SCALE_PER_GROUP, group_rows=2 * I,
                                                           out=wdq), iters, flush, stream)
    wdqt = L.bf16_transpose(wdq, batches=E)
    del wdq, wc, wsf
    dgu = S.randn_bf16((gm, 2 * I), 1e-3, 5).to(dev)
    dx = torch.empty(gm, H, dtype=torch.bfloat16, device=dev)
    bt = time_launches_median(lambda: L.bf16_grouped_gemm(dgu, wdqt, g_pad, g_cnt, H, 2 * I, E, out=dx),
                              iters, flush, stream)
    bf16_tflops = gflops / (bt * 1e-3) / 1e12
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    dq_bytes = E * 2 * I * H // 2 + L.nvfp4_sf_bytes(E * 2 * I, H) + E * 2 * I * H * 2
    dqbwd = {"timing": f"median of {iters} launches, L2 flushed before each",
             "dequantize_w13": {"workload": "DQ of W13, 128 experts x 1536 x 2048, NVFP4 -> BF16",
                                "algorithmic_bytes": dq_bytes, "us": round(dq_t * 1e3, 2),
                                "gbs": round(dq_bytes / (dq_t * 1e-3) / 1e9, 1),
                                "frac_hbm": round(dq_bytes / (dq_t * 1e-3) / 1e9 / hbm_peak, 4)},
             "bf16_grouped_gemm": {"workload": "dgrad of the gate/up projection on the gate/up groups "
                                               "(65,536 routed rows), N=2048, K=1536, BF16 x BF16, BF16 out",
                                   "ms": round(bt, 4), "tflops": round(bf16_tflops, 1),
                                   "frac_of_measured_bf16": round(bf16_tflops / bf16_peak, 4)}}
    del wdqt, dgu, dx

    # ---------------------------------------------------------------- learner step (forward + W4A4 backward)
    # The learner-step expert GEMMs: T=32768 tokens, uniform routing (i.i.d. N(0,1) logits),
    # top-8 of 128 experts, dOut ~ N(0, 1e-3): routing + forward + the W4A4 backward (dgrad
    # and wgrad of both projections, stochastic rounding on gradients).  Algorithmic work:
    # 3 x the forward's 2 * T*k * (2I*H + H*I) flops (the backward's recomputation of the
    # gate/up output is not counted).
    lshape = S.WORKLOADS["learner"]
    lx_h, llog_h, _, _ = S.moe_inputs(lshape, seed=0)
    lx, llog = lx_h.to(dev), llog_h.to(dev)
    ldout = S.randn_bf16((lshape.T, H), 1e-3, 9).to(dev)
    pt = L.moe_prepare_weights_backward(w13_h.to(dev), w2_h.to(dev))
    lids = torch.empty(lshape.T, k, dtype=torch.int32, device=dev)
    lwts = torch.empty(lshape.T, k, dtype=torch.float32, device=dev)
    lout = torch.empty(lshape.T, H, dtype=torch.bfloat16, device=dev)
    lfws = L.moe_forward_workspace(lshape.T, k, pw, dev)
    lbws = L.moe_backward_workspace(lshape.T, k, pw, dev)
    lgrads = (torch.empty(lshape.T, H, dtype=torch.bfloat16, device=dev),
              torch.empty(lshape.T, k, dtype=torch.float32, device=dev),
              torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev),
              torch.empty(E, H, I, dtype=torch.float32, device=dev))

    def learner_fwd():
        L.moe_route_topk(llog, k, True, out=(lids, lwts))
        L.moe_expert_forward(lx, lids, lwts, pw, out=lout, workspace=lfws)

    def learner_bwd():
        L.moe_expert_backward(ldout, lx, lwts, pw, pt, lfws, seed=7, out=lgrads, workspace=lbws)

    def learner_step():
        learner_fwd()
        learner_bwd()

    l_iters = 5
    lt = time_launches_median(learner_step, l_iters, flush, stream)
    lf = time_launches_median(learner_fwd, l_iters, flush, stream)
    learner_fwd()
    lb = time_launches_median(learner_bwd, l_iters, flush, stream)
    assert L.nvfp4_status_check() == 0
    l_fwd_flops = 2.0 * lshape.T * k * (2 * I * H + H * I)
    l_tflops = 3 * l_fwd_flops / (lt * 1e-3) / 1e12
    learner = {"timing": f"median of {l_iters} launches, L2 flushed before each",
               "workload": "learner step: T=32768, hidden 2048, intermediate 768, 128 experts, top-8, uniform "
                           "routing; routing + W4A4 forward + W4A4 backward (dgrad and wgrad, SR on gradients)",
               "algorithmic_tflop": round(3 * l_fwd_flops / 1e12, 3), "ms": round(lt, 4),
               "fwd_ms": round(lf, 4), "bwd_ms": round(lb, 4), "tflops": round(l_tflops, 1),
               "frac_of_9pf": round(l_tflops / PF_TARGET, 4), "tokens_per_s": round(lshape.T / (lt * 1e-3), 1)}
    del lfws, lbws, lgrads, pt, lx, llog, ldout, lout

    # ---------------------------------------------------------------- decode-shaped launches
    # Sampler-shaped batches of 1, 8 and 64 tokens through the same calls (routing + the
    # expert block) on the forward workload's weights: the tiles cover only the experts the
    # batch routes to, so the floor is reading those experts' weights once.
    decode = {"timing": f"median of {iters} launches, L2 flushed before each",
              "us_clean_l2": "the same launches after a flush whose 256 MB write is followed by a 256 MB read, "
                             "so that the flush's dirty lines are not written back inside the timed launch",
              "us_graph": "the same launches captured once in a CUDA graph and replayed (the flush, a write, "
                          "outside the graph before each replay)",
              "batches": []}
    w13_e = L.nvfp4_tiled_bytes(2 * I, H, 256) + 4
    w2_e = L.nvfp4_tiled_bytes(H, pw.Ip, 256) + 4
    for dt in (1, 8, 64):
        dx_ = x[:dt].contiguous()
        dlog = logits[:dt].contiguous()
        dids = torch.empty(dt, k, dtype=torch.int32, device=dev)
        dwts = torch.empty(dt, k, dtype=torch.float32, device=dev)
        dout_ = torch.empty(dt, H, dtype=torch.bfloat16, device=dev)
        dws = L.moe_forward_workspace(dt, k, pw, dev)

        def dstep():
            L.moe_route_topk(dlog, k, True, out=(dids, dwts))
            L.moe_expert_forward(dx_, dids, dwts, pw, out=dout_, workspace=dws)
        dtime = time_launches_median(dstep, iters, flush, stream)
        dtime_clean = time_launches_median(dstep, iters, flush_clean, stream)
        dgraph = capture_graph(dstep)
        dtime_graph = time_launches_median(dgraph.replay, iters, flush, stream)
        del dgraph
        active = int(torch.unique(dids).numel())
        dbytes = active * (w13_e + w2_e) + dt * H * 2 * 2 + dt * E * 4
        decode["batches"].append({"tokens": dt, "active_experts": active, "us": round(dtime * 1e3, 2),
                                  "us_clean_l2": round(dtime_clean * 1e3, 2),
                                  "us_graph": round(dtime_graph * 1e3, 2),
                                  "tokens_per_s": round(dt / (dtime * 1e-3), 1),
                                  "weight_bytes_read": active * (w13_e + w2_e),
                                  "gbs": round(dbytes / (dtime * 1e-3) / 1e9, 1),
                                  "frac_hbm": round(dbytes / (dtime * 1e-3) / 1e9 / hbm_peak, 4)})
        del dws

    # ---------------------------------------------------------------- end to end (host buffers)
    # Every step copies its inputs (x, router logits) from pinned host memory and reads its
    # result back.  Serial: copy in, compute, copy out on one stream.  Pipelined (the
    # reported number): the copy-in of step i+1 and the copy-out of step i-1 run on their
    # own streams while step i computes (double-buffered device inputs and outputs); the
    # timed region runs from the first copy-in to the last copy-out, and the L2 flush stays
    # inside it, on the compute stream before every step.
    x_pin = x_h.pin_memory()
    l_pin = logits_h.pin_memory()
    o_pin = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_e = [torch.empty_like(x) for _ in range(2)]
    l_e = [torch.empty_like(logits) for _ in range(2)]
    out2 = [out, torch.empty_like(out)]
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x_e[0].copy_(x_pin, non_blocking=True)
        l_e[0].copy_(l_pin, non_blocking=True)
        L.moe_route_topk(l_e[0], k, True, out=(ids, wts))
        L.moe_expert_forward(x_e[0], ids, wts, pw, out=out, workspace=ws)
        o_pin[0].copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if it >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e_serial_total = max_over_ranks(float(np.sum(e2e_ms)), world, dev)

    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def pipelined(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_start.record(s_in)
        for i in range(n):
            bi = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])       # step i-2 has read this input buffer
                x_e[bi].copy_(x_pin, non_blocking=True)
                l_e[bi].copy_(l_pin, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])      # step i-2's result has left this buffer
                flush()                                   # L2 flushed before every step, as above
                L.moe_route_topk(l_e[bi], k, True, out=(ids, wts))
                L.moe_expert_forward(x_e[bi], ids, wts, pw, out=out2[bi], workspace=ws)
                ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                o_pin[bi].copy_(out2[bi], non_blocking=True)
                ev_out[i].record(s_out)
        t_end.record(s_out)
        t_end.synchronize()
        return t_start.elapsed_time(t_end)

    pipelined(args.warmup)
    e2e_total = max_over_ranks(pipelined(args.steps), world, dev)
    e2e = {"value": round(job_tokens_per_s(world, T, args.steps, e2e_total), 1), "unit": UNIT,
           "mode": "pipelined: copy-in of step i+1 and copy-out of step i-1 overlap step i's compute",
           "serial_value": round(job_tokens_per_s(world, T, args.steps, e2e_serial_total), 1),
           "h2d_bytes_per_step": x_h.numel() * 2 + logits_h.numel() * 4, "d2h_bytes_per_step": T * H * 2}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(budget_s=args.cpu_seconds)

    launches_per_step = 1 + 9      # route + (3 grouping, token quantise, slot gather, gate/up+SwiGLU GEMM, requant, down GEMM, combine)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3 operands, f32 accumulate)",
        "data": "synthetic",
        "config": {"workload": "MoE expert-block forward, Qwen3-30B-A3B-shaped: T=16384 tokens, hidden 2048, "
                               "intermediate 768, 128 experts, top-8, Zipf(1.1) routing",
                   "tokens_per_gpu": T, "routed_rows": T * k, "l2": "flushed before every step (256 MB write)",
                   "weights": "quantised once before timing (offline per weight update)",
                   "weight_prep_s": round(prep_s, 3), "parallelism": "replicas" if world > 1 else "single"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps, "stages_ms": {k_: round(v_, 4) for k_, v_ in stages.items()},
        "grouped_gemm": grouped, "quantiser": quant, "mxfp8": mxfp8, "dequantised_backward": dqbwd,
        "learner_step": learner, "decode": decode,
        "wall_s_timed": round(wall_s, 3),
    }
    return line


def _cpu_worker_run(kind: str, seconds: float, index: int, workers: int) -> dict:
    """One oracle timing worker (run as its own process): the oracle as it stands, on a
    bounded share of one workload -- `index` of `workers` interleaved shares.  Expert
    weights are drawn per expert from the workloads' distribution (N(0, 0.02) BF16, one
    seed per expert), so a worker builds only the experts it touches.  Setup (inputs,
    weight quantisation) is not timed."""
    from oracle import moe as M
    from oracle import quant as Q
    shape = S.WORKLOADS["forward"]
    H, I, E, k = shape.H, shape.I, shape.E, shape.k
    w13_of = lambda e: S.bf16_bits(S.randn_bf16((2 * I, H), shape.w_std, 50_000 + e))  # noqa: E731
    w2_of = lambda e: S.bf16_bits(S.randn_bf16((H, I), shape.w_std, 60_000 + e))       # noqa: E731
    done, el = 0, 0.0
    if kind == "quantiser":
        rows, cols = S.QUANTISER_SHAPE
        bits = S.bf16_bits(S.outlier_channels_bf16(rows, cols, seed=0))
        g = Q.global_scale(np.array([np.max(np.abs(F_bf16(bits)))]))
        chunk, r = 32, index * 32
        t0 = time.perf_counter()
        while r < rows and time.perf_counter() - t0 < seconds:
            Q.quantize(bits[r:r + chunk], scope="tensor", global_scale_in=g)
            done += chunk
            r += chunk * workers
        el = time.perf_counter() - t0
        per_row = cols * 2 + cols // 2 + cols // 16
        return {"kind": kind, "rate": done * per_row / el / 1e9, "unit": "GB/s", "units": done, "seconds": el}
    if kind == "gemm":
        g_shape = S.WORKLOADS["gateup"]
        x = S.bf16_bits(S.randn_bf16((g_shape.T, H), 1.0, 1))
        ids, _ = M.route_topk(S.router_logits_zipf(g_shape.T, E, g_shape.zipf_s, 2).numpy(), k)
        counts = np.bincount(ids.reshape(-1), minlength=E)
        order = [e for e in np.argsort(-counts, kind="stable") if counts[e] > 0][index::workers]
        flops = 0.0
        for e in order:
            toks = np.nonzero((ids == e).any(axis=1))[0]
            qa = Q.quantize(x[toks], scope="row")
            qw = Q.quantize(w13_of(int(e)), scope="tensor")
            t0 = time.perf_counter()
            M.gemm_rows(qa["codes"], qa["sf"], qa["g"], qw["codes"], qw["sf"], qw["g"][0])
            el += time.perf_counter() - t0
            flops += 2.0 * len(toks) * 2 * I * H
            done += len(toks)
            if el > seconds:
                break
        return {"kind": kind, "rate": flops / max(el, 1e-9) / 1e12, "unit": "TFLOP/s", "units": done, "seconds": el}
    # the expert-block forward, token by token
    x = S.bf16_bits(S.randn_bf16((shape.T, H), 1.0, 1))
    ids, w = M.route_topk(S.router_logits_zipf(shape.T, E, shape.zipf_s, 2).numpy(), k)
    toks = list(range(index, shape.T, workers))[:4]
    prep = {"w13_codes": {}, "w13_sf": {}, "w13_g": {}, "w2_codes": {}, "w2_sf": {}, "w2_g": {}}
    for e in sorted(set(ids[toks].reshape(-1).tolist())):
        q13, q2 = Q.quantize(w13_of(e), scope="tensor"), Q.quantize(w2_of(e), scope="tensor")
        prep["w13_codes"][e], prep["w13_sf"][e], prep["w13_g"][e] = q13["codes"], q13["sf"], q13["g"][0]
        prep["w2_codes"][e], prep["w2_sf"][e], prep["w2_g"][e] = q2["codes"], q2["sf"], q2["g"][0]
    t0 = time.perf_counter()
    for t in toks:
        M.moe_forward_tokens(x, ids, w, prep, [t])
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    el = time.perf_counter() - t0
    return {"kind": kind, "rate": done / el, "unit": UNIT, "units": done, "seconds": el}


def F_bf16(bits):
    """BF16 bit patterns -> float32 (numpy), for the oracle workers' global scale."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _cpu_workers(kind: str, seconds: float, workers: int) -> list:
    """`workers` single-threaded oracle workers side by side (own processes, BLAS and
    OpenMP limited to one thread each); their reports."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs = [subprocess.Popen([sys.executable, os.path.abspath(__file__), "--cpu-worker", kind, "--cpu-seconds",
                               str(seconds), "--worker-index", str(i), "--workers", str(workers)],
                              stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, env=env, text=True)
             for i in range(workers)]
    out = []
    for p in procs:
        so, _ = p.communicate(timeout=600)
        if p.returncode == 0 and so.strip():
            out.append(json.loads(so.strip().splitlines()[-1]))
    return out


def cpu_baseline(budget_s: float = 4.0) -> dict:
    """The oracle (float64 numpy, as it stands) timed on this host on bounded shares of the
    three measured workloads, on 1 thread and on all cores (one single-threaded worker per
    core, interleaved shares; the rates add up).  The headline value is the expert-block
    forward on all cores, in the metric's unit."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    res = {}
    for kind, name in (("forward", "forward_tokens_per_s"), ("gemm", "grouped_gemm_tflops"),
                       ("quantiser", "quantiser_gbs")):
        one = _cpu_workers(kind, budget_s, 1)
        many = _cpu_workers(kind, budget_s, cores)
        res[name] = {"1_thread": round(one[0]["rate"], 6) if one else None,
                     "all_cores": round(sum(r["rate"] for r in many), 6) if many else None,
                     "units_timed_all_cores": int(sum(r["units"] for r in many))}
    fwd = res["forward_tokens_per_s"]
    return {"value": fwd["all_cores"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the oracle (float64 numpy) on bounded interleaved shares of each workload, ~{budget_s:.0f} s "
                      "per worker: the T=16384 forward token by token (up to 4 tokens per worker), the T=8192 "
                      "gate/up grouped GEMM expert by expert, the 16384x2048 quantiser 32 rows at a time; "
                      f"1 thread, and {cores} single-threaded workers side by side (all cores); expert weights "
                      "drawn per expert from the workloads' distribution",
            "configs": res}


def run_profile(args):
    """A short launch sequence on a small case, for ncu captures: the gate/up grouped GEMM
    of a forward over --tokens tokens (Zipf routing, Qwen3 shapes), whole forward steps
    (routing + expert block) over --tokens tokens, the standalone quantiser on a
    --tokens x 2048 tensor, or the MXFP8 grouped GEMM over the routed groups of --tokens
    tokens.  Prints nothing else."""
    import __graft_entry__ as G
    G.build()
    import nvfp4_w4a4_moe_quantize_gb300 as L
    dev = torch.device("cuda", 0)
    shape = S.WORKLOADS["forward"]
    T, H, I, E, k = args.tokens, shape.H, shape.I, shape.E, shape.k
    if args.profile == "quantiser":
        qx = S.outlier_channels_bf16(T, H, seed=0).to(dev)
        mode = {"tensor": L.SCALE_PER_TENSOR, "row": L.SCALE_PER_ROW}[args.quant_scope]
        rnd = L.ROUND_STOCHASTIC if args.quant_sr else L.ROUND_RNE
        for _ in range(args.steps):
            L.nvfp4_quantize(qx, mode, rnd)
        torch.cuda.synchronize()
        return
    if args.profile == "backward":     # forward + W4A4 backward over --tokens tokens (uniform routing)
        bx = S.randn_bf16((T, H), 1.0, 1).to(dev)
        blog = S.router_logits_normal(T, E, 2).to(dev)
        bw13 = S.randn_bf16((E, 2 * I, H), 0.02, 3).to(dev)
        bw2 = S.randn_bf16((E, H, I), 0.02, 4).to(dev)
        bpw = L.moe_prepare_weights(bw13, bw2)
        bpt = L.moe_prepare_weights_backward(bw13, bw2)
        del bw13, bw2
        bids, bwts = L.moe_route_topk(blog, k)
        bfws = L.moe_forward_workspace(T, k, bpw, dev)
        bbws = L.moe_backward_workspace(T, k, bpw, dev)
        bdout = S.randn_bf16((T, H), 1e-3, 9).to(dev)
        for _ in range(args.steps):
            L.moe_expert_forward(bx, bids, bwts, bpw, workspace=bfws)
            L.moe_expert_backward(bdout, bx, bwts, bpw, bpt, bfws, seed=7, workspace=bbws)
        torch.cuda.synchronize()
        assert L.nvfp4_status_check() == 0
        return
    if args.profile == "mxgemm":       # MXFP8 grouped GEMM on the routed groups of --tokens tokens
        glog = S.router_logits_zipf(T, E, shape.zipf_s, 2).to(dev)
        gids, _ = L.moe_route_topk(glog, k)
        grp = L.moe_permute(gids, E)
        counts, padded = grp["counts"], grp["padded_offsets"]
        m = int(padded[-1].item())
        a, sfa = L.mxfp8_quantize(S.randn_bf16((max(m, 128), H), 1.0, 3).to(dev))
        b, sfb = L.mxfp8_quantize(S.randn_bf16((E * 2 * I, H), 0.02, 4).to(dev))
        d = torch.empty(max(m, 128), 2 * I, dtype=torch.bfloat16, device=dev)
        for _ in range(args.steps):
            L.mxfp8_grouped_gemm(a, sfa, b, sfb, padded, counts, 2 * I, H, E, out=d)
        torch.cuda.synchronize()
        assert L.nvfp4_status_check() == 0
        return
    x = S.randn_bf16((T, H), 1.0, 1).to(dev)
    logits = S.router_logits_zipf(T, E, shape.zipf_s, 2).to(dev)
    w13 = S.randn_bf16((E, 2 * I, H), 0.02, 3).to(dev)
    w2 = S.randn_bf16((E, H, I), 0.02, 4).to(dev)
    pw = L.moe_prepare_weights(w13, w2)
    del w13, w2
    ids, w = L.moe_route_topk(logits, k)
    ws = L.moe_forward_workspace(T, k, pw, dev)
    L.moe_expert_forward(x, ids, w, pw, workspace=ws)
    if args.profile == "forward":      # whole forward steps: routing + the expert block
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        for _ in range(args.steps):
            L.moe_route_topk(logits, k, True, out=(ids, w))
            L.moe_expert_forward(x, ids, w, pw, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert L.nvfp4_status_check() == 0
        return
    lay = L.moe_forward_workspace_layout(T, k, E, H, I)
    m = lay[13]
    vw = lambda i, n, dt: ws[lay[i]:lay[i] + n * torch.empty((), dtype=dt).element_size()].view(dt)  # noqa: E731
    h = vw(8, m * I, torch.bfloat16).view(m, I)
    for _ in range(args.steps):
        L.nvfp4_grouped_gemm_tiled(ws[lay[5]:lay[7]], vw(7, m, torch.float32), pw.w13, pw.w13_g,
                                   vw(2, E + 1, torch.int32), vw(0, E, torch.int32), m, 2 * I, H, E,
                                   epilogue=L.EPILOGUE_SWIGLU, out=h)
    torch.cuda.synchronize()
    assert L.nvfp4_status_check() == 0


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step runs it on a bounded sample of the
    same workload (a few tokens), on the host cores; rank 0 only."""
    if rank != 0:
        return None
    shape = S.WORKLOADS["forward"]
    x_h, logits_h, w13_h, w2_h = S.moe_inputs(shape, seed=0)
    from oracle import moe as M
    from oracle import quant as Q
    xb = S.bf16_bits(x_h)
    ids, w = M.route_topk(logits_h.numpy(), shape.k)
    per_step = max(1, args.ref_tokens_per_step)
    n_tok = per_step * (args.warmup + args.steps)
    need = sorted(set(ids[:n_tok].reshape(-1).tolist()))
    w13b, w2b = S.bf16_bits(w13_h), S.bf16_bits(w2_h)
    prep = {"w13_codes": {}, "w13_sf": {}, "w13_g": {}, "w2_codes": {}, "w2_sf": {}, "w2_g": {}}
    for e in need:
        q13 = Q.quantize(w13b[e], scope="tensor")
        q2 = Q.quantize(w2b[e], scope="tensor")
        prep["w13_codes"][e], prep["w13_sf"][e], prep["w13_g"][e] = q13["codes"], q13["sf"], q13["g"][0]
        prep["w2_codes"][e], prep["w2_sf"][e], prep["w2_g"][e] = q2["codes"], q2["sf"], q2["g"][0]
    times = []
    t = 0
    for it in range(args.warmup + args.steps):
        toks = list(range(t, t + per_step))
        t += per_step
        t0 = time.perf_counter()
        M.moe_forward_tokens(xb, ids, w, prep, toks)
        if it >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = float(np.sum(times))
    value = per_step * args.steps / total
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = f"{per_step} token(s) per step of the T=16384 forward workload, token by token (float64 numpy)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "MoE expert-block forward, Qwen3-30B-A3B-shaped: T=16384 tokens, hidden 2048, "
                                   "intermediate 768, 128 experts, top-8, Zipf(1.1) routing",
                       "tokens_per_step": per_step},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=4.0, help="time budget of each oracle timing worker")
    ap.add_argument("--cpu-worker", choices=["forward", "gemm", "quantiser"], default=None,
                    help="(internal) run one oracle timing worker and print its report")
    ap.add_argument("--worker-index", type=int, default=0)
    ap.add_argument("--workers", type=int, default=1)
    ap.add_argument("--ref-tokens-per-step", type=int, default=2)
    ap.add_argument("--profile", choices=["none", "gateup", "quantiser", "forward", "mxgemm", "backward"],
                    default="none",
                    help="run only a short launch sequence of one kernel (for ncu captures)")
    ap.add_argument("--tokens", type=int, default=2048, help="tokens (rows) of the --profile case")
    ap.add_argument("--quant-scope", choices=["tensor", "row"], default="tensor",
                    help="scale scope of the --profile quantiser case")
    ap.add_argument("--quant-sr", action="store_true", help="stochastic rounding in the --profile quantiser case")
    args = ap.parse_args()
    if args.cpu_worker is not None:
        print(json.dumps(_cpu_worker_run(args.cpu_worker, args.cpu_seconds, args.worker_index, args.workers)))
        return
    if args.profile != "none":
        run_profile(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", 1)
    local_rank = _env_int("LOCAL_RANK", 0)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
