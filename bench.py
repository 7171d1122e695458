#!/usr/bin/env python3
"""Benchmark of the Q8_0 x q8_1 hot path on GB300.

One step = one pass of the whole hot path on the headline workload:
  1. the prefill GEMM, m = 512, 4096 -> 4096, q8_1 quantization fused in the call
  2. the same GEMM on the load-time repacked weights (exact binary16 quants + f32 scales)
  3. the Q8_0 -> fp16 dequant of the same 4096 x 4096 weights
  4. q8_1 quantization of one decode token (k = 4096)
  5. the decode GEMV, m = 1, 4096 -> 64448 (the LM-head half; 280.5 MB of Q8_0 weights)
L2 is flushed outside the timed kernels before each GEMM and the dequant (a 256 MiB write,
then a 256 MiB read of another buffer, so that the flush's own dirty lines are written back
before the timed kernel starts); the GEMV's weight stream (280.5 MB) is larger than L2,
needs no flush, and evicts the next step's quantizer input.

`value` is the decode GEMV's weight-stream throughput in GB/s (algorithmic bytes: weights
+ activation + scales + output); the GEMM's TOPS (2*m*n*k / t) and every kernel's roofline
fraction are reported alongside.  Usage:

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica of the workload (weak scaling:
the path has no exchange step); rank 0 prints the JSON line with max-over-ranks times.
`--impl reference` times the CPU oracle (the plain C restatement of the method) on the
same metric, on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "Q8_0 GEMV GB/s (m=1); Q8_0 MMQ GEMM TOPS (m=512); % of roofline"
GEMV = dict(m=1, n=64448, k=4096)
GEMM = dict(m=512, n=4096, k=4096)
DEQ = dict(n=4096, k=4096)
VERIFY_M = 8   # the verify tier's token count (7 drafted + 1)
WORKLOAD = ("decode GEMV m=1 4096->64448 (q8_1 quantize + mmvq) + prefill GEMM m=512 "
            "4096->4096 (q8_1 quantize fused; on raw Q8_0 and on the load-time repack) + "
            "Q8_0->fp16 dequant 4096x4096")
FLUSH_BYTES = 256 << 20


def row_bytes(k):
    return k // 32 * 34


def gemv_bytes(m, n, k):
    """Algorithmic bytes of one GEMV: Q8_0 weights + int8 quants + f32 scales + f32 output."""
    return n * row_bytes(k) + m * k + m * (k // 32) * 4 + m * n * 4


def row_bytes_q4_0(k):
    return k // 32 * 18


def gemv_q4_0_bytes(m, n, k):
    """Algorithmic bytes of one Q4_0 GEMV: Q4_0 weights + int8 quants + f32 scales + output."""
    return n * row_bytes_q4_0(k) + m * k + m * (k // 32) * 4 + m * n * 4


def dequant_q4_0_bytes(n, k):
    return n * row_bytes_q4_0(k) + 2 * n * k


def gemm_flops(m, n, k):
    return 2.0 * m * n * k


def dequant_bytes(n, k):
    return n * row_bytes(k) + 2 * n * k


def quantize_bytes(m, k):
    return 4 * m * k + m * k + m * (k // 32) * 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------------------------
# clocks sampled by nvidia-smi while the timed loop runs
# ------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[2:7], float(parts[7])))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:   # a very short timed region: take the samples nearest to it
            mid = 0.5 * (t0 + t1)
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in inside:
            for nm, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside), "in_timed_region": t0 <= inside[0][0] <= t1}


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import q8_block_quantized_act_gb300 as q8
    from q8_block_quantized_act_gb300 import build as q8build
    from q8_block_quantized_act_gb300 import inputs

    q8build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()

    # ---- inputs: seeded host f32, quantized to Q8_0 on the device by the library ----
    def weights_q8(n, k):
        """Q8_0 and Q4_0 encodings of the same seeded f32 weights."""
        w32 = torch.from_numpy(inputs.weights_f32(n, k)).to(dev)
        wq = q8.quantize_q8_0(w32)
        w4 = q8.quantize_q4_0(w32)
        del w32
        return wq, w4

    w_gemv, w4_gemv = weights_q8(GEMV["n"], GEMV["k"])
    w_gemm, w4_gemm = weights_q8(GEMM["n"], GEMM["k"])
    x_gemv = torch.from_numpy(inputs.activations_f32(GEMV["m"], GEMV["k"])).to(dev)
    x_gemm = torch.from_numpy(inputs.activations_f32(GEMM["m"], GEMM["k"])).to(dev)
    xq = torch.empty((GEMV["m"], GEMV["k"]), dtype=torch.int8, device=dev)
    xd = torch.empty((GEMV["m"], GEMV["k"] // 32), dtype=torch.float32, device=dev)
    y_gemv = torch.empty((GEMV["m"], GEMV["n"]), dtype=torch.float32, device=dev)
    ws = q8.gemm_workspace(GEMM["m"], GEMM["k"], dev)
    y_gemm = torch.empty((GEMM["m"], GEMM["n"]), dtype=torch.float32, device=dev)
    w16 = torch.empty((DEQ["n"], DEQ["k"]), dtype=torch.float16, device=dev)
    wq16, wdt = q8.repack_q8_0(w_gemm, GEMM["n"], GEMM["k"])   # load time, outside the step
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    def flush_l2():
        flush.zero_()
        flush_rd.max()

    def k_quant():
        q8.check(q8.q8act_quantize_q8_1(x_gemv, xq, xd, GEMV["m"], GEMV["k"], stream))

    def k_gemv():
        q8.check(q8.q8act_gemv_q8_0(w_gemv, xq, xd, y_gemv, GEMV["m"], GEMV["n"], GEMV["k"], stream))

    def k_gemm():
        q8.check(q8.q8act_gemm_q8_0(w_gemm, x_gemm, y_gemm, GEMM["m"], GEMM["n"], GEMM["k"], ws,
                                    ws.numel(), stream))

    def k_gemm_rp():
        q8.check(q8.q8act_gemm_q8_0_repacked(wq16, wdt, x_gemm, y_gemm, GEMM["m"], GEMM["n"], GEMM["k"],
                                             ws, ws.numel(), stream))

    def k_deq():
        q8.check(q8.q8act_dequant_q8_0_f16(w_gemm, w16, DEQ["n"], DEQ["k"], stream))

    # Order: the dequant and the two GEMMs (L2 flushed before each), then the decode path -- the
    # token's q8_1 quantization and the GEMV.  The decode path follows a GEMM (8.4 MB output),
    # not the load-time dequant, whose 33.5 MB output would otherwise be written back from L2
    # inside the GEMV's stream.  The quantizer's 16 KB input was evicted by the previous step's
    # 280 MB GEMV stream and the flushes; the GEMV's input is larger than L2.
    parts = [("dequant_q8_0_f16", k_deq), ("gemm_q8_0", k_gemm), ("gemm_q8_0_repacked", k_gemm_rp),
             ("quantize_q8_1", k_quant), ("gemv_q8_0", k_gemv)]
    launches_per_step = {"quantize_q8_1": 1, "gemv_q8_0": 1, "gemm_q8_0": 2, "gemm_q8_0_repacked": 2,
                         "dequant_q8_0_f16": 1}

    # The GEMV's 280 MB weight stream is larger than L2, so it needs no flush; the GEMM's and
    # the dequant's inputs fit in L2 and are flushed before each launch.
    needs_flush = {"quantize_q8_1": False, "gemv_q8_0": False, "gemm_q8_0": True,
                   "gemm_q8_0_repacked": True, "dequant_q8_0_f16": True}

    def step(events=None):
        for i, (name, fn) in enumerate(parts):
            if needs_flush[name]:
                flush_l2()                      # evict L2 before the kernel
            if events is not None:
                events[i][0].record(stream)
            fn()
            if events is not None:
                events[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    q8.device_status(stream)

    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
           for _ in parts] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for s in range(args.steps):
        step(ev[s])
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.stop()
    q8.device_status(stream)

    per = {name: [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)]
           for i, (name, _) in enumerate(parts)}
    mean_ms = {name: float(np.mean(v)) for name, v in per.items()}
    spread = {name: {"median_us": round(float(np.median(v)) * 1e3, 3), "max_us": round(float(np.max(v)) * 1e3, 3),
                     "min_us": round(float(np.min(v)) * 1e3, 3)} for name, v in per.items()}
    step_ms = float(sum(mean_ms.values()))
    if world > 1:
        step_ms, mean_ms = max_over_ranks(step_ms, mean_ms, [nm for nm, _ in parts], dev)

    # ---- the next rows (Q4_0 GEMV and dequant): timed in a loop of their own, after the
    # step, with the same warm-up and flush rules; they are not part of the step ----
    y4 = torch.empty((GEMV["m"], GEMV["n"]), dtype=torch.float32, device=dev)

    def k_gemv4():
        q8.check(q8.q8act_gemv_q4_0(w4_gemv, xq, xd, y4, GEMV["m"], GEMV["n"], GEMV["k"], stream))

    def k_deq4():
        q8.check(q8.q8act_dequant_q4_0_f16(w4_gemm, w16, DEQ["n"], DEQ["k"], stream))

    ws_gemv = q8.gemv_workspace(GEMV["m"], GEMV["k"], dev)

    def k_gemv_f32():
        q8.check(q8.q8act_gemv_q8_0_f32(w_gemv, x_gemv, y4, GEMV["m"], GEMV["n"], GEMV["k"], ws_gemv,
                                        ws_gemv.numel(), stream))

    # the verify tier: 8 tokens (7 drafted + 1) against the decode weights, quantized once here
    mv = VERIFY_M
    xq_v = torch.empty((mv, GEMV["k"]), dtype=torch.int8, device=dev)
    xd_v = torch.empty((mv, GEMV["k"] // 32), dtype=torch.float32, device=dev)
    y_v = torch.empty((mv, GEMV["n"]), dtype=torch.float32, device=dev)
    x_v = torch.from_numpy(inputs.activations_f32(mv, GEMV["k"], seed=2)).to(dev)
    q8.check(q8.q8act_quantize_q8_1(x_v, xq_v, xd_v, mv, GEMV["k"], stream))

    def k_verify():
        q8.check(q8.q8act_gemv_q8_0(w_gemv, xq_v, xd_v, y_v, mv, GEMV["n"], GEMV["k"], stream))

    def k_verify4():
        q8.check(q8.q8act_gemv_q4_0(w4_gemv, xq_v, xd_v, y_v, mv, GEMV["n"], GEMV["k"], stream))

    nxt = [("dequant_q4_0_f16", k_deq4, True), ("gemv_q4_0", k_gemv4, False),
           ("gemv_q8_0_f32", k_gemv_f32, True), ("gemv_q8_0_verify", k_verify, False),
           ("gemv_q4_0_verify", k_verify4, False)]
    k_quant()
    for _ in range(args.warmup):
        for _, fn, fl in nxt:
            if fl:
                flush_l2()
            fn()
    nsteps = min(args.steps, 100)
    ev4 = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in nxt]
           for _ in range(nsteps)]
    for s_ in range(nsteps):
        for i, (_, fn, fl) in enumerate(nxt):
            if fl:
                flush_l2()
            ev4[s_][i][0].record(stream)
            fn()
            ev4[s_][i][1].record(stream)
    torch.cuda.synchronize()
    q8.device_status(stream)
    mean4 = {nm: float(np.mean([ev4[s_][i][0].elapsed_time(ev4[s_][i][1]) for s_ in range(nsteps)]))
             for i, (nm, _, _) in enumerate(nxt)}

    # ---- end to end through the public API: host f32 in (pinned), host f32 out ----
    e2e = run_e2e(args, q8, torch, dev, stream)

    # ---- every configuration of the workload table ----
    configs = None
    if not args.no_configs:
        configs = run_configs(args, q8, torch, dev, stream, load_peaks(), flush_l2,
                              {(GEMV["n"], GEMV["k"]): w_gemv, (GEMM["n"], GEMM["k"]): w_gemm})

    if rank != 0:
        return None
    peaks = load_peaks()
    comps = {}
    gb = gemv_bytes(**GEMV)
    comps["gemv_q8_0"] = roof("hbm", gb / (mean_ms["gemv_q8_0"] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                              mean_ms["gemv_q8_0"], gb)
    comps["quantize_q8_1"] = roof("hbm", quantize_bytes(GEMV["m"], GEMV["k"]) / (mean_ms["quantize_q8_1"] * 1e-3) / 1e9,
                                  peaks["hbm_gbs"], "GB/s", mean_ms["quantize_q8_1"], quantize_bytes(GEMV["m"], GEMV["k"]))
    fl = gemm_flops(**GEMM)
    comps["gemm_q8_0"] = roof("tensor", fl / (mean_ms["gemm_q8_0"] * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s",
                              mean_ms["gemm_q8_0"], fl)
    comps["gemm_q8_0_repacked"] = roof("tensor", fl / (mean_ms["gemm_q8_0_repacked"] * 1e-3) / 1e12,
                                       peaks["bf16_tflops"], "TFLOP/s", mean_ms["gemm_q8_0_repacked"], fl)
    db = dequant_bytes(**DEQ)
    comps["dequant_q8_0_f16"] = roof("hbm", db / (mean_ms["dequant_q8_0_f16"] * 1e-3) / 1e9, peaks["hbm_gbs"],
                                     "GB/s", mean_ms["dequant_q8_0_f16"], db)
    for nm in comps:
        comps[nm].update(spread[nm])
    # The GEMMs' second roofline: the per-block scale fold, acc += (d_w * d_a) * D for every
    # output element and 32-wide block -- 2 m n k / 32 FP32 lane operations -- against the FP32
    # pipes (128 lanes per SM) of the SMs the launch occupies (one 128 x 128 tile per SM at this
    # shape) at the SM clock sampled during the timed region.
    sms_total = torch.cuda.get_device_properties(dev).multi_processor_count
    tiles = -(-GEMM["n"] // 128) * -(-GEMM["m"] // 128)
    sms_used = min(tiles, sms_total)
    clk_mhz = (sampler.summary(t0, t1).get("sm_mhz") if sampler else None) or 2070.0
    fold_ops = 2.0 * GEMM["m"] * GEMM["n"] * GEMM["k"] / 32
    fold_floor_us = fold_ops / (sms_used * 128 * clk_mhz * 1e6) * 1e6
    for nm in ("gemm_q8_0", "gemm_q8_0_repacked"):
        comps[nm]["fold_roofline"] = {
            "bound": "alu (FP32 fold)", "work_per_launch": fold_ops, "unit": "FP32 lane-ops",
            "floor_us": round(fold_floor_us, 2), "sms": sms_used, "sm_mhz": clk_mhz,
            "frac": round(fold_floor_us / comps[nm]["us"], 4)}
    g4 = gemv_q4_0_bytes(**GEMV)
    gf = gemv_bytes(**GEMV) + 4 * GEMV["m"] * GEMV["k"]
    d4 = dequant_q4_0_bytes(**DEQ)
    gv = gemv_bytes(VERIFY_M, GEMV["n"], GEMV["k"])
    gv4 = gemv_q4_0_bytes(VERIFY_M, GEMV["n"], GEMV["k"])
    next_rows = {
        "gemv_q4_0": roof("hbm", g4 / (mean4["gemv_q4_0"] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                          mean4["gemv_q4_0"], g4),
        "dequant_q4_0_f16": roof("hbm", d4 / (mean4["dequant_q4_0_f16"] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                                 mean4["dequant_q4_0_f16"], d4),
        "gemv_q8_0_f32": roof("hbm", gf / (mean4["gemv_q8_0_f32"] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                              mean4["gemv_q8_0_f32"], gf),
        "gemv_q8_0_verify": roof("hbm", gv / (mean4["gemv_q8_0_verify"] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                                 mean4["gemv_q8_0_verify"], gv),
        "gemv_q4_0_verify": roof("hbm", gv4 / (mean4["gemv_q4_0_verify"] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s",
                                 mean4["gemv_q4_0_verify"], gv4),
        "steps": nsteps,
        "note": "Q4_0 (GGUF 18-byte blocks) GEMV m=1 4096->64448 and dequant 4096x4096 on the same seeded weights, and the fused decode call (q8_1 quantization + the Q8_0 GEMV in one call, f32 activation in; bytes = the GEMV's + the f32 activation), and the verify GEMVs (m=8: 7 drafted tokens + 1, 4096->64448, the tensor-core GEMV, on the Q8_0 and the Q4_0 weights); timed after the step in a loop of their own (the dequant and the fused call after an L2 flush)",
    }
    dominant = max(mean_ms, key=lambda nm: mean_ms[nm])
    traffic = load_traffic(dominant)
    d = comps[dominant]
    roofline = {"kernel": dominant, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"], "traffic": traffic,
                "peak_source": f"{peaks['source']} ({'hbm_gbs' if d['bound'] == 'hbm' else 'bf16_tflops burst; f16 pipe, nominal ratio 1'})"}

    value = whole_job_value(comps["gemv_q8_0"]["achieved"], world)
    cpu = cpu_baseline(args) if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    clocks = sampler.summary(t0, t1) if sampler else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded numpy PCG64: weights N(0,0.02) seed 0, activations N(0,1) seed 1)",
        "config": {"workload": WORKLOAD, "gemv": GEMV, "gemm": GEMM, "dequant": DEQ,
                   "l2": "flushed (256 MiB write, then a 256 MiB read) before each GEMM and the dequant; the GEMV's 280.5 MB input is larger than L2 and evicts the quantizer's input between steps",
                   "parallelism": f"replicas x{world}"},
        "gemm_tops": round(comps["gemm_q8_0"]["achieved"], 2),
        "gemm_repacked_tops": round(comps["gemm_q8_0_repacked"]["achieved"], 2),
        "components": comps,
        "next_rows": next_rows,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "configs": configs,
        "gpu_launches": sum(launches_per_step.values()) * args.steps,
        "clocks": clocks,
        "impl": "ours",
    }
    return line


def max_over_ranks(step_ms, mean_ms, names, device):
    """The slowest rank's step time and per-kernel times (every rank gets the same result)."""
    import torch
    t = torch.tensor([step_ms] + [mean_ms[nm] for nm in names], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t[0]), {nm: float(t[i + 1]) for i, nm in enumerate(names)}


def whole_job_value(per_rank_gbs_at_max_time, world):
    """Weak scaling: every rank streams the same bytes, so the job moves world x those bytes in
    the slowest rank's time."""
    return per_rank_gbs_at_max_time * world


def roof(bound, achieved, peak, unit, ms, work):
    return {"bound": bound, "achieved": round(achieved, 3), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "us": round(ms * 1e3, 3), "work_per_launch": work}


KERNEL_SOURCES = {"gemv_q8_0": "gemv.cu", "gemm_q8_0": "gemm.cu", "gemm_q8_0_repacked": "gemm.cu",
                  "dequant_q8_0_f16": "dequant.cu", "quantize_q8_1": "quantize.cu"}


def source_sha(kernel):
    import hashlib
    p = os.path.join(ROOT, "q8_block_quantized_act_gb300", "csrc", KERNEL_SOURCES[kernel])
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_traffic(kernel):
    """Per-launch DRAM bytes (read + write) of `kernel` from the committed ncu summary, or
    None when there is none or the kernel's source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    v = d.get(kernel)
    if not isinstance(v, dict) or v.get("source_sha") != source_sha(kernel):
        return None
    return v.get("bytes_per_launch")


def run_e2e(args, q8, torch, dev, stream):
    """The decode GEMV through the public API with host buffers, two ways.

    `e2e` (a serving step): the Q8_0 weights were uploaded once at load time and stay resident;
    every step copies the token's f32 activation in from pinned host memory, the fused decode
    call quantizes it and runs the GEMV, and y is copied back to pinned host memory.
    `weights_each_step`: the same, with all 280.5 MB of weights also copied in from pinned host
    memory every step (bound by the host link).
    `prefill_gemm`: the fused prefill call (m = 512, 4096 -> 4096) the same way as `e2e`:
    resident weights, the f32 activation in and y out through pinned host memory every step."""
    from q8_block_quantized_act_gb300 import inputs
    m, n, k = GEMV["m"], GEMV["n"], GEMV["k"]
    w_host = torch.empty((n, row_bytes(k)), dtype=torch.uint8).pin_memory()
    w_dev_tmp = q8.quantize_q8_0(torch.from_numpy(inputs.weights_f32(n, k)).to(dev))
    w_host.copy_(w_dev_tmp.cpu())
    del w_dev_tmp
    x_host = torch.from_numpy(inputs.activations_f32(m, k)).pin_memory()
    y_host = torch.empty((m, n), dtype=torch.float32).pin_memory()
    w_dev = torch.empty_like(w_host, device=dev)
    x_dev = torch.empty_like(x_host, device=dev)
    ws = q8.gemv_workspace(m, k, dev)
    y_dev = torch.empty((m, n), dtype=torch.float32, device=dev)

    def one():
        w_dev.copy_(w_host, non_blocking=True)
        x_dev.copy_(x_host, non_blocking=True)
        q8.check(q8.q8act_gemv_q8_0_f32(w_dev, x_dev, y_dev, m, n, k, ws, ws.numel(), stream))
        y_host.copy_(y_dev, non_blocking=True)

    def resident():
        x_dev.copy_(x_host, non_blocking=True)
        q8.check(q8.q8act_gemv_q8_0_f32(w_dev, x_dev, y_dev, m, n, k, ws, ws.numel(), stream))
        y_host.copy_(y_dev, non_blocking=True)

    def timed(fn, reps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    ms_all = timed(one, max(3, min(args.steps, 50)))
    w_dev.copy_(w_host)            # load time: the weights stay resident from here on
    torch.cuda.synchronize()
    ms_res = timed(resident, max(10, min(args.steps, 200)))

    # The prefill call the same way: resident Q8_0 weights, every step copies the f32 activation
    # in from pinned host memory, makes the fused GEMM call (q8_1 quantize + GEMM) and copies y out.
    gm, gn, gk = GEMM["m"], GEMM["n"], GEMM["k"]
    wg_dev = q8.quantize_q8_0(torch.from_numpy(inputs.weights_f32(gn, gk)).to(dev))
    xg_host = torch.from_numpy(inputs.activations_f32(gm, gk)).pin_memory()
    yg_host = torch.empty((gm, gn), dtype=torch.float32).pin_memory()
    xg_dev = torch.empty_like(xg_host, device=dev)
    yg_dev = torch.empty((gm, gn), dtype=torch.float32, device=dev)
    wsg = q8.gemm_workspace(gm, gk, dev)

    def prefill():
        xg_dev.copy_(xg_host, non_blocking=True)
        q8.check(q8.q8act_gemm_q8_0(wg_dev, xg_dev, yg_dev, gm, gn, gk, wsg, wsg.numel(), stream))
        yg_host.copy_(yg_dev, non_blocking=True)

    ms_pf = timed(prefill, max(10, min(args.steps, 100)))
    prefill_gemm = {"value": round(2.0 * gm * gn * gk / (ms_pf * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(xg_host.numel() * 4), "d2h_bytes_per_step": int(yg_host.numel() * 4),
                    "ms_per_step": round(ms_pf, 4),
                    "what": f"fused prefill call (q8_1 quantize + GEMM, m={gm}, {gk}->{gn}) through the C ABI; "
                            "weights resident; every step copies x in from pinned host memory and y out to pinned "
                            "host memory"}
    return {"value": round(gemv_bytes(m, n, k) / (ms_res * 1e-3) / 1e9, 2), "unit": "GB/s",
            "prefill_gemm": prefill_gemm,
            "h2d_bytes_per_step": int(x_host.numel() * 4),
            "d2h_bytes_per_step": int(y_host.numel() * 4), "ms_per_step": round(ms_res, 4),
            "what": "fused decode call (q8_1 quantize + GEMV, m=1, 4096->64448) through the C ABI; weights "
                    "uploaded once and resident; every step copies x in from pinned host memory and y out "
                    "to pinned host memory",
            "weights_each_step": {
                "value": round(gemv_bytes(m, n, k) / (ms_all * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(w_host.numel() + x_host.numel() * 4),
                "d2h_bytes_per_step": int(y_host.numel() * 4), "ms_per_step": round(ms_all, 4)}}


# ------------------------------------------------------------------------------------
# every configuration of the workload table, one row each
# ------------------------------------------------------------------------------------
def cpu_description():
    """The host CPU's model name and core count (lscpu on Arm, /proc/cpuinfo elsewhere)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    return {"model": model or "unknown", "nproc": os.cpu_count()}


def time_events(fn, reps, warmup, stream, torch, flush=None):
    """CUDA-event time of each of `reps` calls (ms), after `warmup` untimed ones; `flush` runs
    before every call, outside the events."""
    for _ in range(warmup):
        if flush:
            flush()
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in evs:
        if flush:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


L2_BYTES = 129 * 1000 * 1000   # GB300 L2 (about 129 MB)


def time_b2b(fns, reps, stream, torch):
    """Mean ms per call of `reps` calls issued back to back inside one event pair (after a
    warm-up), cycling through `fns` -- one closure per weight copy, so that consecutive calls
    read different copies and, with copies totalling more than twice L2, each call reads its
    weights from HBM."""
    for f in fns[:3]:
        f()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(reps):
        fns[i % len(fns)]()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def graph_fields(ms, nbytes, peaks):
    if ms is None:
        return {"us_graph": None, "gbs_graph": None, "frac_graph": None}
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"us_graph": round(ms * 1e3, 2), "gbs_graph": round(gbs, 1), "frac_graph": round(gbs / peaks["hbm_gbs"], 4)}


def time_graph(fns, reps, torch):
    """Mean ms per call when the `reps` calls (cycling through `fns`, each closure issuing its
    call on torch's current stream) are captured once into a CUDA graph and replayed: the
    device's own time per call in a sequence, without the host's per-call launch cost.  None
    when the capture is refused."""
    try:
        for f in fns[:3]:
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                fns[i % len(fns)]()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        del g
        return ms
    except Exception:   # capture unsupported in this environment: no graph figure
        torch.cuda.synchronize()
        return None


def n_copies(nbytes, cap=32):
    """Weight copies whose total exceeds twice L2 (at most `cap`)."""
    return max(1, min(cap, -(-2 * L2_BYTES // max(1, nbytes))))


def oracle_time(wf32_rows, x, k, sample_rows, n):
    """Seconds the single-threaded oracle takes for the whole configuration: its q8_1
    quantization of x plus the fold over `sample_rows` weight rows, scaled by n / sample_rows
    (exact when the sample is every row)."""
    import oracle
    oracle.build()
    wb = oracle.quantize_q8_0(wf32_rows)
    t0 = time.perf_counter()
    xq, xd = oracle.quantize_q8_1(x)
    t1 = time.perf_counter()
    oracle.matmul(wb, xq, xd, k)
    t2 = time.perf_counter()
    return (t1 - t0) + (t2 - t1) * n / sample_rows


def run_configs(args, q8, torch, dev, stream, peaks, flush_l2, resident):
    """Each configuration of the workload table: the GEMV rows (m = 1..8, pre-quantized activation,
    as the pages' decode census times mmvq), the fused-quantize GEMMs on raw Q8_0 and on the
    load-time repack, and the fp16 dequants.  Per row: median and mean us per call, throughput,
    the fraction of the measured peak, and the oracle's time for the same configuration on the
    same seeded inputs (a row sample scaled to all rows, marked extrapolated)."""
    from q8_block_quantized_act_gb300 import inputs
    reps = max(5, min(args.config_reps, 200))
    rows_out = []
    weights = dict(resident)           # (n, k) -> device Q8_0 bytes already built by the step
    host_rows = {}

    def wq(n, k):
        if (n, k) not in weights:
            w32 = torch.from_numpy(inputs.weights_f32(n, k)).to(dev)
            weights[(n, k)] = q8.quantize_q8_0(w32)
            del w32
        if (n, k) not in host_rows:
            # the generator fills rows in order: these are the matrix's first rows
            host_rows[(n, k)] = inputs.weights_f32(min(n, 512), k)
        return weights[(n, k)]

    def orc(n, k, x, sample):
        sample = min(sample, n)
        return oracle_time(host_rows[(n, k)][:sample], x, k, sample, n), sample < n, sample

    for name, m, n, k, kind in inputs.GEMV_CASES:
        w = wq(n, k)
        x = inputs.activations_f32(m, k, kind=kind)
        xq, xd = q8.quantize_q8_1(torch.from_numpy(x).to(dev))
        y = torch.empty((m, n), dtype=torch.float32, device=dev)
        big = n * row_bytes(k) > 200e6

        def fn():
            q8.check(q8.q8act_gemv_q8_0(w, xq, xd, y, m, n, k, stream))

        t = time_events(fn, reps, 3, stream, torch, None if big else flush_l2)
        med, mean = float(np.median(t)), float(np.mean(t))
        by = gemv_bytes(m, n, k)
        copies = [w] + [w.clone() for _ in range(n_copies(n * row_bytes(k)) - 1)]

        def mk(wc, st=stream):
            return lambda: q8.check(q8.q8act_gemv_q8_0(wc, xq, xd, y, m, n, k, st))
        b2b = time_b2b([mk(wc) for wc in copies], max(reps, 4 * len(copies)), stream, torch)
        gr = time_graph([mk(wc, None) for wc in copies], max(reps, 4 * len(copies)), torch)
        del copies
        o_s, extrap, smp = (None, None, None) if args.no_cpu_baseline else orc(n, k, x, 512)
        rows_out.append({"config": name, "op": "gemv", "m": m, "n": n, "k": k, "act": kind,
                         "us_median": round(med * 1e3, 2), "us_mean": round(mean * 1e3, 2),
                         "gbs": round(by / (med * 1e-3) / 1e9, 1), "bound": "hbm",
                         "frac": round(by / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         "us_b2b": round(b2b * 1e3, 2), "gbs_b2b": round(by / (b2b * 1e-3) / 1e9, 1),
                         "frac_b2b": round(by / (b2b * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         **graph_fields(gr, by, peaks),
                         "b2b_weight_copies": n_copies(n * row_bytes(k)),
                         "l2": "resident weights larger than L2" if big else "flushed before each call",
                         "oracle_s": None if o_s is None else round(o_s, 4), "oracle_extrapolated": extrap,
                         "oracle_rows": smp})
    ws = None
    for name, m, n, k, kind in inputs.GEMM_CASES:
        w = wq(n, k)
        wq16, wdt = q8.repack_q8_0(w, n, k)
        x = inputs.activations_f32(m, k, kind=kind)
        x_d = torch.from_numpy(x).to(dev)
        y = torch.empty((m, n), dtype=torch.float32, device=dev)
        need = q8.q8act_gemm_workspace_bytes(m, k)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=dev)

        def raw():
            q8.check(q8.q8act_gemm_q8_0(w, x_d, y, m, n, k, ws, ws.numel(), stream))

        def rp():
            q8.check(q8.q8act_gemm_q8_0_repacked(wq16, wdt, x_d, y, m, n, k, ws, ws.numel(), stream))

        fl = gemm_flops(m, n, k)
        o_s, extrap, smp = (None, None, None) if args.no_cpu_baseline else orc(n, k, x, 32)
        for variant, fn in (("raw", raw), ("repacked", rp)):
            nrep = max(5, reps // 4) if fl > 1e11 else reps
            t = time_events(fn, nrep, 3, stream, torch, flush_l2)
            med, mean = float(np.median(t)), float(np.mean(t))
            tf = fl / (med * 1e-3) / 1e12
            wbytes = n * row_bytes(k) if variant == "raw" else (2 * n * k + 4 * q8.q8act_repack_ldn(n) * (k // 32))
            ncp = n_copies(wbytes, cap=16)
            if variant == "raw":
                cps = [w] + [w.clone() for _ in range(ncp - 1)]

                def mk(wc, st=stream):
                    return lambda: q8.check(q8.q8act_gemm_q8_0(wc, x_d, y, m, n, k, ws, ws.numel(), st))
                fns = [mk(wc) for wc in cps]
                gfns = [mk(wc, None) for wc in cps]
            else:
                cps = [(wq16, wdt)] + [(wq16.clone(), wdt.clone()) for _ in range(ncp - 1)]

                def mk(pr, st=stream):
                    return lambda: q8.check(q8.q8act_gemm_q8_0_repacked(pr[0], pr[1], x_d, y, m, n, k, ws, ws.numel(),
                                                                        st))
                fns = [mk(pr) for pr in cps]
                gfns = [mk(pr, None) for pr in cps]
            b2b = time_b2b(fns, max(nrep, 2 * len(fns)), stream, torch)
            gr = time_graph(gfns, max(nrep, 2 * len(fns)), torch)
            del fns, gfns, cps
            tfb = fl / (b2b * 1e-3) / 1e12
            rows_out.append({"config": name, "op": f"gemm_{variant}", "m": m, "n": n, "k": k, "act": kind,
                             "us_median": round(med * 1e3, 2), "us_mean": round(mean * 1e3, 2),
                             "tflops": round(tf, 1), "bound": "tensor", "frac": round(tf / peaks["bf16_tflops"], 4),
                             "us_b2b": round(b2b * 1e3, 2), "tflops_b2b": round(tfb, 1),
                             "frac_b2b": round(tfb / peaks["bf16_tflops"], 4), "b2b_weight_copies": ncp,
                             "us_graph": None if gr is None else round(gr * 1e3, 2),
                             "tflops_graph": None if gr is None else round(fl / (gr * 1e-3) / 1e12, 1),
                             "frac_graph": None if gr is None else round(fl / (gr * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                             "l2": "flushed before each call",
                             "oracle_s": None if o_s is None else round(o_s, 3), "oracle_extrapolated": extrap,
                             "oracle_rows": smp})
        del wq16, wdt, x_d, y
    for n, k in ((4096, 4096), (5152, 4096)):
        w = wq(n, k)
        w16 = torch.empty((n, k), dtype=torch.float16, device=dev)

        def deq():
            q8.check(q8.q8act_dequant_q8_0_f16(w, w16, n, k, stream))

        t = time_events(deq, reps, 3, stream, torch, flush_l2)
        med, mean = float(np.median(t)), float(np.mean(t))
        by = dequant_bytes(n, k)
        cps = [w] + [w.clone() for _ in range(n_copies(n * row_bytes(k)) - 1)]

        def mk(wc, st=stream):
            return lambda: q8.check(q8.q8act_dequant_q8_0_f16(wc, w16, n, k, st))
        b2b = time_b2b([mk(wc) for wc in cps], max(reps, 4 * len(cps)), stream, torch)
        gr = time_graph([mk(wc, None) for wc in cps], max(reps, 4 * len(cps)), torch)
        del cps
        rows_out.append({"config": f"dequant_{k}x{n}", "op": "dequant_q8_0_f16", "m": 0, "n": n, "k": k,
                         "us_median": round(med * 1e3, 2), "us_mean": round(mean * 1e3, 2),
                         "gbs": round(by / (med * 1e-3) / 1e9, 1), "bound": "hbm",
                         "frac": round(by / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         "us_b2b": round(b2b * 1e3, 2), "gbs_b2b": round(by / (b2b * 1e-3) / 1e9, 1),
                         "frac_b2b": round(by / (b2b * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         **graph_fields(gr, by, peaks),
                         "l2": "flushed before each call", "oracle_s": None, "oracle_extrapolated": None,
                         "oracle_rows": None})
    # The q8_1 quantizers on their own: the MMQ layout that the GEMM's fused quantization writes
    # (m = 512, 2048: binary16 quants + transposed scales) and the row layout of the decode GEMV
    # (m = 1).  Bytes: the f32 activation read once, the quants and scales written once.
    for m, k, layout in ((512, 4096, "mmq"), (2048, 4096, "mmq"), (1, 4096, "row")):
        x_d = torch.from_numpy(inputs.activations_f32(m, k)).to(dev)
        if layout == "mmq":
            ldm = q8.q8act_mmq_ldm(m)
            oq = torch.empty((m, k), dtype=torch.uint16, device=dev)
            od = torch.empty((k // 32, ldm), dtype=torch.float32, device=dev)
            fnq = q8.q8act_quantize_q8_1_mmq
            by = 4 * m * k + 2 * m * k + 4 * (k // 32) * ldm
        else:
            oq = torch.empty((m, k), dtype=torch.int8, device=dev)
            od = torch.empty((m, k // 32), dtype=torch.float32, device=dev)
            fnq = q8.q8act_quantize_q8_1
            by = quantize_bytes(m, k)

        def mkq(xc, st):
            return lambda: q8.check(fnq(xc, oq, od, m, k, st))
        t = time_events(mkq(x_d, stream), reps, 3, stream, torch, flush_l2)
        med, mean = float(np.median(t)), float(np.mean(t))
        ncp = n_copies(4 * m * k)
        cps = [x_d] + [x_d.clone() for _ in range(ncp - 1)]
        b2b = time_b2b([mkq(xc, stream) for xc in cps], max(reps, 4 * ncp), stream, torch)
        gr = time_graph([mkq(xc, None) for xc in cps], max(reps, 4 * ncp), torch)
        del cps, x_d, oq, od
        rows_out.append({"config": f"quantize_q8_1_{layout}_m{m}", "op": f"quantize_q8_1_{layout}", "m": m, "n": 0,
                         "k": k, "us_median": round(med * 1e3, 2), "us_mean": round(mean * 1e3, 2),
                         "gbs": round(by / (med * 1e-3) / 1e9, 1), "bound": "hbm",
                         "frac": round(by / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         "us_b2b": round(b2b * 1e3, 2), "gbs_b2b": round(by / (b2b * 1e-3) / 1e9, 1),
                         "frac_b2b": round(by / (b2b * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         **graph_fields(gr, by, peaks),
                         "b2b_input_copies": ncp, "l2": "flushed before each call",
                         "oracle_s": None, "oracle_extrapolated": None, "oracle_rows": None})
    # K-quant superblocks (Q6_K, Q4_K, Q5_K) on seeded random superblocks: the fp16 mirror of a
    # 4096 x 4096 and a 20480 x 4096 weight, and the GEMV at 4096 -> 64448 for one token (the
    # dp4a kernel) and for eight (the tensor-core kernel)
    xs_kq = {}
    for mm in (1, 8):
        xs_kq[mm] = q8.quantize_q8_1(torch.from_numpy(inputs.activations_f32(mm, 4096)).to(dev))
    for fmt, sbytes in (("q6_k", 210), ("q4_k", 144), ("q5_k", 176)):
        for n, k, what, mm in ((4096, 4096, "dequant", 0), (20480, 4096, "dequant", 0), (64448, 4096, "gemv", 1),
                               (64448, 4096, "gemv", 8)):
            wk = torch.from_numpy(inputs.kquant_superblocks(fmt, n, k)).to(dev)
            wbytes = n * (k // 256) * sbytes
            if what == "dequant":
                w16 = torch.empty((n, k), dtype=torch.float16, device=dev)
                fn_dq = getattr(q8, f"q8act_dequant_{fmt}_f16")

                def mkf(wc, st, fn_dq=fn_dq, w16=w16, n=n, k=k):
                    return lambda: q8.check(fn_dq(wc, w16, n, k, st))
                by = wbytes + 2 * n * k
                big = False
            else:
                xqk, xdk = xs_kq[mm]
                yk = torch.empty((mm, n), dtype=torch.float32, device=dev)
                fn_gv = getattr(q8, f"q8act_gemv_{fmt}")

                def mkf(wc, st, fn_gv=fn_gv, xqk=xqk, xdk=xdk, yk=yk, mm=mm, n=n, k=k):
                    return lambda: q8.check(fn_gv(wc, xqk, xdk, yk, mm, n, k, st))
                by = wbytes + mm * k + mm * (k // 32) * 4 + mm * n * 4
                big = True
            t = time_events(mkf(wk, stream), reps, 3, stream, torch, None if big else flush_l2)
            med, mean = float(np.median(t)), float(np.mean(t))
            ncp = n_copies(wbytes)
            cps = [wk] + [wk.clone() for _ in range(ncp - 1)]
            b2b = time_b2b([mkf(wc, stream) for wc in cps], max(reps, 4 * ncp), stream, torch)
            gr = time_graph([mkf(wc, None) for wc in cps], max(reps, 4 * ncp), torch)
            del cps
            cfg = f"{what}_{fmt}_{k}x{n}" + (f"_m{mm}" if what == "gemv" and mm > 1 else "")
            rows_out.append({"config": cfg, "op": f"{what}_{fmt}", "m": mm, "n": n, "k": k,
                             "us_median": round(med * 1e3, 2), "us_mean": round(mean * 1e3, 2),
                             "gbs": round(by / (med * 1e-3) / 1e9, 1), "bound": "hbm",
                             "frac": round(by / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                             "us_b2b": round(b2b * 1e3, 2), "gbs_b2b": round(by / (b2b * 1e-3) / 1e9, 1),
                             "frac_b2b": round(by / (b2b * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                             **graph_fields(gr, by, peaks),
                             "b2b_weight_copies": ncp,
                             "l2": "weights larger than L2" if big else "flushed before each call",
                             "oracle_s": None, "oracle_extrapolated": None, "oracle_rows": None})
            del wk
    torch.cuda.synchronize()
    q8.device_status(stream)
    cpu = cpu_description()
    cpu["oracle_threads"] = 1
    return {"rows": rows_out, "reps": reps, "cpu": cpu,
            "note": "GEMV rows: the pre-quantized-activation GEMV (as the pages' census times mmvq); GEMM rows: "
                    "the whole fused call (q8_1 quantize + GEMM).  us_median / us_mean: one call between CUDA "
                    "events after an L2 flush (includes the launch and the event pair, a few us); us_b2b: the "
                    "mean of calls issued back to back in one event pair, cycling through b2b_weight_copies "
                    "weight copies (more than twice L2 in total where the cap allows, so each call still reads "
                    "its weights from HBM), the census's way of timing (it repeats one warm buffer); us_graph: "
                    "the same calls captured once into a CUDA graph and replayed, the device's time per call "
                    "without the host's per-call launch cost.  "
                    "oracle_s: the single-threaded C oracle on the same inputs (q8_1 quantize + fold), timed on "
                    "oracle_rows weight rows and scaled to n (oracle_extrapolated)"}


# ------------------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)
# ------------------------------------------------------------------------------------
def oracle_gemv_sample(min_seconds=10.0, max_seconds=30.0, rows_per_rep=16384):
    """Time the oracle on the decode GEMV workload: quantize the token, then the fold over a
    seeded block of weight rows; repeated (different row blocks) until >= min_seconds."""
    import oracle
    from q8_block_quantized_act_gb300 import inputs
    m, n, k = GEMV["m"], GEMV["n"], GEMV["k"]
    oracle.build()
    w = inputs.weights_f32(rows_per_rep, k)
    wb = oracle.quantize_q8_0(w)
    x = inputs.activations_f32(m, k)
    done_bytes, t_total, reps = 0, 0.0, 0
    while reps == 0 or (t_total < min_seconds and t_total < max_seconds):
        t = time.perf_counter()
        xq, xd = oracle.quantize_q8_1(x)
        oracle.matmul(wb, xq, xd, k)
        t_total += time.perf_counter() - t
        done_bytes += gemv_bytes(m, rows_per_rep, k)
        reps += 1
    return done_bytes / t_total / 1e9, reps, rows_per_rep, t_total


def cpu_baseline(args):
    gbs, reps, rows, secs = oracle_gemv_sample(min_seconds=args.cpu_seconds)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"decode GEMV m=1, k=4096: {reps} x {rows} weight rows "
                      f"({reps * rows / GEMV['n']:.2f} x the 64448-row workload), {secs:.1f} s, "
                      "single-threaded C oracle"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    per_step = []
    for _ in range(args.warmup):
        oracle_gemv_sample(min_seconds=0.0, rows_per_rep=1024)
    t_all = 0.0
    bytes_all = 0
    for _ in range(args.steps):
        gbs, reps, rows, secs = oracle_gemv_sample(min_seconds=0.0, rows_per_rep=4096)
        per_step.append(secs)
        t_all += secs
        bytes_all += gemv_bytes(GEMV["m"], rows, GEMV["k"])
    value = bytes_all / t_all / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_all / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemv": GEMV},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "each step: the decode GEMV (m=1, k=4096) over 4096 of the "
                                   "64448 weight rows, single-threaded C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration table")
    ap.add_argument("--config-reps", type=int, default=40, help="timed calls per configuration row")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
