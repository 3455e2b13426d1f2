#!/usr/bin/env python
"""Benchmark of the NVFP4 linear-projection hot path on GB300.

One step = for every projection of the workload: NVFP4 quantization of the
residual weight W_res (both orientations, RTN), the linear forward
(amax + dual RTN quantization of X, BF16 branch factor, block-scaled GEMM
with the fused rank-r branch) and the linear backward (amax + dual SR
quantization of dY, branch factor, dX GEMM with branch, dW GEMM).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload block3b|mlp_up|single]

Prints one JSON line (rank 0).  `value` is NVFP4 GEMM TFLOP/s of the whole
step (3 GEMMs x 2MNK per projection) with inputs resident in HBM; `e2e` is the
same with the step's inputs copied from pinned host memory and its results
copied back inside the timed region.  The reference arm (--impl reference)
times the CPU oracle on a bounded sample of the same workload.
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

METRIC = "NVFP4 linear fwd+bwd TFLOP/s and % dense-FP4 peak; quantize GB/s % HBM (1 GB300)"
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor rate on GB300

WORKLOADS = {
    "block3b": dict(
        name="block3b_T16384_d3072_ff8192_r64",
        desc="3B-class transformer block projections, T=16384 tokens: qkv 9216x3072, o 3072x3072, "
             "gate_up 16384x3072, down 3072x8192; rank-64 LoRA-SVD; RTN fwd, SR bwd; fwd+bwd",
        T=16384, r=64, x="student_t",
        projections=[("qkv", 9216, 3072), ("o", 3072, 3072), ("gate_up", 16384, 3072), ("down", 3072, 8192)]),
    "mlp_up": dict(
        name="mlp_up_T8192_d2048_f5632_r32",
        desc="~1B MLP up projection, T=8192, W 5632x2048, rank-32 LoRA-SVD, fwd+bwd",
        T=8192, r=32, x="normal", projections=[("up", 5632, 2048)]),
    "single": dict(
        name="single_fwd_256x512x512_r16",
        desc="single NVFP4 linear, X 256x512, W 512x512, rank 16 (fwd+bwd)",
        T=256, r=16, x="normal", projections=[("w", 512, 512)]),
}

# ncu DRAM traffic per launch of the block-scaled GEMM on the bench workload,
# keyed by the SHA-256 of the kernel source it was captured on (null once the
# source changes).  Filled from the committed profile summary.
GEMM_TRAFFIC = {
    # launch list of `--part step --steps 2 --warmup 3` with dram__bytes_read.sum and
    # dram__bytes_write.sum (one pass): mean over the 96 GEMM launches of the 3B block
    "537b552b4b8b0248": 215260000,
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gemm_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh"):
        h.update(open(os.path.join(ROOT, "nvfp4_quantized_pretraining_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (monotonic time, line)
        self.thread = None
        self.window = None  # (t0, t1) of the timed region; samples outside it are dropped

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def wait_ready(self, timeout: float = 10.0):
        """Block until nvidia-smi has printed its first sample (it takes a while to start)."""
        t_end = time.monotonic() + timeout
        while self.proc and not self.lines and time.monotonic() < t_end:
            time.sleep(0.01)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if self.window and not (self.window[0] - 0.025 <= ts <= self.window[1] + 0.025):
                continue
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Evicts the inputs of the next timed call from the 129 MB L2 and leaves it clean: a
    512 MB buffer is written (the flush), then a second 256 MB buffer is read, which evicts the
    written lines back to HBM inside the flush.  Without the read, the next timed kernel would
    write back up to 129 MB of the flush's own dirty lines (about 19 us of HBM time)."""

    def __init__(self, torch, dev):
        self.w = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the slowest rank's time); `value` itself on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def whole_job_tflops(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the work of every rank's step over the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def lora_split(F, torch, S, W, r, seed, dev):
    """The LoRA-SVD split W = W_res + L2 L1 of a random-init weight, made on the device by the
    library's randomized-SVD realignment (W_res = W, zero factors in; sketch r + 16, 2 power
    iterations).  Set-up, outside every timed region."""
    N, K = W.shape
    Om = S.normal_device((K, r + REALIGN_OVERSAMPLE), 1.0, seed, dev)
    z1 = torch.zeros((r, K), dtype=torch.bfloat16, device=dev)
    z2 = torch.zeros((N, r), dtype=torch.bfloat16, device=dev)
    Wres, L1, L2, info = F.fp4_lora_realign(W, z1, z2, Om, q=REALIGN_POWER_ITERS)
    if int(info.item()) != 0:
        raise RuntimeError(f"LoRA-SVD split of a {N} x {K} weight failed: info = {int(info.item())}")
    return Wres, L1, L2


def run_ours(args):
    import torch
    import torch.distributed as dist

    import nvfp4_quantized_pretraining_gb300 as F
    from nvfp4_quantized_pretraining_gb300 import build as B
    from nvfp4_quantized_pretraining_gb300 import synthetic as S

    rank, world, local = dist_env()
    B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.part not in ("all", "step"):
        run_part(args, F, torch, S, dev)
        return
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[args.workload]
    T, r = wl["T"], wl["r"]
    stream = torch.cuda.Stream(device=dev)
    projs = []
    seed0 = 1000 * rank
    for i, (name, N, K) in enumerate(wl["projections"]):
        W = S.normal_device((N, K), 0.02, seed0 + 10 * i, dev)
        Wres, L1, L2 = lora_split(F, torch, S, W, r, seed0 + 10 * i + 1, dev) if r else (W, None, None)
        X = (S.student_t_device((T, K), 3, seed0 + 10 * i + 2, dev) if wl["x"] == "student_t"
             else S.normal_device((T, K), 1.0, seed0 + 10 * i + 2, dev))
        dY = S.normal_device((T, N), 1e-3, seed0 + 10 * i + 3, dev)
        p = dict(name=name, N=N, K=K, X=X, dY=dY, Wres=Wres, L1=L1, L2=L2)
        p["Wq"] = F.NVFP4Tensor.empty(N, K, dev)
        p["WqT"] = F.NVFP4Tensor.empty(K, N, dev)
        p["xqT"] = F.NVFP4Tensor.empty(K, T, dev)
        p["Y"] = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        p["dX"] = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
        p["dW"] = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
        # each with the room for the GEMMs' split tail
        p["ws_f"] = torch.empty(F.linear_fwd_workspace(T, N, K, r) + F.gemm_split_workspace(), dtype=torch.uint8,
                                device=dev)
        p["ws_b"] = torch.empty(F.linear_bwd_workspace(T, N, K, r) + F.gemm_split_workspace(), dtype=torch.uint8,
                                device=dev)
        projs.append(p)
    flush = L2Flush(torch, dev)  # > 2x the 129 MB L2, left clean
    gemm_flops = sum(3 * 2 * T * p["N"] * p["K"] for p in projs)
    branch_flops = sum(2 * T * p["K"] * r + 2 * T * p["N"] * r + 2 * T * p["N"] * r + 2 * T * p["K"] * r
                       for p in projs) if r else 0

    def step(seed):
        # a training step's order: the forward of every projection in model order, then the
        # backward in reverse order
        for p in projs:
            F.fp4_quantize_dual(p["Wres"], out_row=p["Wq"], out_col=p["WqT"], stream=stream)
            F.fp4_linear_fwd(p["X"], p["Wq"], p["L1"], p["L2"], Y=p["Y"], xqT_saved=p["xqT"], workspace=p["ws_f"],
                             stream=stream)
        for p in reversed(projs):
            F.fp4_linear_bwd(p["dY"], p["WqT"], p["xqT"], p["L1"], p["L2"], seed=seed, dX=p["dX"], dW=p["dW"],
                             workspace=p["ws_b"], stream=stream)

    def timed(fn, steps, warmup):
        with torch.cuda.stream(stream):
            for i in range(warmup):
                fn(i)
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize(dev)
            times = []
            t_start = time.monotonic()
            for i in range(steps):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn(warmup + i)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            torch.cuda.synchronize(dev)
            t_end = time.monotonic()
            if world > 1:
                dist.barrier()
        return times, (t_start, t_end)

    # ---- main timed region: device-resident inputs
    launches0 = F.fp4_launch_count()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    with ClockSampler(gpu_id) as clk:
        clk.wait_ready()
        times, clk.window = timed(step, args.steps, args.warmup)
    launches = (F.fp4_launch_count() - launches0) * args.steps // (args.steps + args.warmup)
    F.fp4_check_status(stream)
    total_ms = max_over_ranks(sum(times), dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(gemm_flops, world, ms_per_step)

    # ---- kernel breakdown through the public calls (same operands), for the roofline
    bd = breakdown(F, torch, projs, T, r, stream, dev, flush, args)
    if args.part == "step":  # the timed step and its breakdown only (for profiling)
        if rank == 0:
            print(json.dumps({"step": {"ms_per_step": round(ms_per_step, 4), "value": round(value, 2),
                                       "breakdown_ms": {k: round(v, 4) for k, v in bd["per_kind_ms"].items()}}}),
                  flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    lg = lora_grads(F, torch, projs, T, r, stream, dev, flush, args) if r else None
    cq = lora_cholqr(F, torch, projs, r, stream, dev, flush, args) if r else None
    ra = lora_realign(F, torch, S, projs, r, stream, dev, flush, args) if r else None
    ns = newton_schulz(F, torch, S, stream, dev, flush, args)
    vt = qadamw_codec(F, torch, projs, stream, dev, flush, args)
    qsw = quantize_sweep(F, torch, S, stream, dev, flush, args)
    gsw = gemm_sweep(F, torch, S, stream, dev, flush, args)

    # ---- end-to-end: host inputs -> device -> step -> results back to host
    e2e = end_to_end(F, torch, projs, T, r, stream, dev, args, gemm_flops, world)

    pk, pk_kind = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    gemm_tf = bd["gemm_flops"] / (bd["gemm_ms"] * 1e-3) / 1e12
    h = gemm_source_hash()
    traffic = GEMM_TRAFFIC.get(h)
    q_gbs = bd["rtn_bytes"] / (bd["rtn_ms"] * 1e-3) / 1e9
    sr_gbs = bd["sr_bytes"] / (bd["sr_ms"] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic (seeded; random-init weights split by randomized SVD)",
        "config": {"workload": wl["name"], "description": wl["desc"], "tokens": T, "rank": r,
                   "l2": "flushed before every timed step (512 MB written, then 256 MB of another buffer read so that L2 is left clean)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "gemm_nvf4_pair_kernel", "achieved": round(gemm_tf, 1),
                     "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "frac": round(gemm_tf / fp4_peak, 4),
                     "traffic": traffic,
                     "peak_note": f"{pk_kind} bf16 burst {pk['bf16_tflops']} TFLOP/s x {FP4_OVER_BF16:g} "
                                  "(nominal dense FP4:BF16 ratio); datasheet dense FP4 13500 TFLOP/s",
                     "frac_of_datasheet": round(gemm_tf / 13500.0, 4)},
        "quantize_rtn": {"bound": "hbm", "achieved": round(q_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(q_gbs / pk["hbm_gbs"], 4),
                         "note": "X and W: algorithmic bytes of the dual-orientation RTN launches (2 B read + "
                                 "2 x 0.5625 B written per element) over their event time"},
        "quantize_sr": {"bound": "alu", "elements_per_s": round(bd["sr_elems"] / (bd["sr_ms"] * 1e-3), 1),
                        "achieved_gbs": round(sr_gbs, 1), "hbm_frac": round(sr_gbs / pk["hbm_gbs"], 4),
                        "note": "dY, both forms with SR: bound by the integer ALU pipe (two Philox4x32-10 draws "
                                "and the SR rule per element; ncu on 16384^2: ALU pipe 72% busy, 43 instructions "
                                "per element, DRAM 24%)"},
        "breakdown_ms": {k: round(v, 4) for k, v in bd["per_kind_ms"].items()},
        "lora_factor_grads": lg,
        "lora_cholqr": cq,
        "lora_realign": ra,
        "newton_schulz": ns,
        "qadamw_v_codec": vt,
        "quantize_sweep": qsw,
        "gemm_sweep": gsw,
        "branch_tflops_counted_separately": round(branch_flops / 1e12, 4),
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args, wl)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def breakdown(F, torch, projs, T, r, stream, dev, flush, args):
    """Times each public call of one step separately with CUDA events on the
    launching stream (after warm-up, L2 flushed before every step)."""
    ev = []
    gemm_flops = 0
    reps = max(2, min(args.steps, 5))
    kinds = {}
    sk = torch.empty(F.gemm_blockscaled_workspace(T, r), dtype=torch.uint8, device=dev)

    def rec(kind, fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        ev.append((kind, e0, e1))

    with torch.cuda.stream(stream):
        for rep in range(reps + 1):
            flush.zero_()
            ev.clear()
            for p in projs:
                N, K = p["N"], p["K"]
                xq = F.NVFP4Tensor.empty(T, K, dev) if rep == 0 and "xq" not in p else p.get("xq")
                p["xq"] = xq
                dyq = p.get("dyq") or F.NVFP4Tensor.empty(T, N, dev)
                dyqT = p.get("dyqT") or F.NVFP4Tensor.empty(N, T, dev)
                p["dyq"], p["dyqT"] = dyq, dyqT
                if "P" not in p:
                    p["P"] = torch.empty((T, r), dtype=torch.bfloat16, device=dev) if r else None
                    p["P2"] = torch.empty((T, r), dtype=torch.bfloat16, device=dev) if r else None
                    p["L2T"] = p["L2"].t().contiguous() if r else None
                    p["L1T"] = p["L1"].t().contiguous() if r else None
                    p["amax"] = torch.empty(1, dtype=torch.float32, device=dev)
                rec("quantize_w_dual", lambda: F.fp4_quantize_dual(p["Wres"], out_row=p["Wq"], out_col=p["WqT"],
                                                                   stream=stream))
                # as in fp4_linear_fwd/bwd: with a branch, its factor kernel also yields the amax
                if r:
                    rec("branch_factor_amax", lambda: F.fp4_branch_factor(p["X"], p["L1"], out=p["P"],
                                                                          amax=p["amax"], stream=stream))
                else:
                    rec("amax", lambda: F.fp4_amax(p["X"], out=p["amax"], stream=stream))
                rec("quantize_x_dual", lambda: F.fp4_quantize_dual(p["X"], amax=p["amax"], out_row=xq,
                                                                   out_col=p["xqT"], stream=stream))
                rec("gemm", lambda: F.fp4_gemm_blockscaled_ws(xq, p["Wq"], p["P"], p["L2"], out=p["Y"], workspace=sk,
                                                              stream=stream))
                if r:
                    rec("branch_factor_amax", lambda: F.fp4_branch_factor(p["dY"], p["L2T"], out=p["P2"],
                                                                          amax=p["amax"], stream=stream))
                else:
                    rec("amax", lambda: F.fp4_amax(p["dY"], out=p["amax"], stream=stream))
                rec("quantize_dy_dual_sr", lambda: F.fp4_quantize_dual(p["dY"], round_mode=F.SR, seed=rep,
                                                                       amax=p["amax"], out_row=dyq, out_col=dyqT,
                                                                       stream=stream))
                rec("gemm", lambda: F.fp4_gemm_blockscaled_ws(dyq, p["WqT"], p["P2"], p["L1T"], out=p["dX"],
                                                              workspace=sk, stream=stream))
                rec("gemm", lambda: F.fp4_gemm_blockscaled_ws(dyqT, p["xqT"], out=p["dW"], workspace=sk,
                                                              stream=stream))
            torch.cuda.synchronize(dev)
            if rep == 0:
                continue  # warm-up pass
            for kind, e0, e1 in ev:
                kinds.setdefault(kind, 0.0)
                kinds[kind] += e0.elapsed_time(e1) / reps
    rtn_bytes = sr_bytes = 0
    sr_elems = 0
    for p in projs:
        gemm_flops += 3 * 2 * T * p["N"] * p["K"]
        rtn_bytes += int(3.125 * (T * p["K"] + p["N"] * p["K"]))   # X and W: both forms from one read
        sr_bytes += int(3.125 * T * p["N"])                        # dY
        sr_elems += T * p["N"]
    rtn_ms = kinds.get("quantize_x_dual", 0) + kinds.get("quantize_w_dual", 0)
    return dict(gemm_flops=gemm_flops, gemm_ms=kinds["gemm"], rtn_bytes=rtn_bytes, rtn_ms=rtn_ms,
                sr_bytes=sr_bytes, sr_elems=sr_elems, sr_ms=kinds.get("quantize_dy_dual_sr", 0), per_kind_ms=kinds)


def lora_grads(F, torch, projs, T, r, stream, dev, flush, args):
    """Times the LoRA-SVD factor gradients of every projection (dL2 = beta dY^T P and
    dL1 = beta P'^T X, with the step's own P and P'), each call after an L2 flush.
    Not part of the timed step: a separate figure against HBM, the bound of this
    product (it reads dY and X once; the factors and the results are small)."""
    reps = max(2, min(args.steps, 5))
    total = 0.0
    nbytes = 0
    ws = None
    with torch.cuda.stream(stream):
        for p in projs:
            need = max(F.lib().fp4_lora_factor_grad_workspace(T, p["N"], r),
                       F.lib().fp4_lora_factor_grad_workspace(T, p["K"], r))
            if ws is None or ws.numel() < need:
                ws = torch.empty(need, dtype=torch.uint8, device=dev)
            dL2 = torch.empty((p["N"], r), dtype=torch.float32, device=dev)
            dL1 = torch.empty((r, p["K"]), dtype=torch.float32, device=dev)
            calls = [lambda: F.fp4_lora_factor_grad(p["dY"], p["P"], 1.0, out=dL2, workspace=ws, stream=stream),
                     lambda: F.fp4_lora_factor_grad(p["X"], p["P2"], 1.0, transpose=True, out=dL1, workspace=ws,
                                                    stream=stream)]
            for fn, M in zip(calls, (p["N"], p["K"])):
                fn()
                ts = []
                for _ in range(reps):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
                total += sorted(ts)[len(ts) // 2]
                nbytes += T * M * 2 + T * r * 2 + M * r * 4
    F.fp4_check_status(stream)
    hbm = float(peaks()[0]["hbm_gbs"])
    gbs = nbytes / (total * 1e-3) / 1e9
    return {"ms_per_step": round(total, 4), "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(gbs / hbm, 4),
            "note": "dL2 = dY^T P and dL1 = P'^T X of the four projections; algorithmic bytes "
                    "(BF16 dY or X, the T x r factor, the FP32 result) over the summed median call times"}


def lora_cholqr(F, torch, projs, r, stream, dev, flush, args):
    """Times the Cholesky-QR step of each projection's LoRA factors (L1 r x K, L2 N x r),
    out of place, each call after an L2 flush.  Not part of the timed step.  It moves
    only the factors (a few MB), so it is latency-bound: three short launches."""
    reps = max(1, min(args.steps, 5))
    total = 0.0
    with torch.cuda.stream(stream):
        for p in projs:
            o1, o2 = torch.empty_like(p["L1"]), torch.empty_like(p["L2"])
            info = torch.zeros(1, dtype=torch.int32, device=dev)
            ws = torch.empty(F.lib().fp4_lora_cholqr_workspace(p["K"], r), dtype=torch.uint8, device=dev)
            fn = lambda: F.fp4_lora_cholqr(p["L1"], p["L2"], L1_out=o1, L2_out=o2, info=info, workspace=ws,
                                           stream=stream)
            fn()
            ts = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            total += sorted(ts)[len(ts) // 2]
            if int(info.item()) != 0:
                raise RuntimeError(f"Cholesky-QR of {p['name']}: info = {int(info.item())}")
    F.fp4_check_status(stream)
    return {"ms_per_step": round(total, 4), "bound": "latency",
            "note": "L1 <- L^-1 L1, L2 <- L2 L of the four projections (r = 64), summed median call times"}


REALIGN_OVERSAMPLE, REALIGN_POWER_ITERS = 16, 2


def lora_realign(F, torch, S, projs, r, stream, dev, flush, args):
    """Times the randomized-SVD realignment of each projection's weight (W_res + L2 L1, rank r,
    sketch width r + 16, 2 power iterations), out of place, each call after an L2 flush.  Not
    part of the timed step (it runs every few thousand steps).  FLOPs are those of the FP32
    products, 2 N K (2 r + s (2 + 2 q)) per weight (the sketch products run on the tensor cores
    as three TF32 products each, the rest on the CUDA cores), shown against the FP32 CUDA-core
    rate (152 SMs x 128 FMA/clk x 2 FLOP x 2.07 GHz, ~80 TFLOP/s) for scale; most of the call's
    time is now in its one-CTA Jacobi and Cholesky kernels, so it is latency-bound."""
    s_cols, q = r + REALIGN_OVERSAMPLE, REALIGN_POWER_ITERS
    reps = max(1, min(args.steps, 3))
    total, flops = 0.0, 0.0
    with torch.cuda.stream(stream):
        for i, p in enumerate(projs):
            N, K = p["N"], p["K"]
            Om = S.normal_device((K, s_cols), 1.0, 700 + i, dev)
            outs = (torch.empty_like(p["Wres"]), torch.empty_like(p["L1"]), torch.empty_like(p["L2"]))
            info = torch.zeros(1, dtype=torch.int32, device=dev)
            ws = torch.empty(F.lib().fp4_lora_realign_workspace(N, K, r, s_cols), dtype=torch.uint8, device=dev)
            fn = lambda: F.fp4_lora_realign(p["Wres"], p["L1"], p["L2"], Om, q=q, out=outs, info=info,
                                            workspace=ws, stream=stream)
            fn()
            ts = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            total += sorted(ts)[len(ts) // 2]
            flops += 2.0 * N * K * (2 * r + s_cols * (2 + 2 * q))
            if int(info.item()) != 0:
                raise RuntimeError(f"realignment of {p['name']}: info = {int(info.item())}")
            del outs, ws, Om
    F.fp4_check_status(stream)
    fp32_peak = 152 * 128 * 2 * 2.07e9 / 1e12
    tf = flops / (total * 1e-3) / 1e12
    return {"ms_total": round(total, 4), "sketch": s_cols, "power_iters": q, "fp32_tflops": round(tf, 1),
            "bound": "latency", "peak": round(fp32_peak, 1), "unit": "TFLOP/s", "frac": round(tf / fp32_peak, 4),
            "note": "four weights of the block; FP32 product FLOPs over the summed median call times (the "
                    "products with W and W^T on the tensor cores as three TF32 products each, the others on the "
                    "CUDA cores; the one-CTA Jacobi eigensolver and Cholesky factorisations take most of the "
                    "time); the peak is the FP32 FMA rate at the 2.07 GHz maximum SM clock, for scale"}


def run_part(args, F, torch, S, dev):
    """One optimizer-side measurement alone, with the same shapes as in the full line."""
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(torch, dev)
    wl = WORKLOADS[args.workload]
    projs = [dict(name=n, N=N, K=K) for n, N, K in wl["projections"]]
    if args.part == "newton_schulz":
        res = newton_schulz(F, torch, S, stream, dev, flush, args)
    elif args.part == "quantize_sweep":
        res = quantize_sweep(F, torch, S, stream, dev, flush, args)
    elif args.part == "quantize_one":
        res = quantize_one(F, torch, stream, dev, flush, args)
    elif args.part == "branch_one":
        res = branch_one(F, torch, S, stream, dev, flush, args)
    elif args.part == "gemm_one":
        res = gemm_one(F, torch, stream, dev, flush, args)
    elif args.part == "gemm_sweep":
        res = gemm_sweep(F, torch, S, stream, dev, flush, args)
    elif args.part == "qadamw_v_codec":
        res = qadamw_codec(F, torch, projs, stream, dev, flush, args)
    elif args.part == "lora_cholqr":
        r = wl["r"]
        for i, p in enumerate(projs):  # N(0, 0.02) rows: a positive definite Gram matrix (r <= K)
            p["L1"] = S.normal_device((r, p["K"]), 0.02, 810 + i, dev)
            p["L2"] = S.normal_device((p["N"], r), 0.02, 820 + i, dev)
        res = lora_cholqr(F, torch, projs, r, stream, dev, flush, args)
    else:
        r = wl["r"]
        for i, p in enumerate(projs):
            p["Wres"] = S.normal_device((p["N"], p["K"]), 0.02, 800 + i, dev)
            p["L1"] = S.normal_device((r, p["K"]), 0.02, 810 + i, dev)
            p["L2"] = S.normal_device((p["N"], r), 0.02, 820 + i, dev)
        res = lora_realign(F, torch, S, projs, r, stream, dev, flush, args)
    print(json.dumps({args.part: res}), flush=True)


def _warm_clocks(torch, stream, flush, seconds=0.25):
    """Keeps the GPU busy for `seconds` (L2 flushes) so that its clocks have ramped up before a
    short timed call; a fresh process otherwise times its first calls at idle clocks."""
    t0 = time.monotonic()
    with torch.cuda.stream(stream):
        while time.monotonic() - t0 < seconds:
            for _ in range(20):
                flush.zero_()
            torch.cuda.synchronize()


def _median_ms(torch, stream, flush, fn, reps):
    """Median CUDA-event time of fn() on `stream`, L2 flushed before each timed call."""
    fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return sorted(ts)[len(ts) // 2]


def quantize_sweep(F, torch, S, stream, dev, flush, args):
    """The standalone quantize sweep: BF16 tensors of 1M, 16M, 64M and 256M elements shaped
    rows x 4096, N(0, 1) with 0.1% of entries x50; RTN and SR (seed 0); the row form, the
    transposed (column-block) form and both from one read.  Each call after an L2 flush, in two
    variants: the quantize kernel alone with the tensor amax supplied, and the full call with the
    amax pass.  Algorithmic bytes per element: 2 read + 0.5 + 1/16 written per form (2.5625 for
    one form, 3.125 for both), + 2 for the amax pass."""
    hbm = float(peaks()[0]["hbm_gbs"])
    reps = max(3, min(args.steps, 7))
    out = {}
    worst = worst_b2b = None
    with torch.cuda.stream(stream):
        for n in S.QUANT_SWEEP_ELEMS:
            rows, cols = n // 4096, 4096
            # the tensor, plus copies for the back-to-back figure: distinct inputs of at least 256 MB
            # together (more than L2), so that every call of the batch reads its tensor from HBM
            nb = max(4, min(8, -(-(256 << 20) // (2 * n))))
            xs = []
            for c in range(nb):
                g = torch.Generator(device=dev)
                g.manual_seed(600 + rows + 7919 * c)
                x = torch.randn((rows, cols), generator=g, device=dev, dtype=torch.float32)
                xs.append(torch.where(torch.rand((rows, cols), generator=g, device=dev) < 0.001, x * 50.0,
                                      x).to(torch.bfloat16))
                del x
            x = xs[0]
            amaxs = [F.fp4_amax(xi, stream=stream) for xi in xs]
            amax = amaxs[0]
            qr, qc = F.NVFP4Tensor.empty(rows, cols, dev), F.NVFP4Tensor.empty(cols, rows, dev)
            label = f"{n >> 20}M"
            out[label] = {"shape": [rows, cols], "back_to_back_calls": nb}
            for mode, mname in ((F.RTN, "rtn"), (F.SR, "sr")):
                forms = {
                    "row": (2.5625, lambda xi, a: F.fp4_quantize(xi, mode, 0, 0, amax=a, out=qr, stream=stream)),
                    "transposed": (2.5625, lambda xi, a: F.fp4_quantize_transposed(xi, mode, 0, 1, amax=a, out=qc,
                                                                                   stream=stream)),
                    "dual": (3.125, lambda xi, a: F.fp4_quantize_dual(xi, mode, 0, 0, 1, amax=a, out_row=qr,
                                                                      out_col=qc, stream=stream)),
                }
                for form, (bpe, fn) in forms.items():
                    ms_k = _median_ms(torch, stream, flush, lambda: fn(x, amax), reps)
                    ms_a = _median_ms(torch, stream, flush, lambda: fn(x, None), reps)

                    def batch():
                        for xi, ai in zip(xs, amaxs):
                            fn(xi, ai)

                    ms_b = _median_ms(torch, stream, flush, batch, reps) / nb
                    gk = bpe * n / (ms_k * 1e-3) / 1e9
                    ga = (bpe + 2.0) * n / (ms_a * 1e-3) / 1e9
                    gb = bpe * n / (ms_b * 1e-3) / 1e9
                    out[label][f"{form}_{mname}"] = {
                        "ms": round(ms_k, 4), "gbs": round(gk, 1), "frac": round(gk / hbm, 4),
                        "ms_with_amax": round(ms_a, 4), "gbs_with_amax": round(ga, 1),
                        "frac_with_amax": round(ga / hbm, 4),
                        "ms_back_to_back": round(ms_b, 4), "frac_back_to_back": round(gb / hbm, 4)}
                    if n >= (1 << 24) and mode == F.RTN and (worst is None or gk / hbm < worst[0]):
                        worst = (gk / hbm, f"{label} {form}")
                    if n >= (1 << 24) and mode == F.RTN and (worst_b2b is None or gb / hbm < worst_b2b[0]):
                        worst_b2b = (gb / hbm, f"{label} {form}")
            del x, xs, qr, qc, amax, amaxs
    F.fp4_check_status(stream)
    return {"bound": "hbm", "peak": hbm, "unit": "GB/s", "sizes": out,
            "min_rtn_frac_16M_up": None if worst is None else {"frac": round(worst[0], 4), "case": worst[1]},
            "min_rtn_frac_back_to_back_16M_up": None if worst_b2b is None else
            {"frac": round(worst_b2b[0], 4), "case": worst_b2b[1]},
            "note": "kernel-only rate with the amax supplied (frac) and the full call with the amax pass "
                    "(frac_with_amax); algorithmic bytes over the median time of one call, L2 flushed before "
                    "each call, so a call's fixed launch and ramp cost (about 7 us, the whole 1M call) is in "
                    "it. frac_back_to_back: the same calls issued back to back on back_to_back_calls distinct "
                    "tensors (256 MB or more together, more than L2, so each reads HBM), the batch's median "
                    "time per call"}


def quantize_one(F, torch, stream, dev, flush, args):
    """One quantize call on an N(0, 1) tensor of --qshape with 0.1% of entries x50 (--qform row,
    transposed or dual; --qmode rtn or sr), amax supplied: `steps` warm-up calls and a quarter
    second of L2 flushes (clocks up), then the median of 9 calls, each after an L2 flush.  The first
    timed call is launch `steps` + 1 of the kernel: the one to profile."""
    rows, cols = args.qshape
    g = torch.Generator(device=dev)
    g.manual_seed(601)
    x = torch.randn((rows, cols), generator=g, device=dev, dtype=torch.float32)
    x = torch.where(torch.rand((rows, cols), generator=g, device=dev) < 0.001, x * 50.0, x).to(torch.bfloat16)
    amax = F.fp4_amax(x, stream=stream)
    mode = F.SR if args.qmode == "sr" else F.RTN
    qr, qc = F.NVFP4Tensor.empty(rows, cols, dev), F.NVFP4Tensor.empty(cols, rows, dev)
    fn = {"row": lambda: F.fp4_quantize(x, mode, 0, 0, amax=amax, out=qr, stream=stream),
          "transposed": lambda: F.fp4_quantize_transposed(x, mode, 0, 1, amax=amax, out=qc, stream=stream),
          "dual": lambda: F.fp4_quantize_dual(x, mode, 0, 0, 1, amax=amax, out_row=qr, out_col=qc,
                                              stream=stream)}[args.qform]
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            fn()
    _warm_clocks(torch, stream, flush)
    with torch.cuda.stream(stream):
        ms = _median_ms(torch, stream, flush, fn, 9)
    F.fp4_check_status(stream)
    bpe = 3.125 if args.qform == "dual" else 2.5625
    gbs = bpe * rows * cols / (ms * 1e-3) / 1e9
    return {"shape": [rows, cols], "form": args.qform, "mode": args.qmode, "ms": round(ms, 4), "gbs": round(gbs, 1),
            "frac": round(gbs / float(peaks()[0]["hbm_gbs"]), 4)}


def branch_one(F, torch, S, stream, dev, flush, args):
    """One branch-factor call P = bf16(X L^T) with max |X| on X of --qshape (M x K, Student-t
    activations) and L of rank --rank: `steps` warm-up calls and a quarter second of L2
    flushes (clocks up), then the median of 9 calls, each after an L2 flush.  Algorithmic bytes: X read
    once (2 B per element), L and P.  The first timed call is launch `steps` + 1: the one to profile."""
    M, K = args.qshape
    r = args.rank
    X = S.student_t_device((M, K), 3, 611, dev)
    L = S.normal_device((r, K), 0.02, 612, dev)
    P = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    fn = lambda: F.fp4_branch_factor(X, L, out=P, amax=amax, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            fn()
    _warm_clocks(torch, stream, flush)
    with torch.cuda.stream(stream):
        ms = _median_ms(torch, stream, flush, fn, 9)
    F.fp4_check_status(stream)
    nbytes = 2 * M * K + 2 * r * K + 2 * M * r
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"shape": [M, K], "rank": r, "ms": round(ms, 4), "gbs": round(gbs, 1),
            "frac": round(gbs / float(peaks()[0]["hbm_gbs"]), 4)}


def gemm_one(F, torch, stream, dev, flush, args):
    """One block-scaled GEMM of --gshape M N K (operands N(0, 1) quantized RTN, rank --rank branch with
    P, Q ~ N(0, 1), BF16 output): `steps` warm-up calls and a quarter second of L2 flushes (clocks up), then the median of
    9 calls, each after an L2 flush.  The first timed call is launch `steps` + 1: the one to profile."""
    M, N, K = args.gshape
    r = args.rank
    g = torch.Generator(device=dev)
    g.manual_seed(M + 3 * N + 7 * K)
    qa = F.fp4_quantize(torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16), stream=stream)
    qb = F.fp4_quantize(torch.randn((N, K), generator=g, device=dev).to(torch.bfloat16), stream=stream)
    P = torch.randn((M, r), generator=g, device=dev).to(torch.bfloat16) if r else None
    Q = torch.randn((N, r), generator=g, device=dev).to(torch.bfloat16) if r else None
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    sk = torch.empty(F.gemm_blockscaled_workspace(M, r), dtype=torch.uint8, device=dev)
    fn = lambda: F.fp4_gemm_blockscaled_ws(qa, qb, P, Q, out=C, workspace=sk, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            fn()
    _warm_clocks(torch, stream, flush)
    with torch.cuda.stream(stream):
        ms = _median_ms(torch, stream, flush, fn, 9)
    F.fp4_check_status(stream)
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    return {"shape": [M, N, K], "rank": r, "ms": round(ms, 4), "tflops": round(tf, 1)}


def gemm_sweep(F, torch, S, stream, dev, flush, args):
    """The block-scaled NVFP4 GEMM shape sweep: M = N = K in {2048, 4096, 8192, 16384}, the
    16384 x 3072 x 8192 skinny shape and the 3072 x 8192 x 16384 dW shape; operands N(0, 1)
    quantized RTN, rank 0 and rank 64 (P, Q ~ N(0, 1) BF16), BF16 output.  TFLOP/s counts the
    2MNK FP4 FLOPs (the rank-64 branch's 2MNr BF16 FLOPs are extra work, not counted); torch's
    BF16 matmul on the same shapes is reported as context."""
    pk = peaks()[0]
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    reps = max(3, min(args.steps, 7))
    out = {}
    with torch.cuda.stream(stream):
        for (M, N, K) in S.GEMM_SWEEP:
            g = torch.Generator(device=dev)
            g.manual_seed(M + 3 * N + 7 * K)
            A = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
            B = torch.randn((N, K), generator=g, device=dev).to(torch.bfloat16)
            qa, qb = F.fp4_quantize(A, stream=stream), F.fp4_quantize(B, stream=stream)
            P = torch.randn((M, 64), generator=g, device=dev).to(torch.bfloat16)
            Q = torch.randn((N, 64), generator=g, device=dev).to(torch.bfloat16)
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            sk = torch.empty(F.gemm_blockscaled_workspace(M, 64), dtype=torch.uint8, device=dev)
            flops = 2.0 * M * N * K
            row = {}
            for r in (0, 64):
                fn = (lambda: F.fp4_gemm_blockscaled_ws(qa, qb, out=C, workspace=sk, stream=stream)) if r == 0 else \
                     (lambda: F.fp4_gemm_blockscaled_ws(qa, qb, P, Q, out=C, workspace=sk, stream=stream))
                ms = _median_ms(torch, stream, flush, fn, reps)
                tf = flops / (ms * 1e-3) / 1e12
                row[f"r{r}"] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / fp4_peak, 4)}
            ms = _median_ms(torch, stream, flush, lambda: torch.matmul(A, B.t(), out=C), reps)
            row["torch_bf16_matmul"] = {"ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
            out[f"{M}x{N}x{K}"] = row
            del A, B, qa, qb, P, Q, C, sk
    F.fp4_check_status(stream)
    return {"bound": "tensor", "peak": round(fp4_peak, 1), "unit": "TFLOP/s", "shapes": out,
            "note": "gemm_nvf4_pair_kernel; 2MNK FP4 FLOPs over the median call time (L2 flushed); the peak is "
                    "the measured BF16 burst rate x 6 (nominal dense FP4:BF16 ratio)"}


def newton_schulz(F, torch, S, stream, dev, flush, args):
    """Times Q-Root's orthogonalisation (normalise, then 12 cubic Newton-Schulz steps with
    NVFP4 products and the p99 clip) of one gradient of each weight shape of the block,
    each call after an L2 flush.  Not part of the timed step (an optimizer-side figure).
    FLOPs: 4 m^2 n per step (A = X X^T and B X)."""
    reps = max(1, min(args.steps, 3))
    out = {}
    total_ms = total_flops = 0.0
    with torch.cuda.stream(stream):
        for i, (name, m, n) in enumerate(S.NS_SHAPES_3B):
            G = S.normal_device((m, n), 1e-3, 500 + i, dev)
            X = torch.empty_like(G)
            ws = torch.empty(F.newton_schulz_workspace(m, n, F.NS_COEFFS[2]), dtype=torch.uint8, device=dev)
            fn = lambda: F.fp4_newton_schulz(G, out=X, workspace=ws, stream=stream)
            fn()
            ts = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            ms = sorted(ts)[len(ts) // 2]
            flops = F.NS_STEPS * 4.0 * m * m * n
            out[name] = {"m": m, "n": n, "ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
            total_ms += ms
            total_flops += flops
            del G, X, ws
    F.fp4_check_status(stream)
    return {"shapes": out, "steps": F.NS_STEPS, "coeffs": list(F.NS_COEFFS), "clip": "p99 of the iterate",
            "ms_total": round(total_ms, 4), "tflops": round(total_flops / (total_ms * 1e-3) / 1e12, 1),
            "note": "one orthogonalisation per weight-gradient shape (m <= n); FP4 GEMM FLOPs over the "
                    "whole call's event time (normalisation, clips, quantizations and GEMMs)"}


def qadamw_codec(F, torch, projs, stream, dev, flush, args):
    """Times the Q-AdamW second-moment codec on the AdamW state of each weight of the block
    (FP32 v with the weight's shape), encode and decode separately, each call after an L2
    flush.  Not part of the timed step (an optimizer-side figure).  Algorithmic bytes per
    element: encode reads v once (4 B) and writes codes, scales and means (0.6875 B); decode
    the reverse.  The encoder reads v twice (max |h| first), so its ceiling is ~54% of HBM."""
    reps = max(1, min(args.steps, 5))
    enc = dec = 0.0
    elems = 0
    with torch.cuda.stream(stream):
        for i, p in enumerate(projs):
            R, C = p["N"], p["K"]
            g = torch.Generator(device=dev)
            g.manual_seed(900 + i)
            v = (torch.randn((R, C), generator=g, device=dev) ** 2) * 1e-6
            q = F.NVFP4Tensor.empty(R, C, dev)
            mean = torch.empty((R, C // 16), dtype=torch.bfloat16, device=dev)
            out = torch.empty_like(v)
            calls = (lambda: F.fp4_qadamw_v_encode(v, out=q, mean=mean, stream=stream),
                     lambda: F.fp4_qadamw_v_decode(q, mean, out=out, stream=stream))
            med = []
            for fn in calls:
                fn()
                ts = []
                for _ in range(reps):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
                med.append(sorted(ts)[len(ts) // 2])
            enc += med[0]
            dec += med[1]
            elems += R * C
            del v, q, mean, out
    F.fp4_check_status(stream)
    hbm = float(peaks()[0]["hbm_gbs"])
    nbytes = elems * (4 + 0.5 + 1 / 16 + 2 / 16)
    ge, gd = nbytes / (enc * 1e-3) / 1e9, nbytes / (dec * 1e-3) / 1e9
    return {"elements": elems, "encode_ms": round(enc, 4), "decode_ms": round(dec, 4), "bound": "hbm",
            "encode_gbs": round(ge, 1), "decode_gbs": round(gd, 1), "peak": hbm, "unit": "GB/s",
            "encode_frac": round(ge / hbm, 4), "decode_frac": round(gd / hbm, 4),
            "note": "v_t of the four weights (FP32 state); 4.6875 algorithmic B/element each way over the "
                    "summed median call times; the encoder reads v twice by design"}


def end_to_end(F, torch, projs, T, r, stream, dev, args, gemm_flops, world):
    """Same step, with X and dY copied from pinned host memory before and Y, dX
    and dW copied back to pinned host memory after, all inside the timed region."""
    hosts = []
    h2d = d2h = 0
    for p in projs:
        hx = torch.empty_like(p["X"], device="cpu").pin_memory()
        hx.copy_(p["X"])
        hdy = torch.empty_like(p["dY"], device="cpu").pin_memory()
        hdy.copy_(p["dY"])
        outs = [torch.empty_like(p[k], device="cpu").pin_memory() for k in ("Y", "dX", "dW")]
        hosts.append((hx, hdy, outs))
        h2d += hx.numel() * 2 + hdy.numel() * 2
        d2h += sum(o.numel() * o.element_size() for o in outs)
    # Three streams, as a user of the C ABI would run it: host-to-device copies on one, the step on the
    # compute stream as each input lands, the copies back on a third.  The host link (measured 210 GB/s
    # in, 193 GB/s out, 340 GB/s both ways at once, whatever the number of streams) bounds this
    # measurement, the outbound channel most, so that channel is kept busy from as early as possible:
    # every X is sent first, so that each forward starts as soon as its own X has landed and its Y
    # goes back at once (the forwards' outputs, 1 GB, then stream out while the dY still come in);
    # the dY follow in the order of the backward passes, and each dX and dW goes back as soon as its
    # backward is done.
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    fwd_order = list(range(len(projs)))
    bwd_order = fwd_order[::-1]
    times = []
    for it in range(args.warmup + args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        d2h_stream.wait_event(e0)
        x_in, dy_in = {}, {}
        with torch.cuda.stream(h2d_stream):
            for i in fwd_order:
                projs[i]["X"].copy_(hosts[i][0], non_blocking=True)
                x_in[i] = torch.cuda.Event()
                x_in[i].record(h2d_stream)
            for i in bwd_order:
                projs[i]["dY"].copy_(hosts[i][1], non_blocking=True)
                dy_in[i] = torch.cuda.Event()
                dy_in[i].record(h2d_stream)
        for i in fwd_order:
            p, outs = projs[i], hosts[i][2]
            with torch.cuda.stream(stream):
                stream.wait_event(x_in[i])
                F.fp4_quantize_dual(p["Wres"], out_row=p["Wq"], out_col=p["WqT"], stream=stream)
                F.fp4_linear_fwd(p["X"], p["Wq"], p["L1"], p["L2"], Y=p["Y"], xqT_saved=p["xqT"],
                                 workspace=p["ws_f"], stream=stream)
                fwd_done = torch.cuda.Event()
                fwd_done.record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(fwd_done)
                outs[0].copy_(p["Y"], non_blocking=True)
        for i in bwd_order:
            p, outs = projs[i], hosts[i][2]
            with torch.cuda.stream(stream):
                stream.wait_event(dy_in[i])
                F.fp4_linear_bwd(p["dY"], p["WqT"], p["xqT"], p["L1"], p["L2"], seed=it, dX=p["dX"], dW=p["dW"],
                                 workspace=p["ws_b"], stream=stream)
                bwd_done = torch.cuda.Event()
                bwd_done.record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(bwd_done)
                outs[1].copy_(p["dX"], non_blocking=True)
                outs[2].copy_(p["dW"], non_blocking=True)
        end = torch.cuda.Event()
        end.record(d2h_stream)
        stream.wait_event(end)
        e1.record(stream)
        e1.synchronize()
        if it >= args.warmup:
            times.append(e0.elapsed_time(e1))
    ms = sum(times) / len(times)
    return {"value": round(world * gemm_flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

_ORACLE_CACHE = {}


def oracle_sample(wl, tokens):
    """One bounded sample of the workload on the CPU oracle: the smallest
    projection's full weight quantization plus forward+backward on a slice of
    `tokens` tokens.  Returns (flops, seconds, description, threads)."""
    import oracle
    from nvfp4_quantized_pretraining_gb300 import synthetic as S

    oracle.build()
    name, N, K = min(wl["projections"], key=lambda p: p[1] * p[2])
    r = wl["r"]
    t = min(wl["T"], tokens)
    key = (wl["name"], t)
    if key not in _ORACLE_CACHE:
        W = S.normal((N, K), 0.02, 1)
        Wres, L1, L2 = oracle.lora_svd_split(W, r)
        X = S.student_t((t, K), 3.0, 2) if wl["x"] == "student_t" else S.normal((t, K), 1.0, 2)
        dY = S.normal((t, N), 1e-3, 3)
        _ORACLE_CACHE[key] = (Wres, L1, L2, X, dY)
    Wres, L1, L2, X, dY = _ORACLE_CACHE[key]
    t0 = time.perf_counter()
    oracle.linear_fwd(X, Wres, L1, L2)
    oracle.linear_bwd(dY, X, Wres, L1, L2, seed=1)
    dt = time.perf_counter() - t0
    flops = 3 * 2 * t * N * K
    desc = (f"oracle (C quantizer + NumPy FP64 GEMMs) on projection '{name}' {N}x{K} with {t} of {wl['T']} tokens: "
            f"weight quantization (row+col) and linear fwd+bwd")
    return flops, dt, desc, oracle.max_threads()


CPU_BASELINE_SECONDS = 10.0  # the oracle sample is repeated until about this much CPU work is timed


def oracle_rate(wl, tokens: int, seconds: float):
    """Repeats the oracle sample until about `seconds` of work is timed; (TFLOP/s, reps, desc, threads)."""
    total_flops, total_s, reps = 0.0, 0.0, 0
    desc = threads = None
    while total_s < seconds and reps < 200:
        flops, dt, desc, threads = oracle_sample(wl, tokens=tokens)
        total_flops += flops
        total_s += dt
        reps += 1
    return total_flops / total_s / 1e12, reps, desc, threads, total_s


def cpu_baseline(args, wl):
    """The oracle on the host cores: all cores (OpenMP quantizer, threaded BLAS), then one thread
    (a child process started with every thread pool at 1)."""
    value, reps, desc, threads, secs = oracle_rate(wl, 2048, CPU_BASELINE_SECONDS)
    out = {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{reps} repetitions of: {desc}", "seconds": round(secs, 3)}
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-single-thread", "--workload",
                            args.workload], env=env, capture_output=True, text=True, timeout=600)
        out["single_thread"] = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # the all-core figure stands on its own
        out["single_thread"] = {"error": f"{type(e).__name__}: {e}"}
    return out


def run_oracle_single_thread(args):
    import oracle
    oracle.build()
    oracle.set_threads(1)
    wl = WORKLOADS[args.workload]
    value, reps, desc, threads, secs = oracle_rate(wl, 512, 8.0)
    print(json.dumps({"value": round(value, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                      "sample": f"{reps} repetitions of: {desc}", "seconds": round(secs, 3)}), flush=True)


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    times, flops_all = [], 0
    desc = threads = None
    for i in range(args.warmup + args.steps):
        flops, dt, desc, threads = oracle_sample(wl, tokens=512)
        if i >= args.warmup:
            times.append(dt)
            flops_all = flops
    ms = 1e3 * sum(times) / len(times)
    value = flops_all / (ms * 1e-3) / 1e12
    out = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": wl["name"], "description": wl["desc"]},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)  # ~0.2 s timed: about ten clock samples
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="block3b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-single-thread", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--qshape", type=int, nargs=2, default=[16384, 16384], help="--part quantize_one: rows cols")
    ap.add_argument("--qform", choices=["row", "transposed", "dual"], default="dual")
    ap.add_argument("--qmode", choices=["rtn", "sr"], default="sr")
    ap.add_argument("--rank", type=int, default=64, help="--part branch_one / gemm_one: the branch rank")
    ap.add_argument("--gshape", type=int, nargs=3, default=[16384, 3072, 8192], help="--part gemm_one: M N K")
    ap.add_argument("--part", choices=["all", "step", "newton_schulz", "qadamw_v_codec", "lora_realign", "lora_cholqr", "quantize_sweep",
                             "gemm_sweep", "quantize_one", "branch_one", "gemm_one"], default="all",
                    help="run one optimizer-side measurement alone (prints its JSON object; for profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.oracle_single_thread:
        run_oracle_single_thread(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
