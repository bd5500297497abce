"""Benchmark: causal attention fwd+bwd (d20 shape) and KV-cache decode on B300.

One step = one pass of the whole hot path over the d20 workload
(B=32, T=2048, H=10, D=128): nc_attn_fwd (RoPE table, QK RMSNorm+RoPE
prologue, tcgen05 forward) then nc_attn_bwd (backward preprocess, tcgen05
key-side kernel with the fused dk epilogue, tcgen05 query-side kernel with
the fused dq epilogue).  Inputs are seeded synthetic bf16 Gaussians already
resident in HBM; q, k, v and dout together are 671 MB, more than the 126 MB
L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `value` is fwd+bwd TFLOP/s under the
algorithmic FLOP count (causal half of 2 matmuls forward, 5 backward).
Decode (32 streams, H=10, D=128, capacity 2048, seeded lengths) is timed too
and reported under "decode" in GB/s of algorithmic cache bytes.

--impl reference times the fp64 CPU oracle (the only other implementation
of this method there is) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# B300 datasheet figures (dense bf16 tensor throughput, HBM3e bandwidth): the
# second denominator the fractions are reported against
SPEC = {"bf16_tflops": 2250.0, "hbm_gbs": 7700.0}


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own batch: replicas process independent batches
    (weak scaling, no data-path collective); rank 0 keeps the workload's."""
    return seed + 1000 * rank


def job_throughput(ms_local: float, ws_n: int, flops_per_step: float, steps: int, device="cpu"):
    """(max over ranks of the timed region in ms, whole-job TFLOP/s): every
    rank ran `steps` steps of `flops_per_step`, and the job is as fast as its
    slowest rank.  Collective only when ws_n > 1 (NCCL on the GPUs, gloo in
    the CPU tests)."""
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if ws_n > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, ws_n * flops_per_step * steps / (ms_max * 1e-3) / 1e12


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms by a reader
    thread that stamps each line on arrival; summary() keeps the samples that
    arrived inside the window set by mark_start() / mark_end() (the timed
    region).  A timed region shorter than the sampling interval still gets
    the first sample that arrived after its end, so the record is never
    empty while nvidia-smi runs."""
    PERIOD_S = 0.02
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.samples = []  # (host time, line)
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.samples.append((time.time(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(int(self.PERIOD_S * 1000))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        # wait for one sample that covers the end of the region
        deadline = self.t1 + 0.5
        while self.proc is not None and time.time() < deadline:
            if any(t >= self.t1 for t, _ in self.samples):
                break
            time.sleep(0.005)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # a sample describes the sampling period before it arrived
        lo = (self.t0 or 0.0) + self.PERIOD_S
        hi = (self.t1 or float("inf")) + self.PERIOD_S
        window = [l for t, l in self.samples if lo <= t <= hi]
        if not window:
            after = [l for t, l in self.samples if t >= (self.t1 or 0.0)]
            window = after[:1]
        for l in window:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our impl -----

def bench_ours(args, ws_n, rank, local):
    import causal_attention_rope_nc_b300 as nc
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.ATTN_WORKLOADS[args.workload]
    B, T, H, D = w.B, w.T, w.H, w.D
    eps, base = workloads.EPS, workloads.ROPE_BASE
    # weak scaling: every rank runs its own d20 batch (seed offset by rank)
    q, k, v, dout = workloads.attn_inputs(B, T, H, D, rank_seed(w.seed, rank))
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dout))
    out = torch.empty_like(qd)
    qh, kh = torch.empty_like(qd, dtype=torch.float16), torch.empty_like(kd, dtype=torch.float16)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_f = nc.new_workspace(nc.NC_OP_FWD, B, T, H, D, dev)
    ws_b = nc.new_workspace(nc.NC_OP_BWD, B, T, H, D, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        nc.nc_attn_fwd(qd, kd, vd, None, out, lse, qh, kh, None, ws_f, eps, base, stream)
        nc.nc_attn_bwd(qd, kd, vd, None, out, lse, qh, kh, dod, dq, dk, dv, ws_b, eps, base, stream)

    def barrier():
        if ws_n > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if nc.device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    # ---- timed region: K steps, per-kernel events on the launch stream ----
    nc.nc_profile_read()  # clear
    nc.nc_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.5)  # let nvidia-smi start sampling
        barrier()
        torch.cuda.synchronize(dev)
        clk.mark_start()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
        barrier()
        time.sleep(0.3)  # the sample covering the end of the region
    nc.nc_profile_enable(False)
    ms_total = ev0.elapsed_time(ev1)
    kern = nc.nc_profile_read()
    kern_kernels = dict(nc.last_profile_kernels)  # kernel launches per step name
    if nc.device_status() != 0:
        raise RuntimeError("device status set during the timed region")

    # max over ranks
    flops = w.fwd_bwd_flops()
    ms_max, value = job_throughput(ms_total, ws_n, flops, args.steps, dev)
    ms_per_step = ms_max / args.steps

    # ---- decode (same rank, own timing; L2 flushed between calls) ----
    dec = e2e = win = pre = gqa = fp8 = None
    if not args.no_extras:
        dec = bench_decode(nc, dev, args, rank)
        # ---- the short-window layers: the same step with W = T / 4 ----
        win = bench_window(nc, dev, args, w, qd, kd, vd, dod, out, lse, qh, kh, dq, dk, dv, ws_f, ws_b, stream)
        win["decode"] = bench_decode(nc, dev, args, rank, window=w.T // 4)
        # ---- a 512-token chunk appended to every stream's cache ----
        pre = bench_prefill(nc, dev, args)
        # ---- grouped-query attention: 2 key/value heads for the 10 query heads ----
        gqa = bench_gqa(nc, dev, args, w, GQA_KV_HEADS)
        gqa["decode"] = bench_decode(nc, dev, args, rank, kv_heads=GQA_KV_HEADS)
        # ---- the FP8 forward on the same inputs ----
        fp8 = bench_fp8(nc, dev, args, w, qd, kd, vd, stream)
        # ---- end to end through the public API with host buffers ----
        e2e = bench_e2e(nc, dev, args, w, q, k, v, dout, ws_f, ws_b)

    if rank != 0:
        return None
    pk, pk_kind = peaks()
    launches = sum(kern_kernels.get(k_, n) for k_, (n, _) in kern.items())
    # dominant kernel by total time
    name, (n_l, tot) = max(kern.items(), key=lambda kv: kv[1][1])
    per_launch_ms = tot / max(n_l, 1)
    # algorithmic tensor FLOPs per launch (the causal half of each matmul):
    # forward 2 matmuls; the backward's 5 are split between the key-side kernel
    # (S^T, dP^T, dV, dK) and the query-side kernel (dQ; its S and dP are
    # recomputation, not counted)
    alg = {"attn_fwd": w.fwd_flops(), "attn_bwd_dkdv": 2.0 * w.fwd_flops(),
           "attn_bwd_dq": 0.5 * w.fwd_flops()}
    timed_s = ms_total * 1e-3
    peak_t = pk["bf16_tflops_sustained"] if timed_s > 2.0 else pk["bf16_tflops"]
    roof = None
    if name in alg:
        ach = alg[name] / (per_launch_ms * 1e-3) / 1e12
        tr = DRAM_TRAFFIC.get(name) if args.workload == "d20" else None
        roof = {"kernel": name, "bound": "tensor", "achieved": round(ach, 1), "peak": peak_t,
                "unit": "TFLOP/s", "frac": round(ach / peak_t, 4), "traffic": tr,
                "peak_kind": f"{pk_kind} {'sustained' if timed_s > 2.0 else 'burst'} bf16"}
    kernels = {k_: {"launches": n_, "avg_us": round(1e3 * t_ / max(n_, 1), 2),
                    "share": round(t_ / max(sum(x[1] for x in kern.values()), 1e-9), 4)}
               for k_, (n_, t_) in sorted(kern.items(), key=lambda kv: -kv[1][1])}
    for k_ in alg:
        if k_ in kern:
            n_, t_ = kern[k_]
            kernels[k_]["tflops"] = round(alg[k_] / (t_ / n_ * 1e-3) / 1e12, 1)
            kernels[k_]["frac_of_peak"] = round(kernels[k_]["tflops"] / pk["bf16_tflops"], 4)
    line = {
        "metric": "causal attn fwd+bwd TFLOP/s (% bf16 peak) at d20; decode GB/s (% HBM peak)",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, d20 shapes)",
        "config": {"workload": f"{w.name} block attention fwd+bwd: B={B} T={T} H={H} D={D}, causal, "
                               "QK RMSNorm eps=1e-6, RoPE base 10000",
                   "B": B, "T": T, "H": H, "D": D, "parallelism": f"replicas x{ws_n} (batch shards)",
                   "l2": "inputs 671 MB > 126 MB L2; no flush between steps"},
        "frac_of_peak": round(value / ws_n / pk["bf16_tflops"], 4),
        "frac_of_spec_peak": round(value / ws_n / SPEC["bf16_tflops"], 4),
        "peak_kind": pk_kind,
        "tokens_per_s": round(ws_n * B * T * args.steps / (ms_max * 1e-3), 1),
        "roofline": roof,
        "kernels": kernels,
        "decode": dec,
        "window": win,
        "prefill": pre,
        "gqa": gqa,
        "fp8": fp8,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    return line


# DRAM bytes (read + write) of one launch of a kernel at the d20 workload,
# from one ncu capture of the current kernel (dram__bytes_read.sum +
# dram__bytes_write.sum, summarised under profiles/ with its command).
# Must go back to None whenever that kernel's code changes.
DRAM_TRAFFIC = {"attn_bwd_dkdv": 881.08e6 + 1.71e9, "attn_bwd_dq": 1.79e9 + 157.83e6,
                "attn_fwd": 505.57e6 + 145.83e6}
# The same for the decode kernels at the d20 decode workload (plain multi-head
# attention, and 2 key/value heads).
DECODE_TRAFFIC = {"mha": 176.36e6 + 1.46e6, "gqa2": 35.88e6 + 0.0}


def band_pairs(T, W):
    """Score pairs per (b, h) under a sliding window W, in the convention of
    the causal count (T^2/2 = the area under the diagonal): T*W - W^2/2."""
    W = min(W, T)
    return T * W - W * W / 2.0


def bench_window(nc, dev, args, w, qd, kd, vd, dod, out, lse, qh, kh, dq, dk, dv, ws_f, ws_b, stream):
    """The fwd+bwd step through the sliding-window calls with W = T/4 (the
    short-window layers of the pages' SSSL pattern), timed like the main step;
    algorithmic FLOPs over the band only (tiles outside it are skipped)."""
    W = w.T // 4
    eps, base = workloads.EPS, workloads.ROPE_BASE

    def step():
        nc.nc_attn_fwd_ex(qd, kd, vd, None, out, lse, qh, kh, None, ws_f, eps, base, W, stream)
        nc.nc_attn_bwd_ex(qd, kd, vd, None, out, lse, qh, kh, dod, dq, dk, dv, ws_b, eps, base, W, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 5)
    nc.nc_profile_read()
    nc.nc_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    nc.nc_profile_enable(False)
    kern = nc.nc_profile_read()
    if nc.device_status() != 0:
        raise RuntimeError("device status set during the window leg")
    ms = e0.elapsed_time(e1) / steps
    fwd = 4.0 * w.B * w.H * w.D * band_pairs(w.T, W)
    pk, _ = peaks()
    alg = {"attn_fwd": fwd, "attn_bwd_dkdv": 2.0 * fwd, "attn_bwd_dq": 0.5 * fwd}
    kernels = {}
    for k_, (n_, t_) in sorted(kern.items(), key=lambda kv: -kv[1][1]):
        kernels[k_] = {"avg_us": round(1e3 * t_ / max(n_, 1), 2)}
        if k_ in alg:
            tf = alg[k_] / (t_ / n_ * 1e-3) / 1e12
            kernels[k_]["tflops"] = round(tf, 1)
            kernels[k_]["frac_of_peak"] = round(tf / pk["bf16_tflops"], 4)
    return {"workload": f"{w.name} fwd+bwd with a sliding window W = T/4 = {W}", "W": W,
            "ms_per_step": round(ms, 4), "value": round(3.5 * fwd / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "flops_per_step": 3.5 * fwd, "kernels": kernels}


GQA_KV_HEADS = 2  # key/value heads of the grouped-query leg (d20: groups of 5 query heads)


def bench_gqa(nc, dev, args, w, Hkv):
    """The fwd+bwd step through the grouped-query calls with Hkv key/value
    heads for the workload's H query heads, timed like the main step.  The
    score matmuls are those of the multi-head step (every query head still
    meets every visible key), so the algorithmic FLOPs are the same."""
    eps, base = workloads.EPS, workloads.ROPE_BASE
    q, k, v, dout = workloads.attn_inputs(w.B, w.T, w.H, w.D, w.seed, kv_heads=Hkv)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dout))
    del q, k, v, dout
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    qh = torch.empty_like(qd, dtype=torch.float16)
    kh = torch.empty_like(kd, dtype=torch.float16)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_f = nc.new_workspace(nc.NC_OP_FWD, w.B, w.T, w.H, w.D, dev)
    ws_b = nc.new_workspace(nc.NC_OP_BWD, w.B, w.T, w.H, w.D, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        nc.nc_attn_fwd_ex(qd, kd, vd, None, out, lse, qh, kh, None, ws_f, eps, base, 0, stream)
        nc.nc_attn_bwd_ex(qd, kd, vd, None, out, lse, qh, kh, dod, dq, dk, dv, ws_b, eps, base, 0, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 5)
    nc.nc_profile_read()
    nc.nc_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    nc.nc_profile_enable(False)
    kern = nc.nc_profile_read()
    if nc.device_status() != 0:
        raise RuntimeError("device status set during the grouped-query leg")
    ms = e0.elapsed_time(e1) / steps
    fwd = w.fwd_flops()
    pk, _ = peaks()
    alg = {"attn_fwd": fwd, "attn_bwd_dkdv": 2.0 * fwd, "attn_bwd_dq": 0.5 * fwd}
    kernels = {}
    for k_, (n_, t_) in sorted(kern.items(), key=lambda kv: -kv[1][1]):
        kernels[k_] = {"launches_per_step": n_ // steps, "avg_us": round(1e3 * t_ / max(n_, 1), 2)}
        if k_ in alg:
            tf = alg[k_] / (t_ / n_ * 1e-3) / 1e12
            kernels[k_]["tflops"] = round(tf, 1)
            kernels[k_]["frac_of_peak"] = round(tf / pk["bf16_tflops"], 4)
    return {"workload": f"{w.name} fwd+bwd, grouped-query: H={w.H} query heads, {Hkv} key/value heads",
            "kv_heads": Hkv, "ms_per_step": round(ms, 4), "value": round(3.5 * fwd / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "kernels": kernels}


def bench_prefill(nc, dev, args, B=32, H=10, D=128, Tcap=2048, C=512):
    """nc_attn_prefill of a C-token chunk per stream at position Tcap - C of a
    full cache (the d20 decode shapes): prologue + attention of the chunk over
    its cache prefix.  FLOPs: 4 D per visible score pair, pairs counted like the
    causal forward (C (Tcap - C) + C^2/2 per (b, h))."""
    eps, base = workloads.EPS, workloads.ROPE_BASE
    s0 = Tcap - C
    start_t, q, k_raw, v = workloads.prefill_inputs(B, C, H, D, Tcap, seed=5, start=[s0] * B)
    kcache = nc.qk_norm_rope(k_raw.to(dev), eps=eps, rope_base=base)
    vcache = v.to(dev)
    qd = q.to(dev)
    kc = k_raw[:, s0:].contiguous().to(dev)
    vc = v[:, s0:].contiguous().to(dev)
    st = start_t.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, C), dtype=torch.float32, device=dev)
    ws = nc.new_workspace(nc.NC_OP_PREFILL, B, C, H, D, dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        nc.nc_attn_prefill(qd, kc, vc, st, kcache, vcache, out, lse, ws, eps, base, 0, stream)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 5)
    nc.nc_profile_read()
    nc.nc_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    nc.nc_profile_enable(False)
    kern = nc.nc_profile_read()
    if nc.device_status() != 0:
        raise RuntimeError("device status set during the prefill leg")
    ms = e0.elapsed_time(e1) / steps
    flops = 4.0 * B * H * D * (C * s0 + C * C / 2.0)
    pk, _ = peaks()
    kernels = {k_: {"avg_us": round(1e3 * t_ / max(n_, 1), 2)} for k_, (n_, t_) in kern.items()}
    if "attn_prefill" in kern:
        n_, t_ = kern["attn_prefill"]
        tf = flops / (t_ / n_ * 1e-3) / 1e12
        kernels["attn_prefill"]["tflops"] = round(tf, 1)
        kernels["attn_prefill"]["frac_of_peak"] = round(tf / pk["bf16_tflops"], 4)
    return {"workload": f"chunk prefill: {B} streams, H={H}, D={D}, {C} new tokens at position {s0} of a "
                        f"{Tcap}-slot cache", "us": round(ms * 1e3, 2),
            "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "tokens_per_s": round(B * C / (ms * 1e-3), 1), "kernels": kernels}


def bench_fp8(nc, dev, args, w, qd, kd, vd, stream):
    """nc_attn_fwd_fp8 on the d20 workload: RoPE table, QK RMSNorm+RoPE into
    E4M3, value quantisation, and the E4M3 forward (two passes over the keys:
    the row maximum, then P and PV).  FLOPs: the forward's algorithmic count;
    the kernel's peak is the fp8 dense rate, twice the measured bf16 one (the
    datasheet ratio: 4.5 against 2.25 PFLOP/s)."""
    eps, base = workloads.EPS, workloads.ROPE_BASE
    B, T, H, D = w.B, w.T, w.H, w.D
    out = torch.empty_like(qd)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    ws = nc.new_workspace(nc.NC_OP_FWD_FP8, B, T, H, D, dev)

    def call():
        nc.nc_attn_fwd_fp8(qd, kd, vd, None, out, lse, ws, eps, base, 0, stream)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 5)
    nc.nc_profile_read()
    nc.nc_profile_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    nc.nc_profile_enable(False)
    kern = nc.nc_profile_read()
    if nc.device_status() != 0:
        raise RuntimeError("device status set during the fp8 leg")
    ms = e0.elapsed_time(e1) / steps
    flops = w.fwd_flops()
    pk, _ = peaks()
    peak8 = 2.0 * pk["bf16_tflops"]
    kernels = {k_: {"avg_us": round(1e3 * t_ / max(n_, 1), 2)} for k_, (n_, t_) in kern.items()}
    if "attn_fwd_fp8" in kern:
        n_, t_ = kern["attn_fwd_fp8"]
        tf = flops / (t_ / n_ * 1e-3) / 1e12
        kernels["attn_fwd_fp8"]["tflops"] = round(tf, 1)
        kernels["attn_fwd_fp8"]["frac_of_fp8_peak"] = round(tf / peak8, 4)
    return {"workload": f"{w.name} forward with E4M3 products (qhat, khat at 2^5; v per head; P at 2^8)",
            "ms_per_call": round(ms, 4), "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "fp8_peak_tflops": round(peak8, 1), "kernels": kernels}


def bench_decode(nc, dev, args, rank, window=0, kv_heads=None):
    w = workloads.D20_DECODE
    lens, q, k_raw, v = workloads.decode_workload_inputs(w, kv_heads=kv_heads)
    kcache = nc.qk_norm_rope(k_raw.to(dev), eps=workloads.EPS, rope_base=workloads.ROPE_BASE)
    vcache = v.to(dev)
    qd, lens_d = q.to(dev), lens.to(dev)
    out = torch.empty((w.B, w.H, w.D), dtype=torch.bfloat16, device=dev)
    ws = nc.new_workspace(nc.NC_OP_DECODE, w.B, w.Tcap, w.H, w.D, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        if window or kv_heads:
            nc.nc_attn_decode_ex(qd, None, None, kcache, vcache, lens_d, out, ws, workloads.EPS,
                                 workloads.ROPE_BASE, window, stream)
        else:
            nc.nc_attn_decode(qd, None, None, kcache, vcache, lens_d, out, ws, workloads.EPS,
                              workloads.ROPE_BASE, stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(max(args.steps, 5)):
        # evict the cache and the previous call's lines from L2: write a buffer
        # larger than L2, then read it back, so that no dirty line of the flush
        # is still being written back to HBM while the timed call runs
        flush.zero_()
        flush.view(torch.int32).sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    if nc.device_status() != 0:
        raise RuntimeError("device status set during decode")
    byt = workloads.decode_bytes(torch.clamp(lens, max=window) if window else lens, w.H, w.D, kv_heads)
    ms = statistics.median(times)
    pk, kind = peaks()
    gbs = byt / (ms * 1e-3) / 1e9
    name = "d20 decode: 32 streams, H=10, D=128, cache capacity 2048, lens ~ U[1,2048] seed 4"
    if window:
        name += f", sliding window W = {window} (the last W slots)"
    if kv_heads:
        name += f", {kv_heads} key/value heads (grouped-query)"
    return {"workload": name,
            "bytes": byt, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm_gbs"], 4),
                         "traffic": None if window else DECODE_TRAFFIC.get("gqa2" if kv_heads == 2 else
                                                                       "mha" if not kv_heads else None),
                         "frac_of_spec": round(gbs / SPEC["hbm_gbs"], 4)},
            "l2": "256 MB buffer written, then read, between calls", "tokens_per_s": round(w.B / (ms * 1e-3), 1)}


def bench_e2e(nc, dev, args, w, q, k, v, dout, ws_f, ws_b):
    """fwd+bwd through the public API with pinned host buffers: every step
    copies its q, k, v, dout host->device and its dq, dk, dv device->host
    inside the timed region.  Steps are pipelined over two device buffer sets
    and three streams (host->device copies, compute, device->host copies), so
    one step's copies overlap its neighbours' compute and the other copy
    direction; the region ends when the last step's results are on the host."""
    hq, hk, hv, hdo = (x.pin_memory() for x in (q, k, v, dout))
    hout = [[torch.empty_like(hq).pin_memory() for _ in range(3)] for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def dbuf(dtype=torch.bfloat16):
        return torch.empty(q.shape, dtype=dtype, device=dev)

    ins = [[dbuf() for _ in range(4)] for _ in range(2)]    # q, k, v, dout
    outs = [[dbuf() for _ in range(3)] for _ in range(2)]   # dq, dk, dv
    out = dbuf()
    qh, kh = dbuf(torch.float16), dbuf(torch.float16)
    lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "comp", "out")}
    used = [False, False]

    def step(i):
        j = i % 2
        qd_, kd_, vd_, do_ = ins[j]
        dq_, dk_, dv_ = outs[j]
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev["comp"][j])  # step i-2 has finished reading these inputs
            for d_, h_ in ((qd_, hq), (kd_, hk), (vd_, hv), (do_, hdo)):
                d_.copy_(h_, non_blocking=True)
            ev["in"][j].record(s_in)
        comp.wait_event(ev["in"][j])
        if used[j]:
            comp.wait_event(ev["out"][j])  # step i-2's results have left these buffers
        nc.nc_attn_fwd(qd_, kd_, vd_, None, out, lse, qh, kh, None, ws_f, workloads.EPS,
                       workloads.ROPE_BASE, comp)
        nc.nc_attn_bwd(qd_, kd_, vd_, None, out, lse, qh, kh, do_, dq_, dk_, dv_, ws_b, workloads.EPS,
                       workloads.ROPE_BASE, comp)
        ev["comp"][j].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][j])
            for h_, d_ in zip(hout[j], (dq_, dk_, dv_)):
                h_.copy_(d_, non_blocking=True)
            ev["out"][j].record(s_out)
        used[j] = True

    def run(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        s_in.wait_event(e0)
        for i in range(n):
            step(i)
        for j in range(2):
            if used[j]:
                comp.wait_event(ev["out"][j])
        e1.record(comp)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    run(3)
    n = max(3, min(args.steps, 10))
    ms = run(n) / n
    if nc.device_status() != 0:
        raise RuntimeError("device status set during the end-to-end leg")
    # the last step's results arrived intact
    assert torch.equal(hout[(n - 1) % 2][0], outs[(n - 1) % 2][0].cpu())
    nbytes = q.numel() * 2
    return {"value": round(w.fwd_bwd_flops() / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": 4 * nbytes, "d2h_bytes_per_step": 3 * nbytes, "ms_per_step": round(ms, 3),
            "steps": n, "pipeline": "2 buffer sets; H2D, compute and D2H on separate streams"}


# ------------------------------------------------------ CPU oracle legs ----

def oracle_sample(n_slices: int):
    """Time the fp64 oracle on `n_slices` whole (b, h) slices of the d20
    workload (fwd + bwd); returns (TFLOP/s, seconds, threads)."""
    import oracle
    w = workloads.D20
    q, k, v, dout = workloads.workload_inputs(w)
    picks = [(i % w.B, (i * 7) % w.H) for i in range(n_slices)]
    qs = torch.stack([q[b, :, h] for b, h in picks]).unsqueeze(2)
    ks = torch.stack([k[b, :, h] for b, h in picks]).unsqueeze(2)
    vs = torch.stack([v[b, :, h] for b, h in picks]).unsqueeze(2)
    ds = torch.stack([dout[b, :, h] for b, h in picks]).unsqueeze(2)
    t0 = time.perf_counter()
    oracle.attn_fwd(qs, ks, vs, eps=workloads.EPS, base=workloads.ROPE_BASE)
    oracle.attn_bwd(qs, ks, vs, ds, eps=workloads.EPS, base=workloads.ROPE_BASE)
    dt = time.perf_counter() - t0
    flops = w.fwd_bwd_flops() * n_slices / (w.B * w.H)
    return flops / dt / 1e12, dt


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline():
    cores = cpu_cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    n = min(cores, 64)
    tf, dt = oracle_sample(n)
    return {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} whole (b,h) slices of d20 (T=2048, D=128) fwd+bwd, fp64, {dt:.1f} s"}


def bench_reference(args, ws_n, rank):
    if rank != 0:
        return None
    cores = cpu_cores()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    import oracle
    oracle.build()
    # one slice costs ~5 s on one core; keep the whole run to a few minutes
    budget = 150.0 / max(args.steps + args.warmup, 1)
    n = min(cores, 64) if budget >= 12.0 else 1
    for _ in range(args.warmup):
        oracle_sample(n)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        tf, dt = oracle_sample(n)
        vals.append(tf)
        secs += dt
    value = args.steps / sum(1.0 / x for x in vals)
    return {
        "impl": "reference",
        "metric": "causal attn fwd+bwd TFLOP/s (% bf16 peak) at d20; decode GB/s (% HBM peak)",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16, d20 shapes)",
        "config": {"workload": "d20 block attention fwd+bwd: B=32 T=2048 H=10 D=128, causal, "
                               "QK RMSNorm eps=1e-6, RoPE base 10000", "B": 32, "T": 2048, "H": 10, "D": 128},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} whole (b,h) slice(s) of d20 per step, fp64 C oracle"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def bench_leg(args):
    """One side leg alone (for profiling a single kernel family under ncu):
    prints that leg's JSON object and nothing else."""
    import causal_attention_rope_nc_b300 as nc
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.leg == "decode":
        res = bench_decode(nc, dev, args, 0)
    elif args.leg == "decode-gqa":
        res = bench_decode(nc, dev, args, 0, kv_heads=GQA_KV_HEADS)
    elif args.leg == "decode-window":
        res = bench_decode(nc, dev, args, 0, window=workloads.D20.T // 4)
    elif args.leg == "window":
        w = workloads.ATTN_WORKLOADS[args.workload]
        q, k, v, dout = workloads.attn_inputs(w.B, w.T, w.H, w.D, w.seed)
        qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dout))
        out = torch.empty_like(qd)
        qh, kh = torch.empty_like(qd, dtype=torch.float16), torch.empty_like(kd, dtype=torch.float16)
        lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws_f = nc.new_workspace(nc.NC_OP_FWD, w.B, w.T, w.H, w.D, dev)
        ws_b = nc.new_workspace(nc.NC_OP_BWD, w.B, w.T, w.H, w.D, dev)
        res = bench_window(nc, dev, args, w, qd, kd, vd, dod, out, lse, qh, kh, dq, dk, dv, ws_f, ws_b,
                           torch.cuda.current_stream(dev))
    else:  # fp8
        w = workloads.ATTN_WORKLOADS[args.workload]
        q, k, v, _ = workloads.attn_inputs(w.B, w.T, w.H, w.D, w.seed)
        qd, kd, vd = (x.to(dev) for x in (q, k, v))
        res = bench_fp8(nc, dev, args, w, qd, kd, vd, torch.cuda.current_stream(dev))
    res["leg"] = args.leg
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=sorted(workloads.ATTN_WORKLOADS), default="d20",
                    help="fwd+bwd shape (the headline metric is quoted on d20; others for profiling)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the decode and end-to-end legs (short runs under a profiler)")
    ap.add_argument("--leg", choices=["all", "decode", "decode-gqa", "decode-window", "window", "fp8"], default="all",
                    help="run one side leg alone and print its object (profiling); default: the full line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.leg != "all":
        bench_leg(args)
        return
    ws_n, rank, local = dist_env()
    if args.impl == "reference":
        line = bench_reference(args, ws_n, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if ws_n > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        line = bench_ours(args, ws_n, rank, local)
        if line is not None:
            if ws_n == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline()
            print(json.dumps(line), flush=True)
    finally:
        if ws_n > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
