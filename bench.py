#!/usr/bin/env python3
"""Benchmark: exact fused attention forward on GB300, bf16, d=128, causal and full.

One step = one forward of each of the two bf16 d=128 workloads the headline metric
names: B=2,H=8,Nq=Nk=4096 full and B=2,H=8,Nq=Nk=8192 causal (synthetic N(0,1) inputs,
scale 1/sqrt(128)). value = their FLOPs (4*B*H*Nq*Nk*d, halved when causal) divided by
the summed device time of the two launches (CUDA events on the launching stream, L2
flushed by a 256 MiB write before every launch). Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (the only reference this method has) on
the host cores, on bounded row samples of the same two workloads.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (bf16, causal & full) and % of GB300 dense tensor peak"
UNIT = "TFLOPS"
WORKLOADS = ("b2h8_n4096_d128_full", "b2h8_n8192_d128_causal")
DOMINANT = "b2h8_n8192_d128_causal"
FP8_WORKLOADS = ("b2h8_n4096_d128_full_fp8", "b2h8_n8192_d128_causal_fp8")
FP8_DOMINANT = "b2h8_n8192_d128_causal_fp8"
FP8_OVER_BF16 = 2.0  # nominal dense E4M3 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)
FLUSH_BYTES = 256 << 20
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCES = ("exact_attention_forward_02_gb300/csrc/fa_fwd_kernel.cuh",
                  "exact_attention_forward_02_gb300/csrc/sm103_ptx.cuh",
                  "exact_attention_forward_02_gb300/csrc/philox.cuh")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_over_ranks(values):
    """Element-wise maximum of `values` over all ranks (identity on one process)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(flops_per_rank_step: float, world: int, step_ms_max: float) -> float:
    """Replicas: every rank runs the same step; the job's rate is all ranks' FLOPs over the
    slowest rank's step time."""
    return world * flops_per_rank_step / (step_ms_max * 1e-3) / 1e12


EX2_PER_CLK_PER_SM = 32  # ex2.approx rate measured on the GB300 (lanes per clock per SM)


def visible_scores(w) -> int:
    """Scores that take an exponential: one per (row, visible key); causal rows see keys
    j <= i (top-left), so row i has min(i + 1, Nk) of them."""
    if not w.causal:
        return w.B * w.H * w.Nq * w.Nk
    n = min(w.Nq, w.Nk)
    per_head = n * (n + 1) // 2 + (w.Nq - n) * w.Nk
    return w.B * w.H * per_head


def sfu_bound(w, ms: float, sms: int, sm_mhz: float, counters=None) -> dict:
    """The secondary bound of the forward pass: its exponentials. One ex2 per visible score
    runs on the special-function (XU) pipe, whose measured rate is 32 lanes per clock per SM.
    Where the committed ncu record of this kernel holds its XU warp-instruction count
    (sm__inst_executed_pipe_xu.sum), that count is given beside the ex2 warp instructions
    the scores need (ex2_count / 32): the ex2s are nearly all of the pipe's work."""
    n = visible_scores(w)
    peak = EX2_PER_CLK_PER_SM * sms * sm_mhz * 1e6
    achieved = n / (ms * 1e-3)
    out = {"bound": "sfu", "ex2_count": n, "achieved_ex2_per_s": achieved, "peak_ex2_per_s": peak,
           "frac": round(achieved / peak, 4),
           "peak_source": f"{EX2_PER_CLK_PER_SM} ex2/clk/SM x {sms} SMs x {sm_mhz:g} MHz (median SM clock "
                          "sampled in the timed region)"}
    if counters and counters.get("xu_inst"):
        out["xu_inst_counted"] = counters["xu_inst"]
        out["xu_inst_per_ex2_warp_inst"] = round(counters["xu_inst"] / (n / 32), 4)
    return out


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_counters(workload, entry: str):
    """The committed ncu counters of the kernel that runs `workload` through `entry`
    ("fa_fwd" or "fa_fwd_ws"), only while the kernel source is the one they were taken on."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256") != kernel_source_hash():
            return None
        k = rec["kernels"][workload]
        return k if k.get("entry") == entry else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons around the timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None

    def wait_first_sample(self, timeout=5.0):
        end = time.time() + timeout
        while self.proc and time.time() < end:
            if os.path.getsize(self.f.name) > 0:
                return
            time.sleep(0.05)

    def start(self):
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        time.sleep(0.15)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.f.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 10:
                        continue
                    rows.append(parts)
        finally:
            os.unlink(self.f.name)
        # keep the samples taken inside the timed region (plus one sampling period)
        import datetime
        inside = []
        for r in rows:
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if self.t0 is not None and self.t0 - 0.1 <= ts <= (self.t1 or ts) + 0.1:
                inside.append(r)
        if inside:
            rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside),
                "power_w_max": max((float(r[4]) for r in rows if r[4].replace(".", "").isdigit()), default=None)}


# ----------------------------------------------------------------------------- ours
def run_ours(args):
    import torch
    import torch.distributed as dist

    import exact_attention_forward_02_gb300 as fa
    import gen

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)

    allw = {**gen.WORKLOADS, **gen.FP8_WORKLOADS}
    names = (tuple(args.workloads.split(",")) if args.workloads else
             FP8_WORKLOADS if args.fp8 else WORKLOADS)
    wl = [allw[n] for n in names]
    host = {}
    devbuf = {}
    fp8ws = {}
    for w in wl:
        q, k, v = gen.make_qkv(w)
        host[w.name] = [t.pin_memory() for t in (q, k, v)]
        qd, kd, vd = (t.to(dev) for t in (q, k, v))
        O = torch.empty((w.B, w.H, w.Nq, w.d), dtype=gen.torch_dtype(w.out_dtype), device=dev)
        if w.dtype == gen.FP8:
            fp8ws[w.name] = torch.empty(fa.fa_fwd_fp8_workspace_bytes(w.B, w.H, w.Nk, w.d),
                                        dtype=torch.uint8, device=dev)
        L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
        # stream-K workspace for full attention (zero-filled once; calls keep it zeroed):
        # --sched auto calls fa_fwd_ws wherever the library asks for one (full attention
        # whose work items do not fill whole waves of SMs), --sched plain calls fa_fwd
        nws = (fa.fa_fwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, w.causal)
               if args.sched != "plain" and w.dtype != gen.FP8 and args.dropout == 0 else 0)
        wsp = torch.zeros(max(nws, 256), dtype=torch.uint8, device=dev) if nws else None
        devbuf[w.name] = (qd, kd, vd, O, L, wsp)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    drop_offset = [0]

    def launch(w):
        qd, kd, vd, O, L, wsp = devbuf[w.name]
        dt = fa.FA_BF16 if w.out_dtype == gen.BF16 else fa.FA_F16
        if w.dtype == gen.FP8:
            wsf = fp8ws[w.name]
            rc = fa.fa_fwd_fp8(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(),
                               L.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                               1.0, 1.0, 1.0, dt, wsf.data_ptr(), wsf.numel(), sp)
        elif args.dropout > 0:
            # a fresh mask per call: the offset advances like a training loop's would
            drop_offset[0] += 1
            rc = fa.fa_fwd_dropout(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(),
                                   L.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt,
                                   args.dropout, 1234, drop_offset[0], sp)
        elif wsp is None:
            rc = fa.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(), L.data_ptr(),
                           w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt, sp)
        else:
            rc = fa.fa_fwd_ws(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), O.data_ptr(),
                              L.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt,
                              wsp.data_ptr(), wsp.numel(), sp)
        if rc != 0:
            raise fa.FAError(rc)

    fa.fa_clear_status()
    # warm-up
    for _ in range(args.warmup):
        for w in wl:
            flush.zero_()
            launch(w)
    torch.cuda.synchronize(dev)

    n = args.steps
    ev = {w.name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)] for w in wl}
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.wait_first_sample()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = fa.fa_num_kernel_launches()
    if clocks:
        clocks.start()
    t_wall0 = time.perf_counter()
    for i in range(n):
        for w in wl:
            flush.zero_()
            a, b = ev[w.name][i]
            a.record(stream)
            launch(w)
            b.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if ws > 1:
        dist.barrier()
    if clocks:
        clocks.stop()
    launches = fa.fa_num_kernel_launches() - launches0
    status = fa.fa_last_status()
    if status != 0:
        raise fa.FAError(status, "device status")

    per = {w.name: [a.elapsed_time(b) for a, b in ev[w.name]] for w in wl}  # ms
    step_ms = sum(statistics.fmean(per[w.name]) for w in wl)
    flops_step = sum(w.flops for w in wl)

    # ---- end to end through the C ABI with host buffers (fa_fwd_host): every step copies
    # Q, K, V from pinned host memory and O, L back to pinned host memory, overlapped with
    # the computation by the library's chunked pipeline (the FP8, dropout and stream-K
    # variants keep the plain sequence: copy in, launch, copy out)
    ne2e = max(3, min(n, 50))
    pin_out = {w.name: (torch.empty((w.B, w.H, w.Nq, w.d), dtype=gen.torch_dtype(w.out_dtype)).pin_memory(),
                        torch.empty((w.B, w.H, w.Nq), dtype=torch.float32).pin_memory()) for w in wl}
    h2d = sum(t.numel() * t.element_size() for w in wl for t in host[w.name])
    d2h = sum(t.numel() * t.element_size() for w in wl for t in pin_out[w.name])
    use_host_api = not (args.fp8 or args.dropout > 0)
    host_ws = {}
    if use_host_api:
        for w in wl:
            nb = fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
            host_ws[w.name] = torch.empty(nb, dtype=torch.uint8, device=dev)

    # one caller stream per workload, so that the two calls' pipelines overlap; the step
    # still ends with both results in host memory
    e2e_streams = [torch.cuda.Stream(dev) for _ in wl]

    # the calls are queued in descending order of their last chunk's cost, so that the one
    # whose last chunk finishes soonest after its copy-in (full attention: no long causal
    # rows) ends the step
    e2e_order = sorted(range(len(wl)), key=lambda i: not wl[i].causal)

    def e2e_step():
        for wi in e2e_order:
            w = wl[wi]
            po, pl = pin_out[w.name]
            if use_host_api:
                hq, hk, hv = host[w.name]
                wsh = host_ws[w.name]
                rc = fa.fa_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), po.data_ptr(),
                                    pl.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal,
                                    fa.FA_BF16 if w.out_dtype == gen.BF16 else fa.FA_F16,
                                    wsh.data_ptr(), wsh.numel(),
                                    ctypes.c_void_p(e2e_streams[wi].cuda_stream))
                if rc != 0:
                    raise fa.FAError(rc, "fa_fwd_host")
            else:
                qd, kd, vd, O, L, _ = devbuf[w.name]
                for dst, src in zip((qd, kd, vd), host[w.name]):
                    dst.copy_(src, non_blocking=True)
                launch(w)
                po.copy_(O, non_blocking=True)
                pl.copy_(L, non_blocking=True)
        torch.cuda.synchronize(dev)

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(ne2e):
        e2e_step()
    e2e_s = time.perf_counter() - t0

    # ---- max over ranks
    step_ms_max, e2e_ms_max, wall_max = reduce_max_over_ranks([step_ms, e2e_s / ne2e * 1e3, t_wall])

    if rank == 0:
        peak, peak_sus, peak_kind = peaks()
        dom_pref = FP8_DOMINANT if args.fp8 else DOMINANT
        dominant = dom_pref if dom_pref in per else max(per, key=lambda n: statistics.fmean(per[n]))
        wd = allw[dominant]
        if wd.dtype == gen.FP8:  # the E4M3 contraction's own peak: measured bf16 x nominal ratio
            peak = peak * FP8_OVER_BF16
            peak_kind = f"{peak_kind} bf16 x {FP8_OVER_BF16:g} (nominal E4M3/BF16 ratio), e4m3"
        else:
            peak_kind = f"{peak_kind} bf16"
        dom_ms = statistics.fmean(per[dominant])
        achieved = wd.flops / (dom_ms * 1e-3) / 1e12
        clk = clocks.summary() if clocks else None
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sm_mhz = (clk or {}).get("sm_mhz") or (clk or {}).get("sm_max_mhz") or 2070.0
        value = whole_job_tflops(flops_step, ws, step_ms_max)
        breakdown = {}
        for w in wl:
            ms = statistics.fmean(per[w.name])
            breakdown[w.name] = {"ms": round(ms, 5), "tflops": round(w.flops / (ms * 1e-3) / 1e12, 1),
                                 "pct_of_peak": round(100 * w.flops / (ms * 1e-3) / 1e12 / peak, 1),
                                 "ms_median": round(statistics.median(per[w.name]), 5),
                                 "ms_min": round(min(per[w.name]), 5), "ms_max": round(max(per[w.name]), 5)}
        cpu = cpu_baseline(budget_s=args.cpu_budget) if (args.cpu_budget > 0 and ws == 1) else None
        also = secondary_measurements(args) if (ws == 1 and args.also and not (
            args.fp8 or args.dropout > 0 or args.sched != "auto" or args.workloads)) else None
        entry = {w.name: ("fa_fwd_fp8 (V^T transpose + attention kernel)" if w.dtype == gen.FP8 else
                          "fa_fwd_dropout" if args.dropout > 0 else
                          "fa_fwd" if devbuf[w.name][5] is None else
                          "fa_fwd_ws (stream-K split of the key range, caller workspace)")
                 for w in wl}
        dom_entry = entry[dominant].split(" ")[0]
        dom_counters = recorded_counters(dominant, dom_entry) if dom_entry in ("fa_fwd", "fa_fwd_ws") else None
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
            "steps": n, "warmup": args.warmup, "ms_per_step": round(step_ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "+".join(sorted({w.dtype for w in wl})), "data": "synthetic",
            "config": {"workload": "+".join(names),
                       "shapes": [w.describe() for w in wl],
                       "l2": "flushed before every launch (256 MiB write, outside the events)",
                       "parallelism": "replicas" if ws > 1 else "single GPU",
                       "entry_point": entry,
                       "sched": args.sched,
                       "dropout": args.dropout,
                       "pct_of_peak": round(100 * value / ws / peak, 1)},
            "breakdown": breakdown,
            "roofline": {"bound": "tensor",
                         "kernel": f"fa_fwd_kernel<{wd.d}, {wd.dtype}, {'causal' if wd.causal else 'full'}"
                                   f"{', dropout' if args.dropout > 0 else ''}> on {dominant}",
                         "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_kind} dense (burst: kernel timed alone)",
                         "traffic": (dom_counters or {}).get("dram_bytes_per_launch"),
                         "algorithmic_bytes": wd.io_bytes,
                         "secondary": sfu_bound(wd, dom_ms, sms, sm_mhz, dom_counters)},
            "clocks": clk,
            "e2e": {"value": round(whole_job_tflops(flops_step, ws, e2e_ms_max), 2), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": ne2e,
                    "entry_point": "fa_fwd_host (chunked copies overlapped with compute)" if use_host_api
                    else "copy in, launch, copy out"},
            "gpu_launches": int(launches),
            "wall_s_timed": round(wall_max, 4),
            "cpu_baseline": cpu,
            "also": also,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def secondary_measurements(args):
    """The library's other paths, each timed by this script in its own process the same way
    (L2 flushed before every launch, CUDA events on the launching stream, medians over the
    steps): the backward pass, dropout forward and backward, E4M3 inputs, plain fa_fwd (no
    stream-K) on the full N=4096 workload, the d=64 cross-attention shape with and without
    stream-K, the B=1, H=16, N=32768 causal workload and the two 128 x 128 d=64 workloads,
    so that every workload of the method's test set has a measured rate. Not part of the
    headline metric."""
    runs = {
        "bwd": ["--bwd"],
        "bwd_dropout_0.1": ["--bwd", "--dropout", "0.1"],
        "fwd_dropout_0.1": ["--dropout", "0.1"],
        "fwd_fp8_e4m3": ["--fp8"],
        "fwd_full_n4096_plain_fa_fwd": ["--workloads", "b2h8_n4096_d128_full", "--sched", "plain"],
        "fwd_cross_d64_plain": ["--workloads", "b4h12_q1000_k4097_d64_cross", "--sched", "plain"],
        "fwd_cross_d64_streamk": ["--workloads", "b4h12_q1000_k4097_d64_cross", "--sched", "auto"],
        "fwd_n32768_causal_x2": ["--workloads", "b1h16_n32768_d128_causal_x2"],
        "fwd_tiny_full_and_causal": ["--workloads", "tiny,tiny_causal"],
    }
    steps = str(max(20, min(args.steps, 100)))
    out = {}
    for name, extra in runs.items():
        cmd = [sys.executable, os.path.abspath(__file__), "--steps", steps, "--warmup", "5",
               "--cpu-budget", "0", "--no-also", *extra]
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
            line = json.loads(r.stdout.strip().splitlines()[-1])
            out[name] = {"value": line["value"], "unit": line["unit"],
                         "entry_point": line["config"].get("entry_point"),
                         "sfu": (line.get("roofline") or {}).get("secondary"),
                         "breakdown": {k: {"ms": v["ms"], "tflops": v["tflops"],
                                           "pct_of_peak": v.get("pct_of_peak")}
                                       for k, v in line.get("breakdown", {}).items()}}
        except Exception as e:  # a failed side run is reported, never hidden
            out[name] = {"error": f"{type(e).__name__}: {str(e)[:200]}"}
    return out


# ----------------------------------------------------------------------------- backward
def run_bwd(args):
    """Backward pass (fa_bwd) on the same two workloads: one step = one backward of each.
    FLOPs: the five products of the backward, 10*B*H*Nq*Nk*d (halved when causal)."""
    import numpy as np
    import torch

    import exact_attention_forward_02_gb300 as fa
    import gen

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    names = tuple(args.workloads.split(",")) if args.workloads else WORKLOADS
    wl = [gen.WORKLOADS[n] for n in names]
    bufs = {}
    for w in wl:
        q, k, v = (t.to(dev) for t in gen.make_qkv(w))
        rng = np.random.default_rng([int(w.seed), 3])
        do = torch.from_numpy(rng.standard_normal((w.B, w.H, w.Nq, w.d))).to(gen.torch_dtype(w.dtype)).to(dev)
        O = torch.empty_like(q)
        L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
        dt = fa.FA_BF16 if w.dtype == gen.BF16 else fa.FA_F16
        if args.dropout > 0:  # the forward whose mask the backward regenerates
            rc = fa.fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(),
                                   L.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt,
                                   args.dropout, 1234, 1, sp)
        else:
            rc = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), L.data_ptr(),
                           w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt, sp)
        if rc != 0:
            raise fa.FAError(rc)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nws = fa.fa_bwd_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        bufs[w.name] = (q, k, v, O, do, L, dq, dk, dv, ws, dt)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def launch(w):
        q, k, v, O, do, L, dq, dk, dv, ws, dt = bufs[w.name]
        if args.dropout > 0:
            rc = fa.fa_bwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(),
                                   do.data_ptr(), L.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.d, w.scale, w.causal, dt,
                                   args.dropout, 1234, 1, ws.data_ptr(), ws.numel(), sp)
        else:
            rc = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), do.data_ptr(),
                           L.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H,
                           w.Nq, w.Nk, w.d, w.scale, w.causal, dt, ws.data_ptr(), ws.numel(), sp)
        if rc != 0:
            raise fa.FAError(rc)

    fa.fa_clear_status()
    for _ in range(args.warmup):
        for w in wl:
            flush.zero_()
            launch(w)
    torch.cuda.synchronize(dev)
    n = args.steps
    ev = {w.name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)] for w in wl}
    launches0 = fa.fa_num_kernel_launches()
    for i in range(n):
        for w in wl:
            flush.zero_()
            a, b = ev[w.name][i]
            a.record(stream)
            launch(w)
            b.record(stream)
    torch.cuda.synchronize(dev)
    launches = fa.fa_num_kernel_launches() - launches0
    status = fa.fa_last_status()
    if status != 0:
        raise fa.FAError(status, "device status")
    flops = {w.name: 2.5 * w.flops for w in wl}
    per = {w.name: [a.elapsed_time(b) for a, b in ev[w.name]] for w in wl}
    step_ms = sum(statistics.fmean(per[w.name]) for w in wl)
    peak, _, peak_kind = peaks()
    value = sum(flops.values()) / (step_ms * 1e-3) / 1e12
    line = {
        "metric": "attention bwd TFLOPS (dQ, dK, dV; bf16, causal & full)", "value": round(value, 2),
        "unit": UNIT, "n_gpus": 1, "steps": n, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "+".join(sorted({w.dtype for w in wl})), "data": "synthetic",
        "config": {"workload": "+".join(names), "shapes": [w.describe() for w in wl],
                   "l2": "flushed before every call (256 MiB write, outside the events)",
                   "flops": "10*B*H*Nq*Nk*d, halved when causal",
                   "entry_point": "fa_bwd_dropout" if args.dropout > 0 else "fa_bwd",
                   "dropout": args.dropout},
        "breakdown": {w.name: {"ms": round(statistics.fmean(per[w.name]), 5),
                               "tflops": round(flops[w.name] / (statistics.fmean(per[w.name]) * 1e-3) / 1e12, 1),
                               "pct_of_peak": round(100 * flops[w.name] / (statistics.fmean(per[w.name]) * 1e-3) / 1e12 / peak, 1)}
                      for w in wl},
        "roofline": {"bound": "tensor", "achieved": round(value, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(value / peak, 4), "peak_source": f"{peak_kind} bf16 dense",
                     "traffic": None},
        "gpu_launches": int(launches),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- oracle
_HEADS = {}


def _oracle_head(name):
    """Q, K, V of head (b=0, h=0) of a workload, widened to float64 (generated once)."""
    if name not in _HEADS:
        import gen
        w = gen.WORKLOADS[name]
        q, k, v = gen.make_qkv(w)
        _HEADS[name] = tuple(gen.to_f64_numpy(t[0, 0])[None, None] for t in (q, k, v))
    return _HEADS[name]


def _oracle_sample(budget_s: float, seed: int = 0):
    """Time the float64 oracle on row samples of both workloads for about budget_s
    seconds of host time. Returns (tflops, seconds, threads, description)."""
    import numpy as np

    import gen
    import oracle

    rng = np.random.default_rng(seed)
    total_flops = 0.0
    total_s = 0.0
    threads = oracle.hw_threads()
    desc = []
    share = budget_s / len(WORKLOADS)
    for name in WORKLOADS:
        w = gen.WORKLOADS[name]
        qh, kh, vh = _oracle_head(name)
        n_rows = 0
        spent = 0.0
        batch = max(threads * 32, 256)  # enough rows per call to keep every thread busy
        while spent < share:
            rows = rng.integers(0, w.Nq, size=batch)
            t0 = time.perf_counter()
            oracle.attention_rows(qh, kh, vh, w.scale, w.causal, rows)
            dt = time.perf_counter() - t0
            spent += dt
            vis = (np.minimum(rows + 1, w.Nk) if w.causal else np.full(rows.shape, w.Nk)).astype(np.float64)
            total_flops += float((4.0 * vis * w.d).sum())
            n_rows += batch
            if dt < 0.5 * share:
                batch = min(batch * 2, 1 << 16)
        total_s += spent
        desc.append(f"{n_rows} random rows of head (0,0) of {name}")
    return total_flops / total_s / 1e12, total_s, threads, "; ".join(desc)


WHOLE_CONFIGS = (("tiny", True), ("tiny_causal", True), ("b4h12_q1000_k4097_d64_cross", True),
                 ("b2h8_n4096_d128_full", False), ("b2h8_n8192_d128_causal", False))


def _oracle_whole_configs(configs=WHOLE_CONFIGS):
    """The oracle on whole configurations, end to end (the inputs already widened to
    float64): the two 128 x 128 d=64 workloads and the d=64 cross-attention workload
    (B=4, H=12, Nq=1000, Nk=4097; 50 GFLOP) on all host threads and on one thread, and the
    two benchmark workloads (137 and 275 GFLOP, a few seconds each) on all host threads."""
    import gen
    import oracle

    out = {}
    for name, single in configs:
        w = gen.WORKLOADS[name]
        q, k, v = (gen.to_f64_numpy(t) for t in gen.make_qkv(w))
        res = {}
        modes = (("all_threads", oracle.hw_threads()),) + ((("one_thread", 1),) if single else ())
        for label, nthreads in modes:
            reps, t0 = 0, time.perf_counter()
            while True:
                oracle.attention(q, k, v, w.scale, w.causal, nthreads=nthreads)
                reps += 1
                dt = time.perf_counter() - t0
                if dt >= 0.2:
                    break
            res[label] = {"ms": round(dt / reps * 1e3, 3), "tflops": round(w.flops * reps / dt / 1e12, 6),
                          "threads": nthreads}
        out[name] = res
    out["note"] = ("whole configurations, float64, inputs already widened; the N=32768 causal workload "
                   "(4.4 TFLOP, about a minute) is not timed here")
    return out


def cpu_baseline(budget_s: float):
    tf, secs, threads, desc = _oracle_sample(budget_s)
    line = {"value": round(tf, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{desc}; float64, {secs:.1f} s of host time; FLOPs 4*visible_keys*d per row"}
    try:
        line["whole_configs"] = _oracle_whole_configs()
    except Exception as e:  # reported, never allowed to suppress the bench line
        line["whole_configs"] = {"error": f"{type(e).__name__}: {str(e)[:200]}"}
    return line


def reference_step_budget(steps: int, warmup: int) -> float:
    """Host seconds of oracle work per reference-arm step: the whole --steps/--warmup run
    holds about 100 s of oracle time, 10 s per step at most (each step still times at
    least one batch of rows of each workload, so a step never does zero work)."""
    return min(10.0, 100.0 / max(1, steps + warmup))


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    per_step = reference_step_budget(args.steps, args.warmup)
    for _ in range(args.warmup):
        _oracle_sample(per_step, seed=1)
    vals, secs = [], 0.0
    threads = oracle.hw_threads()
    desc = ""
    t0 = time.perf_counter()
    for i in range(args.steps):
        tf, s, threads, desc = _oracle_sample(per_step, seed=100 + i)
        vals.append(tf)
        secs += s
    wall = time.perf_counter() - t0
    value = statistics.fmean(vals) if vals else 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "+".join(WORKLOADS),
                   "note": "float64 CPU oracle on bounded row samples per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}; about {per_step:.3g} s of host time"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workloads", default="",
                    help="comma-separated workload names (default: the two headline workloads)")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward pass (fa_bwd) instead of the forward")
    ap.add_argument("--fp8", action="store_true",
                    help="time fa_fwd_fp8 on the E4M3 versions of the two d=128 workloads")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="time fa_fwd_dropout with this dropout probability (default: no dropout)")
    ap.add_argument("--sched", choices=("auto", "plain"), default="auto",
                    help="auto (default): fa_fwd_ws with a workspace wherever the library's "
                         "stream-K split applies (full attention whose work items do not fill "
                         "whole waves of SMs), fa_fwd elsewhere; plain: fa_fwd only")
    ap.add_argument("--no-also", dest="also", action="store_false",
                    help="skip the side measurements of the other paths (backward, dropout, "
                         "E4M3, stream-K) that a default run adds under 'also'")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of host time for the oracle CPU baseline (0 = skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.bwd:
        run_bwd(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
