#!/usr/bin/env python
"""Benchmark of the batch-invariant W8A8 hot path.

Headline workload (synthetic, seeded): the high-concurrency FFN block of
the StartLux-Prism pages -- 64 clients x 32 tokens = 2048 token rows, hidden
size 5120, FFN width 17408.  One step is one pass of the hot path over it:
  1. prism_quant_act_f16   X [2048, 5120] bf16 -> codes + scales (smoothing on)
  2. prism_w8a8_linear_f16 gate/up projection, N = 34816, no residual
  3. prism_quant_act_f16   the down projection's input [2048, 17408]
  4. prism_w8a8_linear_f16 down projection, N = 5120, + bf16 residual
The weights are int8 codes with per-channel scales; they are converted once,
at load time and outside the timed region, to binary16 codes
(prism_codes_to_f16), the operand form of the tensor-core kernel on sm_103a,
which has no integer MMA (the f16 MMA is exact on these codes).  The metric
is int8 operations per second, 2*M*N*K per linear, over the whole step.

Timing: W warm-up steps, then exactly K steps of direct C-ABI launches on one
stream between CUDA events (device-resident inputs; the step's weights, 534
MB of codes, are larger than twice the L2).  Events around every gate/up
launch give the dominant kernel's mean duration for the roofline.
nvidia-smi samples SM clocks during the timed region.  The e2e figure
repeats the step through the Python binding with the step's inputs copied
from pinned host memory and the down projection's output copied back, all
inside the timed region (the next step's input copies run on a second
stream while the current step computes).

Sub-records in the same line (world size 1): the other configurations of the
method, each timed alone -- the short-request forest bucket (quantise, QKV,
quantise, o_proj, read-out of 3 answer positions), the decode-like weight
stream at every row count and split-K factor (with the bit-identity check
across all of them), the 8192-row long-evidence linear, the 192-position
candidate read-out next to a plain gather of the same rows, and the
quantiser.

`--impl reference` times the CPU oracle (the only other implementation of
this method) on a bounded sample of the same workload.  Multi-GPU
(torchrun): each rank runs its own FFN block, no collective on the data path
(weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

import workloads as wl

METRIC = "W8A8 linear int8 TOPS & % of int8 peak / GB/s % HBM; bit-exact vs oracle"
UNIT = "TOPS"
GATEUP, DOWN = "load_gateup_m2048_k5120_n34816", "load_down_m2048_k17408_n5120"
WORKLOAD = ("ffn_block_m2048: quant + gate_up(k5120,n34816) + quant + down(k17408,n5120,+res), "
            "64 clients x 32 tokens")
M_ROWS = 304                        # forest bucket rows (sub-record)
ANSWER_ROWS = (271, 287, 303)       # last token of each 16-token question
N_ROTATE = 3


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------- workloads ---
class FfnWorkload:
    """Host-side inputs of the headline FFN block (numpy)."""

    def __init__(self):
        self.gu = wl.make_linear(GATEUP)
        self.dn = wl.make_linear(DOWN)
        self.M = self.gu.M
        self.ops_gu = 2 * self.M * self.gu.N * self.gu.K
        self.ops_dn = 2 * self.M * self.dn.N * self.dn.K
        self.ops = self.ops_gu + self.ops_dn
        # algorithmic HBM bytes (int8 codes read once, outputs written once)
        self.bytes_gu = self.M * self.gu.K + self.gu.N * self.gu.K + 4 * self.gu.N + 4 * self.M + 2 * self.M * self.gu.N
        self.bytes_dn = (self.M * self.dn.K + self.dn.N * self.dn.K + 4 * self.dn.N + 4 * self.M
                         + 2 * self.M * self.dn.N * 2)
        self.bytes_quant = sum(3 * self.M * k + 4 * self.M + 4 * k for k in (self.gu.K, self.dn.K))
        self.bytes = self.bytes_gu + self.bytes_dn + self.bytes_quant


class ForestWorkload:
    """Host-side inputs of one short-request forest bucket (numpy)."""

    def __init__(self):
        self.qkv = wl.make_linear("forest_qkv_m304_k5120_n15360")
        self.o = wl.make_linear("forest_oproj_m304_k5120_n5120")
        self.ro = wl.readout_case("forest_answers", P=len(ANSWER_ROWS), K=wl.HIDDEN, V=wl.VOCAB, seed=9)
        self.cand_unique = np.unique(self.ro.cand_ids)
        self.cand_rows = self.ro.lm_rows(self.cand_unique)
        M, K = M_ROWS, wl.HIDDEN
        self.ops_linear_qkv = 2 * M * self.qkv.N * K
        self.ops_linear_o = 2 * M * self.o.N * K
        self.ops_readout = 2 * int(self.ro.cand_ids.size) * K
        self.ops = self.ops_linear_qkv + self.ops_linear_o + self.ops_readout


def reduce_max(value: float, device) -> float:
    """Max of ``value`` over all ranks of the default process group (the value
    itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(ops_per_step: float, steps: int, world: int, t_ms: float) -> float:
    """Whole-job TOPS: every rank runs ``steps`` steps of its own block; the
    job time is the slowest rank's."""
    return ops_per_step * steps * world / (t_ms / 1e3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def load_sustained_bf16():
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops_sustained"])
    except Exception:
        return None


def kernel_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary for this kernel and
    workload, or None when absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    try:
        rec = json.load(open(path))
        src = open(os.path.join(ROOT, "deterministic_w8a8_int8_gb300", "csrc", kernel_file), "rb").read()
        if rec.get("source_sha256") != hashlib.sha256(src).hexdigest():
            return None
        return int(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# --------------------------------------------------------------- clocks ----
class ClockSampler:
    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- CPU oracle ----
def ffn_sample_rows(n: int) -> np.ndarray:
    """n token rows of the FFN block, always including the first and last."""
    M = wl.LINEAR_CONFIGS[GATEUP][0]
    pick = np.random.default_rng(0).choice(np.arange(1, M - 1), size=max(0, n - 2), replace=False)
    return np.sort(np.concatenate([[0, M - 1], pick])).astype(np.int64)


def cpu_oracle_ffn(work: FfnWorkload, rows: np.ndarray):
    """The oracle on ``rows`` of the FFN block (both linears).  Returns
    (ops, (gate/up output rows, down output rows))."""
    import oracle
    q1, a1 = oracle.quant_act(work.gu.x_bits[rows], work.gu.inv_s)
    y, _ = oracle.w8a8_linear(q1, a1, work.gu.w, work.gu.w_scale, None)
    q2, a2 = oracle.quant_act(work.dn.x_bits[rows], work.dn.inv_s)
    h, _ = oracle.w8a8_linear(q2, a2, work.dn.w, work.dn.w_scale, work.dn.residual_bits[rows])
    ops = 2 * rows.size * (work.gu.N * work.gu.K + work.dn.N * work.dn.K)
    return ops, (y, h)


def run_cpu_baseline(work: FfnWorkload, budget_s: float = 12.0):
    import oracle
    cores = host_cores()
    oracle.set_threads(cores)
    rows = ffn_sample_rows(32)
    t0 = time.perf_counter()
    ops, outs = cpu_oracle_ffn(work, rows)
    dt = time.perf_counter() - t0
    reps, total_ops, total_t = 1, ops, dt
    while total_t < budget_s and reps < 50:
        t0 = time.perf_counter()
        o, _ = cpu_oracle_ffn(work, rows)
        total_t += time.perf_counter() - t0
        total_ops += o
        reps += 1
    return {"value": total_ops / total_t / 1e12, "unit": UNIT, "cores": int(oracle.get_threads()),
            "kind": "oracle",
            "sample": f"{rows.size} of {work.M} token rows (first and last included) through both "
                      f"linears, {reps} repetitions, {total_t:.1f} s"}, rows, outs


def run_reference(args):
    rank = env_int("RANK", 0)
    if rank != 0:
        return 0
    import oracle
    work = FfnWorkload()
    cores = host_cores()
    oracle.set_threads(cores)
    rows = ffn_sample_rows(8)
    for _ in range(args.warmup):
        cpu_oracle_ffn(work, rows)
    t0 = time.perf_counter()
    ops = 0
    for _ in range(args.steps):
        o, _ = cpu_oracle_ffn(work, rows)
        ops += o
    dt = time.perf_counter() - t0
    value = ops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_rows": int(rows.size)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(oracle.get_threads()), "kind": "oracle",
                         "sample": f"{rows.size} of {work.M} token rows of both linears per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU ----
def _timed(stream, fn, n, warm=3):
    """Mean and all per-call device times (us) of fn(i), i = 0..n-1, each
    bracketed by CUDA events on ``stream``."""
    import torch
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        evs[i][0].record(stream)
        fn(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    return statistics.mean(us), us


def run_gpu(args):
    import ctypes

    import torch
    import torch.distributed as dist

    import deterministic_w8a8_int8_gb300 as prism

    rank, world, local = env_int("RANK", 0), env_int("WORLD_SIZE", 1), env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    L = prism.lib()

    work = FfnWorkload()
    gu, dn, M = work.gu, work.dn, work.M

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    # model state, made once at load time: binary16 codes of the int8 weights
    Wgu = prism.prism_codes_to_f16(t(gu.w))
    Wdn = prism.prism_codes_to_f16(t(dn.w))
    Sgu, Sdn, Igu, Idn = t(gu.w_scale), t(dn.w_scale), t(gu.inv_s), t(dn.inv_s)
    # per-step inputs and outputs (preallocated)
    X, Xd, Res = bf16(gu.x_bits), bf16(dn.x_bits), bf16(dn.residual_bits)
    q1 = torch.empty((M, gu.K), dtype=torch.float16, device=dev)
    q2 = torch.empty((M, dn.K), dtype=torch.float16, device=dev)
    a1 = torch.empty((M,), dtype=torch.float32, device=dev)
    a2 = torch.empty_like(a1)
    Y = torch.empty((M, gu.N), dtype=torch.bfloat16, device=dev)
    H = torch.empty((M, dn.N), dtype=torch.bfloat16, device=dev)
    ws_gu = prism.new_workspace_f16(M, gu.N, gu.K, 0, dev)
    ws_dn = prism.new_workspace_f16(M, dn.N, dn.K, 0, dev)
    torch.cuda.synchronize()

    vp = lambda x: ctypes.c_void_p(x.data_ptr()) if x is not None else None
    stream = torch.cuda.Stream(device=dev)
    st = ctypes.c_void_p(stream.cuda_stream)
    nb = lambda w: 0 if w is None else w.numel()
    calls = [
        (L.prism_quant_act_f16, (vp(X), gu.K, vp(Igu), M, gu.K, vp(q1), gu.K, vp(a1), st)),
        (L.prism_w8a8_linear_f16, (vp(q1), gu.K, vp(a1), vp(Wgu), gu.K, vp(Sgu), None, 0, vp(Y), gu.N, None,
                                   M, gu.N, gu.K, 0, vp(ws_gu), nb(ws_gu), st)),
        (L.prism_quant_act_f16, (vp(Xd), dn.K, vp(Idn), M, dn.K, vp(q2), dn.K, vp(a2), st)),
        (L.prism_w8a8_linear_f16, (vp(q2), dn.K, vp(a2), vp(Wdn), dn.K, vp(Sdn), vp(Res), dn.N, vp(H), dn.N,
                                   None, M, dn.N, dn.K, 0, vp(ws_dn), nb(ws_dn), st)),
    ]
    launches_per_step = len(calls)

    def step(i, ev=None):
        for j, (fn, a) in enumerate(calls):
            if ev is not None and j == 1:
                ev[0].record(stream)
            rc = fn(*a)
            if rc != 0:
                raise RuntimeError(f"{fn.__name__} failed with status {rc}")
            if ev is not None and j == 1:
                ev[1].record(stream)

    torch.cuda.synchronize()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(i, evs[i])
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    gu_us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    if prism.prism_device_status() != 0:
        raise RuntimeError("a kernel raised a device status bit during the timed steps")
    t_max = reduce_max(elapsed_ms, dev)
    secs = t_max / 1e3
    value = weak_scaling_value(work.ops, args.steps, world, t_max)

    # ---- end to end through the binding, host buffers, copies inside timing
    pin = lambda a: a.pin_memory()
    hX = pin(torch.from_numpy(gu.x_bits.view(np.int16)).view(torch.bfloat16))
    hXd = pin(torch.from_numpy(dn.x_bits.view(np.int16)).view(torch.bfloat16))
    hRes = pin(torch.from_numpy(dn.residual_bits.view(np.int16)).view(torch.bfloat16))
    hH = torch.empty((M, dn.N), dtype=torch.bfloat16).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hX, hXd, hRes))
    d2h = hH.numel() * hH.element_size()
    # two device input sets: the copies of step i + 1 run on a copy stream
    # while step i computes; every copy is inside the timed region
    dX, dXd, dRes = [X, torch.empty_like(X)], [Xd, torch.empty_like(Xd)], [Res, torch.empty_like(Res)]
    copy_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def e2e_copy(i):
        b = i % 2
        copy_stream.wait_event(free[b])
        with torch.cuda.stream(copy_stream):
            dX[b].copy_(hX, non_blocking=True)
            dXd[b].copy_(hXd, non_blocking=True)
            dRes[b].copy_(hRes, non_blocking=True)
            ready[b].record(copy_stream)

    def e2e_compute(i):
        b = i % 2
        stream.wait_event(ready[b])
        with torch.cuda.stream(stream):
            prism.prism_quant_act_f16(dX[b], Igu, qh=q1, a_scale=a1)
            prism.prism_w8a8_linear_f16(q1, a1, Wgu, Sgu, out=Y, workspace=ws_gu)
            prism.prism_quant_act_f16(dXd[b], Idn, qh=q2, a_scale=a2)
            prism.prism_w8a8_linear_f16(q2, a2, Wdn, Sdn, residual=dRes[b], out=H, workspace=ws_dn)
            hH.copy_(H, non_blocking=True)
            free[b].record(stream)

    def e2e_run(n):
        e2e_copy(0)
        for i in range(n):
            if i + 1 < n:
                e2e_copy(i + 1)
            e2e_compute(i)

    e2e_run(3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dev)
    e2e_value = weak_scaling_value(work.ops, args.steps, world, e2e_ms)

    # ---- roofline of the dominant kernel (the gate/up linear)
    hbm_gbs, bf16_tflops, peak_src = load_peaks()
    sustained = load_sustained_bf16()
    gu_avg_s = statistics.mean(gu_us) / 1e6
    achieved = work.ops_gu / gu_avg_s / 1e12
    traffic = kernel_traffic("linear_f16.cu", "linear_f16_gateup_m2048_k5120_n34816")
    roofline = {"kernel": "prism_w8a8_linear_f16 (gate/up, M=2048 K=5120 N=34816)", "bound": "tensor",
                "achieved": achieved, "peak": bf16_tflops, "unit": "TFLOP/s",
                "frac": achieved / bf16_tflops, "traffic": traffic,
                "peak_source": f"{peak_src} bf16 dense burst (the exact int8 contraction runs on the f16 "
                               f"tensor pipe: sm_103a has no integer MMA)",
                "frac_of_sustained": None if sustained is None else achieved / sustained,
                "algorithmic_ops_per_launch": work.ops_gu,
                "algorithmic_bytes_per_launch": work.bytes_gu,
                "achieved_gbs": work.bytes_gu / gu_avg_s / 1e9, "hbm_peak_gbs": hbm_gbs,
                "avg_launch_us": gu_avg_s * 1e6}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch_rows": M * world,
                   "operands": "int8 codes held as binary16 (weights converted once at load time)",
                   "schedule": "balanced persistent schedule, one CTA per SM",
                   "l2": "inputs larger than L2: 534 MB of weight codes per step",
                   "launch": "direct C-ABI calls, arguments marshalled once",
                   "step_gbs": work.bytes * args.steps * world / secs / 1e9},
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, rows, outs = run_cpu_baseline(work)
        y_o, h_o = outs
        yb = Y.cpu().view(torch.int16).numpy().view(np.uint16)
        hb = H.cpu().view(torch.int16).numpy().view(np.uint16)
        cpu["matches_gpu_bitwise"] = bool(np.array_equal(yb[rows], y_o) and np.array_equal(hb[rows], h_o))
        line["cpu_baseline"] = cpu
    del Wgu, Wdn, Y
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_subrecords:
        line["configs"] = run_subrecords(prism, L, dev)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_subrecords(prism, L, dev):
    """Every other configuration of the method, timed alone on this GPU."""
    import torch
    out = {}
    for name, fn in (("forest_bucket_m304", sub_forest), ("decode_m1_64_k17408_n5120", sub_decode),
                     ("long_m8192_k5120_n5120", sub_long), ("readout_p192_v248000", sub_readout)):
        try:
            out[name] = fn(prism, L, dev)
        except Exception as e:   # a sub-record never hides the headline
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return out


def _linear_record(ops, byts, us, hbm, bf16):
    return {"us": us, "tops": ops / us / 1e6, "frac_bf16_peak": ops / us / 1e6 / bf16,
            "gbs": byts / us / 1e3, "frac_hbm": byts / us / 1e3 / hbm}


def sub_forest(prism, L, dev):
    """Short-request forest bucket: quantise X [304, 5120] -> QKV (N 15360) ->
    quantise -> o_proj (N 5120, +residual) -> read-out of the 3 answer
    positions against a 248,000 x 5120 LM head.  Each linear takes the faster
    of the two contraction kernels for its shape (binary16 codes for QKV, int8
    operands for o_proj); three weight sets are rotated so that weights come
    from HBM.  Per-linear times are events around that linear's launches."""
    import ctypes
    import torch
    work = ForestWorkload()
    M, K = M_ROWS, wl.HIDDEN
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf16 = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    sets = [dict(wq=prism.prism_codes_to_f16(t(work.qkv.w)), sq=t(work.qkv.w_scale), iq=t(work.qkv.inv_s),
                 wo=t(work.o.w), so=t(work.o.w_scale), io=t(work.o.inv_s)) for _ in range(N_ROTATE)]
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    lm_head = torch.randint(-127, 128, (wl.VOCAB, K), dtype=torch.int8, device=dev, generator=g)
    lm_head[t(work.cand_unique.astype(np.int64))] = t(work.cand_rows)
    lm_scale = t(work.ro.lm_scale)
    X, Xo, Res = bf16(work.qkv.x_bits), bf16(work.o.x_bits), bf16(work.o.residual_bits)
    off, ids = t(work.ro.cand_offsets), t(work.ro.cand_ids)
    T = int(ids.numel())
    q1 = torch.empty((M, K), dtype=torch.float16, device=dev)
    q2 = torch.empty((M, K), dtype=torch.int8, device=dev)
    a1 = torch.empty((M,), dtype=torch.float32, device=dev)
    a2 = torch.empty_like(a1)
    Y = torch.empty((M, work.qkv.N), dtype=torch.bfloat16, device=dev)
    H = torch.empty((M, work.o.N), dtype=torch.bfloat16, device=dev)
    logits = torch.empty((T,), dtype=torch.float32, device=dev)
    probs = torch.empty((T,), dtype=torch.float32, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    ws_q = prism.new_workspace_f16(M, work.qkv.N, K, 0, dev)
    ws_o = prism.new_workspace(M, work.o.N, K, 0, dev)
    hid = H[ANSWER_ROWS[0]::16]
    vp = lambda x: ctypes.c_void_p(x.data_ptr()) if x is not None else None
    stream = torch.cuda.Stream(device=dev)
    st = ctypes.c_void_p(stream.cuda_stream)
    nb = lambda w: 0 if w is None else w.numel()
    Nq, No = work.qkv.N, work.o.N

    def calls_for(s):
        return [
            (L.prism_quant_act_f16, (vp(X), K, vp(s["iq"]), M, K, vp(q1), K, vp(a1), st)),
            (L.prism_w8a8_linear_f16, (vp(q1), K, vp(a1), vp(s["wq"]), K, vp(s["sq"]), None, 0, vp(Y), Nq,
                                       None, M, Nq, K, 0, vp(ws_q), nb(ws_q), st)),
            (L.prism_quant_act, (vp(Xo), K, vp(s["io"]), M, K, vp(q2), K, vp(a2), st)),
            (L.prism_w8a8_linear, (vp(q2), K, vp(a2), vp(s["wo"]), K, vp(s["so"]), vp(Res), No, vp(H), No,
                                   None, M, No, K, 0, vp(ws_o), nb(ws_o), st)),
            (L.prism_candidate_readout, (vp(hid), hid.stride(0), None, vp(lm_head), K, vp(lm_scale),
                                         wl.VOCAB, K, vp(off), vp(ids), len(ANSWER_ROWS), T, vp(logits),
                                         vp(probs), vp(err), None, 0, st)),
        ]

    rot = [calls_for(s) for s in sets]
    ev = {j: [] for j in (1, 3, 4)}

    def step(i, record=False):
        for j, (fn, a) in enumerate(rot[i % N_ROTATE]):
            if record and j in ev:
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                e[0].record(stream)
            assert fn(*a) == 0
            if record and j in ev:
                e[1].record(stream)
                ev[j].append(e)

    for i in range(5):
        step(i)
    torch.cuda.synchronize()
    n = 30
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(n):
        step(i)
    s1.record(stream)
    torch.cuda.synchronize()
    step_us = s0.elapsed_time(s1) * 1e3 / n
    for i in range(n):
        step(i, record=True)
    torch.cuda.synchronize()
    us = {j: statistics.mean(a.elapsed_time(b) * 1e3 for a, b in ev[j]) for j in ev}
    assert int(err.item()) == 0

    def isolated(j):
        # launch j of every weight set, back to back in one CUDA graph on the
        # capturing stream (events around single calls also time launch gaps)
        calls = []
        for r in rot:
            fn, a = r[j]
            calls.append(lambda fn=fn, a=a: fn(*[ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
                                                 if x is st else x for x in a]))
        return graph_time_us(calls * 4)

    gq, go = isolated(1), isolated(3)
    hbm, bf16p, _ = load_peaks()
    bq = M * K + Nq * K + 4 * Nq + 4 * M + 2 * M * Nq
    bo = M * K + No * K + 4 * No + 4 * M + 2 * M * No * 2
    br = 2 * 3 * K + T * (K + 4) + 16 + 12 * T
    return {"step_us": step_us, "step_tops": work.ops / step_us / 1e6, "launches_per_step": 5,
            "qkv_m304_k5120_n15360": dict(_linear_record(work.ops_linear_qkv, bq, gq, hbm, bf16p),
                                          kernel="binary16 codes", events_us=us[1]),
            "oproj_m304_k5120_n5120": dict(_linear_record(work.ops_linear_o, bo, go, hbm, bf16p),
                                           kernel="int8 operands", events_us=us[3]),
            "readout_p3": {"us": us[4], "gbs": br / us[4] / 1e3, "frac_hbm": br / us[4] / 1e3 / hbm},
            "timing": ("step: back-to-back steps on one stream, 3 rotated weight sets; QKV and o_proj us: "
                       "each alone, a CUDA graph of back-to-back calls over the weight sets (events_us: "
                       "events around the call inside the step); read-out: events")}


def sub_decode(prism, L, dev):
    """Decode-like weight stream: M in {1, 8, 16, 64} rows of a 5120 x 17408
    weight (+ residual) at split-K in {1, 4, 8, 16} and the library's
    automatic choice (0): device time per call (a CUDA graph of back-to-back
    calls, four weight copies rotated so each call reads its weight from
    HBM), GB/s of the int8 weight stream, and the bit identity of every row
    across all 20 runs."""
    import torch
    c = wl.make_linear("decode_m64_k17408_n5120")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    X = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    q, a = prism.prism_quant_act(X, t(c.inv_s))
    n_rot = 4
    Ws = [t(c.w) for _ in range(n_rot)]
    S = t(c.w_scale)
    R = torch.from_numpy(c.residual_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    hbm, bf16p, _ = load_peaks()
    recs, ref = {}, None
    identical = True
    for M in wl.DECODE_M:
        best = None
        for split in (0,) + tuple(wl.DECODE_SPLITS):
            ws = prism.new_workspace(M, c.N, c.K, split, dev)
            out = torch.empty((M, c.N), dtype=torch.bfloat16, device=dev)
            fn = lambda i: prism.prism_w8a8_linear(q[:M], a[:M], Ws[i % n_rot], S, residual=R[:M], out=out,
                                                   split_k=split, workspace=ws)
            us = graph_time_us([lambda i=i: fn(i) for i in range(2 * n_rot)])
            bits = out.view(torch.int16)
            if ref is None:
                ref = torch.empty((64, c.N), dtype=torch.int16, device=dev)
                ref[:M] = bits
                filled = M
            elif M > filled:
                ref[filled:M] = bits[filled:M]
                filled = M
            identical = identical and torch.equal(bits, ref[:M])
            byts = M * c.K + c.N * c.K + 4 * c.N + 4 * M + 2 * M * c.N * 2
            r = dict(_linear_record(2 * M * c.N * c.K, byts, us, hbm, bf16p),
                     kind=prism.prism_w8a8_kernel_kind(M, c.N, c.K))
            recs[f"m{M}_split{split}"] = r
            if best is None or us < best[1]:
                best = (split, us, r["frac_hbm"])
        recs[f"m{M}_best"] = {"split": best[0], "us": best[1], "frac_hbm": best[2]}
    torch.cuda.synchronize()
    recs["all_rows_bit_identical_across_m_and_split"] = bool(identical)
    return recs


def sub_long(prism, L, dev):
    """Long-evidence linear: M = 8192, K = N = 5120, + residual, binary16
    codes (four weight copies rotated)."""
    import torch
    c = wl.make_linear("long_m8192_k5120_n5120")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    X = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    qh, a = prism.prism_quant_act_f16(X, t(c.inv_s))
    w8 = t(c.w)
    Ws = [prism.prism_codes_to_f16(w8) for _ in range(4)]
    S = t(c.w_scale)
    R = torch.from_numpy(c.residual_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    ws = prism.new_workspace_f16(c.M, c.N, c.K, 0, dev)
    fn = lambda i: prism.prism_w8a8_linear_f16(qh, a, Ws[i % 4], S, residual=R, out=out, workspace=ws)
    us, _ = _timed(torch.cuda.current_stream(), fn, 20)
    hbm, bf16p, _ = load_peaks()
    byts = c.M * c.K + c.N * c.K + 4 * c.N + 4 * c.M + 2 * c.M * c.N * 2
    return dict(_linear_record(2 * c.M * c.N * c.K, byts, us, hbm, bf16p), kernel="binary16 codes")


def sub_readout(prism, L, dev):
    """Candidate read-out of 192 answer positions (2-10 candidates each)
    against a 248,000 x 5120 LM head, next to a plain gather of the same
    candidate rows (torch.index_select, the rows' bytes copied once): the
    gather is the measured ceiling of a read-out that must fetch those rows.
    Several candidate sets and two heads are rotated so that rows come from
    HBM; both are CUDA graphs of back-to-back calls."""
    import torch
    P, K = 192, wl.HIDDEN
    case = wl.readout_case("readout", P=P, K=K, V=wl.VOCAB, seed=7)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    uniq = np.unique(case.cand_ids)
    rows = torch.from_numpy(case.lm_rows(uniq)).to(dev)
    heads = []
    for _ in range(2):
        W = torch.randint(-127, 128, (case.V, K), dtype=torch.int8, device=dev, generator=g)
        W[torch.from_numpy(uniq.astype(np.int64)).to(dev)] = rows
        heads.append(W)
    n_sets = max(8, int(np.ceil(2 * 129e6 / (P * 6 * (K + 4)))))
    sets = []
    for r in range(n_sets):
        cs = wl.readout_case("readout", P=P, K=K, V=wl.VOCAB, seed=100 + r)
        sets.append((torch.from_numpy(cs.h_bits.view(np.int16)).view(torch.bfloat16).to(dev),
                     torch.from_numpy(cs.cand_offsets).to(dev), torch.from_numpy(cs.cand_ids).to(dev),
                     int(cs.cand_ids.size)))
    ls = torch.from_numpy(case.lm_scale).to(dev)
    Tmax = max(x[3] for x in sets)
    lg = torch.empty((Tmax,), dtype=torch.float32, device=dev)
    pr = torch.empty((Tmax,), dtype=torch.float32, device=dev)
    gath = torch.empty((Tmax, K), dtype=torch.int8, device=dev)

    def call(i):
        h, off, ids, T = sets[i % n_sets]
        prism.prism_candidate_readout(h, None, heads[i % 2], ls, off, ids, logits=lg[:T], probs=pr[:T])

    def gather(i):
        h, off, ids, T = sets[i % n_sets]
        torch.index_select(heads[i % 2], 0, ids.long(), out=gath[:T])

    n = 2 * n_sets
    us = graph_time_us([lambda i=i: call(i) for i in range(n)])
    gus = graph_time_us([lambda i=i: gather(i) for i in range(n)])
    T = statistics.mean(x[3] for x in sets)
    byts = 2 * P * K + T * (K + 4) + 4 * (P + 1) + 4 * T + 8 * T
    gbytes = 2 * T * K   # the gather reads and writes every row once
    hbm, _, _ = load_peaks()
    return {"P": P, "T_avg": T, "us": us, "gbs": byts / us / 1e3, "frac_hbm": byts / us / 1e3 / hbm,
            "gather_ceiling": {"us": gus, "row_bytes_gbs": T * K / gus / 1e3,
                               "copy_gbs": gbytes / gus / 1e3, "frac_hbm": gbytes / gus / 1e3 / hbm},
            "frac_of_gather_ceiling": gus / us,
            "timing": f"CUDA graphs of back-to-back calls, {n_sets} candidate sets x 2 heads"}


def run_kernel(args):
    """Time one contraction call type alone on a named workload case (for
    per-kernel numbers and focused ncu captures).  Rotates enough weight copies
    that every launch reads its weights from HBM."""
    import ctypes
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    L = prism.lib()
    f16 = args.kernel == "linear_f16"
    c = wl.make_linear(args.case)
    M, K, N = c.M, c.K, c.N
    rows = M if args.rows is None else args.rows
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = torch.from_numpy(c.x_bits[:rows].view(np.int16)).view(torch.bfloat16).to(dev)
    inv = t(c.inv_s)
    a = torch.empty((rows,), dtype=torch.float32, device=dev)
    if f16:
        q = torch.empty((rows, K), dtype=torch.float16, device=dev)
        prism.prism_quant_act_f16(x, inv, qh=q, a_scale=a)
    else:
        q = torch.empty((rows, K), dtype=torch.int8, device=dev)
        prism.prism_quant_act(x, inv, q=q, a_scale=a)
    wbytes = N * K * (2 if f16 else 1)
    n_rot = max(1, int(np.ceil(3 * 129e6 / wbytes)))
    w8 = t(c.w)
    Ws = [prism.prism_codes_to_f16(w8) if f16 else w8.clone() for _ in range(n_rot)]
    del w8
    S = t(c.w_scale)
    R = None if c.residual_bits is None else torch.from_numpy(c.residual_bits[:rows].view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((rows, N), dtype=torch.bfloat16, device=dev)
    if f16:
        split = args.split if args.split is not None else 0
        ws = prism.new_workspace_f16(rows, N, K, split, dev)
        fn = L.prism_w8a8_linear_f16
    else:
        split = args.split if args.split is not None else prism.prism_w8a8_auto_split(rows, N, K)
        ws = prism.new_workspace(rows, N, K, split, dev)
        fn = L.prism_w8a8_linear
    stream = torch.cuda.Stream(device=dev)
    st = ctypes.c_void_p(stream.cuda_stream)
    vp = lambda z: None if z is None else ctypes.c_void_p(z.data_ptr())
    calls = [(vp(q), K, vp(a), vp(W), K, vp(S), vp(R), N, vp(out), N, None, rows, N, K, split, vp(ws),
              0 if ws is None else ws.numel(), st) for W in Ws]
    torch.cuda.synchronize()
    for i in range(args.warmup):
        assert fn(*calls[i % n_rot]) == 0
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        evs[i][0].record(stream)
        assert fn(*calls[i % n_rot]) == 0
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    us = [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]
    # device time per call without host gaps: a CUDA graph of back-to-back
    # calls on the capturing stream (per-call events above also time the
    # host's enqueue when a call is shorter than it)
    def gcall(i):
        cs = torch.cuda.current_stream().cuda_stream
        assert fn(*calls[i % n_rot][:-1], ctypes.c_void_p(cs)) == 0

    avg = graph_time_us([lambda i=i: gcall(i) for i in range(2 * n_rot)])
    ops = 2 * rows * N * K
    byts = rows * K + N * K + 4 * N + 4 * rows + 2 * rows * N * (2 if R is not None else 1)
    hbm, bf16, src = load_peaks()
    print(json.dumps({"kernel": "prism_w8a8_linear_f16" if f16 else "prism_w8a8_linear", "case": args.case,
                      "M": rows, "N": N, "K": K,
                      "split": split, "kind": "f16 codes" if f16 else prism.prism_w8a8_kernel_kind(rows, N, K),
                      "avg_us": avg, "events_avg_us": statistics.mean(us), "min_us": min(us),
                      "timing": "CUDA graph of back-to-back calls", "tflops": ops / avg / 1e6,
                      "frac_bf16_peak": ops / avg / 1e6 / bf16, "gbs": byts / avg / 1e3,
                      "frac_hbm": byts / avg / 1e3 / hbm, "weight_copies": n_rot,
                      "status": prism.prism_device_status()}), flush=True)
    return 0


def graph_time_us(calls, reps: int = 5):
    """Mean device time per call of the no-argument launch callables in
    ``calls``: they are captured back to back in one CUDA graph (so host
    marshalling is not timed) and the graph is replayed ``reps`` times."""
    import torch
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for c in calls:          # warm: per-device attributes, lazy module loading
            c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * len(calls))


def run_kernel_quant(args):
    """Time prism_quant_act alone on the activations of --case (HBM-bound)."""
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    dev = torch.device("cuda", 0)
    c = wl.make_linear(args.case)
    rows = c.M if args.rows is None else args.rows
    K = c.K
    n_rot = max(1, int(np.ceil(3 * 129e6 / (rows * K * 3))))
    xs = [torch.from_numpy(c.x_bits[:rows].view(np.int16)).view(torch.bfloat16).to(dev) for _ in range(n_rot)]
    inv = torch.from_numpy(c.inv_s).to(dev)
    qs = [torch.empty((rows, K), dtype=torch.int8, device=dev) for _ in range(n_rot)]
    a = torch.empty((rows,), dtype=torch.float32, device=dev)
    calls = [lambda i=i: prism.prism_quant_act(xs[i % n_rot], inv, q=qs[i % n_rot], a_scale=a)
             for i in range(max(args.steps, n_rot))]
    avg = graph_time_us(calls)
    byts = 3 * rows * K + 4 * rows + 4 * K
    hbm, _, _ = load_peaks()
    print(json.dumps({"kernel": "prism_quant_act", "case": args.case, "M": rows, "K": K, "avg_us": avg,
                      "gbs": byts / avg / 1e3, "frac_hbm": byts / avg / 1e3 / hbm,
                      "timing": "CUDA graph of back-to-back calls, %d activation copies" % n_rot}), flush=True)
    return 0


def run_kernel_requant(args):
    """Time prism_smooth_requant alone on one projection's Q8_0 weight
    (load-time step, HBM-bound); --case names a REQUANT_CONFIGS entry."""
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    dev = torch.device("cuda", 0)
    c = wl.make_q8_0(args.case)
    N, K = c.q.shape
    # enough input copies that one pass over them exceeds L2 twice over
    n_rot = max(1, int(np.ceil(2 * 129e6 / (N * K))))
    qs = [torch.from_numpy(c.q).to(dev) for _ in range(n_rot)]
    d = torch.from_numpy(c.d.view(np.int16)).to(dev)
    s = torch.from_numpy(c.s).to(dev)
    w = torch.empty((N, K), dtype=torch.int8, device=dev)
    ws = torch.empty((N,), dtype=torch.float32, device=dev)
    calls = [lambda i=i: prism.prism_smooth_requant(qs[i % n_rot], d, s, w=w, w_scale=ws)
             for i in range(max(args.steps, n_rot))]
    avg = graph_time_us(calls)
    byts = 2 * N * K + 2 * N * (K // 32) + 4 * K + 4 * N
    hbm, _, _ = load_peaks()
    print(json.dumps({"kernel": "prism_smooth_requant", "case": args.case, "N": N, "K": K, "avg_us": avg,
                      "gbs": byts / avg / 1e3, "frac_hbm": byts / avg / 1e3 / hbm,
                      "timing": "CUDA graph of back-to-back calls, %d weight copies" % n_rot}), flush=True)
    return 0


def answer_rows(M: int, P: int) -> np.ndarray:
    """P answer positions among M tokens: the last token of each of P
    16-token questions at the end of the sequence when they fit (256
    evidence tokens + 3 x 16 question tokens for M = 304), else the last
    token of P equal segments."""
    if M >= 16 * P + 1:
        return np.array([M - 1 - 16 * (P - 1 - i) for i in range(P)], np.int32)
    return np.array([(i + 1) * M // P - 1 for i in range(P)], np.int32)


def run_kernel_restricted(args):
    """The last layer's projection restricted to the answer positions
    (gathered quantisation + linear with the residual rows of the full hidden
    state) against the same projection on every position; --case is the
    linear case (default the o_proj shape), --rows the number of answer
    positions (default 3)."""
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    dev = torch.device("cuda", 0)
    c = wl.make_linear(args.case)
    M, K, N = c.M, c.K, c.N
    P = 3 if args.rows is None else args.rows
    rows = torch.from_numpy(answer_rows(M, P)).to(dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    inv = t(c.inv_s)
    n_rot = max(1, int(np.ceil(3 * 129e6 / (N * K))))
    Ws = [t(c.w) for _ in range(n_rot)]
    S = t(c.w_scale)
    res = c.residual_bits if c.residual_bits is not None else wl.bf16_bits(
        np.random.default_rng(1).standard_normal((M, N), dtype=np.float32))
    R = torch.from_numpy(res.view(np.int16)).view(torch.bfloat16).to(dev)
    qr = torch.empty((P, K), dtype=torch.int8, device=dev)
    ar = torch.empty((P,), dtype=torch.float32, device=dev)
    outr = torch.empty((P, N), dtype=torch.bfloat16, device=dev)
    wsr = prism.new_workspace(P, N, K, 0, dev)
    qf = torch.empty((M, K), dtype=torch.int8, device=dev)
    af = torch.empty((M,), dtype=torch.float32, device=dev)
    outf = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wsf = prism.new_workspace(M, N, K, 0, dev)

    def restricted(i):
        prism.prism_quant_act_rows(x, rows, inv, q=qr, a_scale=ar)
        prism.prism_w8a8_linear_rows(qr, ar, Ws[i % n_rot], S, R, rows, out=outr, workspace=wsr)

    def full(i):
        prism.prism_quant_act(x, inv, q=qf, a_scale=af)
        prism.prism_w8a8_linear(qf, af, Ws[i % n_rot], S, residual=R, out=outf, workspace=wsf)

    n = max(args.steps, n_rot)
    t_r = graph_time_us([lambda i=i: restricted(i) for i in range(n)])   # per quantise + linear pair
    t_f = graph_time_us([lambda i=i: full(i) for i in range(n)])
    torch.cuda.synchronize()
    assert torch.equal(outr.view(torch.int16), outf[rows.long()].view(torch.int16)), "restricted != full rows"
    byts = 3 * P * K + 4 * P + P * K + N * K + 4 * N + 4 * P + 4 * P * N
    hbm, _, _ = load_peaks()
    print(json.dumps({"kernel": "restricted_last_layer", "case": args.case, "M_full": M, "M_answer": P,
                      "N": N, "K": K, "restricted_us": t_r, "full_us": t_f, "speedup": t_f / t_r,
                      "restricted_gbs": byts / t_r / 1e3, "frac_hbm": byts / t_r / 1e3 / hbm,
                      "check": "restricted output == full output rows (bitwise)",
                      "timing": "CUDA graph of back-to-back quantise + linear pairs, %d weight copies" % n_rot}),
          flush=True)
    return 0


def run_kernel_tp(args):
    """One rank of a row-parallel tensor-parallel layer over --rows ranks
    (default 2) on --case: its shard maxima, its codes with the shared
    maximum, its exact int32 partial and the epilogue after the combine,
    timed on one GPU (the two all-reduces between them are the caller's
    collectives and are not timed here), next to the one-device layer."""
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    dev = torch.device("cuda", 0)
    c = wl.make_linear(args.case)
    M, K, N = c.M, c.K, c.N
    world = 2 if args.rows is None else args.rows
    Kr = K // world
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    xr = x[:, :Kr].contiguous()
    inv = t(c.inv_s)
    invr = inv[:Kr].contiguous()
    n_rot = max(1, int(np.ceil(3 * 129e6 / (N * Kr))))
    Wr = [t(c.w[:, :Kr]) for _ in range(n_rot)]
    Wf = [t(c.w) for _ in range(max(1, int(np.ceil(3 * 129e6 / (N * K)))))]
    S = t(c.w_scale)
    R = None if c.residual_bits is None else torch.from_numpy(c.residual_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    amax = torch.empty((M,), dtype=torch.float32, device=dev)
    q = torch.empty((M, Kr), dtype=torch.int8, device=dev)
    a = torch.empty((M,), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N), dtype=torch.int32, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    # the epilogue rotates accumulator, residual and output copies that
    # together exceed L2 twice over
    n_acc = max(2, int(np.ceil(2 * 129e6 / (M * N * 8))))
    accs = [torch.randint(-2**20, 2**20, (M, N), dtype=torch.int32, device=dev) for _ in range(n_acc)]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(n_acc)]
    Rs = [None if R is None else R.clone() for _ in range(n_acc)]
    wsr = prism.new_workspace(M, N, Kr, 0, dev)
    qf = torch.empty((M, K), dtype=torch.int8, device=dev)
    af = torch.empty((M,), dtype=torch.float32, device=dev)
    wsf = prism.new_workspace(M, N, K, 0, dev)
    n = max(args.steps, n_rot)
    steps = {
        "act_amax": [lambda: prism.prism_act_amax(xr, invr, amax=amax)] * n,
        "quant_act_amax": [lambda: prism.prism_quant_act_amax(xr, invr, amax, q=q, a_scale=a)] * n,
        "gemm_s32": [lambda i=i: prism.prism_w8a8_gemm_s32(q, Wr[i % n_rot], acc=acc, workspace=wsr)
                     for i in range(n)],
        "epilogue": [lambda i=i: prism.prism_w8a8_epilogue(accs[i % n_acc], a, S, residual=Rs[i % n_acc],
                                                           out=outs[i % n_acc])
                     for i in range(max(n, n_acc))],
    }
    prism.prism_act_amax(xr, invr, amax=amax)
    us = {k: graph_time_us(v) for k, v in steps.items()}
    full = graph_time_us([lambda i=i: (prism.prism_quant_act(x, inv, q=qf, a_scale=af),
                                       prism.prism_w8a8_linear(qf, af, Wf[i % len(Wf)], S, residual=R, out=outf,
                                                               workspace=wsf))
                          for i, outf in zip(range(n), [torch.empty_like(out)] * n)])
    epi_bytes = M * N * (4 + 2 + (2 if R is not None else 0)) + 4 * (M + N)
    hbm, _, _ = load_peaks()
    print(json.dumps({"kernel": "tp_row_parallel_rank", "case": args.case, "ranks": world, "M": M, "N": N,
                      "K_rank": Kr, "rank_us": us, "rank_total_us": sum(us.values()), "one_device_us": full,
                      "epilogue_gbs": epi_bytes / us["epilogue"] / 1e3,
                      "epilogue_frac_hbm": epi_bytes / us["epilogue"] / 1e3 / hbm,
                      "timing": "CUDA graphs of back-to-back calls; collectives not included; the epilogue "
                                "rotates %d accumulator / residual / output copies" % n_acc}), flush=True)
    return 0


def run_kernel_w4a8(args):
    """W4A8 on packed 4-bit weights of --case's shape (codes drawn like the
    pages' 4-bit weights; --rows token rows, default 1) next to W8A8 on the
    same shape, graph-timed on rotated weight copies."""
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    dev = torch.device("cuda", 0)
    c = wl.make_linear(args.case)
    M = 1 if args.rows is None else args.rows
    K, N = c.K, c.N
    rng = np.random.default_rng(17)
    codes = wl.draw_w4_codes(rng, (N, K))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x = torch.from_numpy(c.x_bits[:M].view(np.int16)).view(torch.bfloat16).to(dev)
    q, a = prism.prism_quant_act(x, t(c.inv_s))
    S = t(c.w_scale)
    R = None if c.residual_bits is None else torch.from_numpy(c.residual_bits[:M].view(np.int16)).view(torch.bfloat16).to(dev)
    n4 = max(1, int(np.ceil(3 * 129e6 / (N * K // 2))))
    n8 = max(1, int(np.ceil(3 * 129e6 / (N * K))))
    W4 = [t(wl.pack_w4(codes)) for _ in range(n4)]
    W8 = [t(codes) for _ in range(n8)]
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    need = prism.prism_w4a8_workspace_bytes(M, N, K, 0)
    ws4 = torch.zeros(need, dtype=torch.uint8, device=dev) if need else None
    ws8 = prism.new_workspace(M, N, K, 0, dev)
    n = max(args.steps, n4, n8)
    t4 = graph_time_us([lambda i=i: prism.prism_w4a8_linear(q, a, W4[i % n4], S, residual=R, out=out,
                                                            workspace=ws4) for i in range(n)])
    t8 = graph_time_us([lambda i=i: prism.prism_w8a8_linear(q, a, W8[i % n8], S, residual=R, out=out,
                                                            workspace=ws8) for i in range(n)])
    byts = N * K // 2 + M * K + 4 * (M + N) + 2 * M * N * (2 if R is not None else 1)
    hbm, _, _ = load_peaks()
    print(json.dumps({"kernel": "prism_w4a8_linear", "case": args.case, "M": M, "N": N, "K": K,
                      "kind": prism.prism_w8a8_kernel_kind(M, N, K), "w4a8_us": t4, "w8a8_us": t8,
                      "speedup_vs_w8a8": t8 / t4, "w4a8_gbs": byts / t4 / 1e3,
                      "frac_hbm": byts / t4 / 1e3 / hbm,
                      "timing": "CUDA graphs of back-to-back calls, %d / %d weight copies" % (n4, n8)}), flush=True)
    return 0


def run_kernel_readout(args):
    """Time prism_candidate_readout alone: P answer positions of a 248,000 x
    5120 LM head (several head copies rotated so gathers come from HBM)."""
    import torch

    import deterministic_w8a8_int8_gb300 as prism

    dev = torch.device("cuda", 0)
    P = 192 if args.rows is None else args.rows
    case = wl.readout_case("readout", P=P, K=wl.HIDDEN, V=wl.VOCAB, seed=7)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    heads = []
    uniq = np.unique(case.cand_ids)
    rows = torch.from_numpy(case.lm_rows(uniq)).to(dev)
    for _ in range(2):
        W = torch.randint(-127, 128, (case.V, case.K), dtype=torch.int8, device=dev, generator=g)
        W[torch.from_numpy(uniq.astype(np.int64)).to(dev)] = rows
        heads.append(W)
    # candidate lists rotated through independent id sets, enough of them that
    # the rows all calls gather (about 5.8 MB per call at P=192) exceed L2
    n_sets = max(8, int(np.ceil(2 * 129e6 / (P * 6 * (wl.HIDDEN + 4)))))
    sets = []
    for r in range(n_sets):
        cs = wl.readout_case("readout", P=P, K=wl.HIDDEN, V=wl.VOCAB, seed=100 + r)
        sets.append((torch.from_numpy(cs.h_bits.view(np.int16)).view(torch.bfloat16).to(dev),
                     torch.from_numpy(cs.cand_offsets).to(dev), torch.from_numpy(cs.cand_ids).to(dev),
                     cs.cand_ids.size))
    ls = torch.from_numpy(case.lm_scale).to(dev)
    Tmax = max(x[3] for x in sets)
    lg = torch.empty((Tmax,), dtype=torch.float32, device=dev)
    pr = torch.empty((Tmax,), dtype=torch.float32, device=dev)

    def call(i):
        h, off, ids, T = sets[i % n_sets]
        prism.prism_candidate_readout(h, None, heads[i % 2], ls, off, ids, logits=lg[:T], probs=pr[:T])

    avg = graph_time_us([lambda i=i: call(i) for i in range(max(args.steps, 2 * n_sets))])
    T = statistics.mean(x[3] for x in sets)
    K = case.K
    byts = 2 * P * K + T * (K + 4) + 4 * (P + 1) + 4 * T + 8 * T
    hbm, _, _ = load_peaks()
    print(json.dumps({"kernel": "prism_candidate_readout", "P": P, "T_avg": T, "K": K, "avg_us": avg,
                      "gbs": byts / avg / 1e3, "frac_hbm": byts / avg / 1e3 / hbm,
                      "timing": "CUDA graph of back-to-back calls, %d candidate sets x 2 heads" % n_sets}),
          flush=True)
    return 0


def run_kernel_int8_peak(args):
    """The dense int8 rate a library reaches on this GPU, beside bf16: torch's
    int8 matmul (torch._int_mm, int8 x int8 -> int32) and bf16 torch.matmul,
    8192^3 each, best of 10 timed calls (burst) and back to back for 4 s
    (sustained), with SM clocks sampled during the sustained loops.  This is
    what decides which tensor pipe the exact contraction runs on."""
    import torch

    dev = torch.device("cuda", 0)
    n = 8192
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    a8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev, generator=g)
    b8 = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev, generator=g).t().contiguous().t()
    a16 = a8.to(torch.bfloat16)
    b16 = b8.to(torch.bfloat16)
    ops = 2.0 * n ** 3
    res = {}
    for name, fn in (("int8_int_mm", lambda: torch._int_mm(a8, b8)), ("bf16_matmul", lambda: a16 @ b16)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) * 1e-3)
        with ClockSampler(0) as cs:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(10, int(4.0 / best))
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
        sus = e0.elapsed_time(e1) * 1e-3 / reps
        res[name] = {"burst_tops": ops / best / 1e12, "sustained_tops": ops / sus / 1e12, "reps": reps,
                     "clocks": cs.summary()}
    # the int8 product is exact: a block of it against int64 arithmetic on the host
    blk = a8[:64].cpu().to(torch.int64) @ b8[:, :64].cpu().to(torch.int64)
    assert torch.equal(torch._int_mm(a8, b8)[:64, :64].cpu().to(torch.int64), blk)
    print(json.dumps({"kernel": "library dense peaks", "n": n, **res,
                      "gpu": torch.cuda.get_device_name(dev)}), flush=True)
    return 0


_MMA_RATE_SRC = r"""
#include <torch/extension.h>
#include <cstdint>
// Register-resident loops of the warp-level MMAs (independent accumulators):
// the issue rate of mma.sync m16n8k16 f16 -> f32 and m16n8k32 s8 -> s32.
template <int kAcc>
__global__ void f16_loop(float* out, int iters) {
  uint32_t a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 + 1, b1 = a0 + 2;
  float c[kAcc][4] = {};
  for (int i = 0; i < iters; ++i)
#pragma unroll
    for (int j = 0; j < kAcc; ++j)
      asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                   : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                   : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  float s = 0.f;
  for (int j = 0; j < kAcc; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}
template <int kAcc>
__global__ void s8_loop(float* out, int iters) {
  uint32_t a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 + 1, b1 = a0 + 2;
  int c[kAcc][4] = {};
  for (int i = 0; i < iters; ++i)
#pragma unroll
    for (int j = 0; j < kAcc; ++j)
      asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                   : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                   : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  int s = 0;
  for (int j = 0; j < kAcc; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = static_cast<float>(s);
}
void launch(torch::Tensor out, int64_t which, int64_t blocks, int64_t threads, int64_t iters) {
  auto st = at::cuda::getCurrentCUDAStream();
  if (which == 0) f16_loop<8><<<blocks, threads, 0, st>>>(out.data_ptr<float>(), static_cast<int>(iters));
  else s8_loop<8><<<blocks, threads, 0, st>>>(out.data_ptr<float>(), static_cast<int>(iters));
}
"""


def run_kernel_mma_rate(args):
    """Issue rate of the warp-level tensor-core MMAs that the weight-streaming
    kernel uses (mma.sync m16n8k16 f16 -> f32 and m16n8k32 s8 -> s32): each
    warp loops over 8 independent accumulators in registers, 4 to 16 warps per
    CTA, one or two CTAs per SM, timed with CUDA events (a probe compiled at
    run time for sm_103a)."""
    import torch
    from torch.utils.cpp_extension import load_inline

    ext = load_inline("prism_mma_rate_probe", cpp_sources="void launch(torch::Tensor, int64_t, int64_t, int64_t, int64_t);",
                      cuda_sources="#include <ATen/cuda/CUDAContext.h>\n" + _MMA_RATE_SRC, functions=["launch"],
                      extra_cuda_cflags=["-gencode", "arch=compute_103a,code=sm_103a", "-O3"], verbose=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.empty(sms * 2 * 512, dtype=torch.float32, device="cuda")
    iters = 20000
    res = {}
    for which, name, ops_per in ((0, "f16_m16n8k16_tflops", 2 * 16 * 8 * 16), (1, "s8_m16n8k32_tops", 2 * 16 * 8 * 32)):
        best = 0.0
        for warps in (4, 8, 16):
            for per_sm in (1, 2):
                blocks, threads = sms * per_sm, warps * 32
                ext.launch(out, which, blocks, threads, 100)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                ext.launch(out, which, blocks, threads, iters)
                e1.record()
                torch.cuda.synchronize()
                rate = ops_per * 8.0 * iters * blocks * warps / (e0.elapsed_time(e1) * 1e-3) / 1e12
                res[f"{name}_w{warps}_b{per_sm}"] = rate
                best = max(best, rate)
        res[name] = best
    print(json.dumps({"kernel": "warp-level mma.sync issue rate", **res,
                      "gpu": torch.cuda.get_device_name(0)}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true", help="headline line only (no per-config sub-records)")
    ap.add_argument("--kernel", choices=["linear", "linear_f16", "quant", "readout", "requant", "restricted", "tp",
                                         "w4a8", "int8_peak", "mma_rate"],
                    help="time one call type alone")
    ap.add_argument("--case", default=None, choices=sorted(wl.LINEAR_CONFIGS) + sorted(wl.REQUANT_CONFIGS),
                    help="workload of --kernel (a linear case; for requant a weight as loaded)")
    ap.add_argument("--rows", type=int, default=None, help="use the first ROWS token rows of --case")
    ap.add_argument("--split", type=int, default=None, help="split-K for --kernel (default automatic)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel == "int8_peak":
        return run_kernel_int8_peak(args)
    if args.kernel == "requant":
        args.case = args.case or "qkv_n15360_k5120"
        if args.case not in wl.REQUANT_CONFIGS:
            ap.error("--kernel requant takes --case from " + ", ".join(sorted(wl.REQUANT_CONFIGS)))
        return run_kernel_requant(args)
    if args.kernel == "restricted":
        args.case = args.case or "forest_oproj_m304_k5120_n5120"
    args.case = args.case or "forest_qkv_m304_k5120_n15360"
    if args.case not in wl.LINEAR_CONFIGS:
        ap.error("--case must be a linear case for this mode")
    if args.kernel == "quant":
        return run_kernel_quant(args)
    if args.kernel == "restricted":
        return run_kernel_restricted(args)
    if args.kernel == "tp":
        return run_kernel_tp(args)
    if args.kernel == "w4a8":
        return run_kernel_w4a8(args)
    if args.kernel == "readout":
        return run_kernel_readout(args)
    if args.kernel == "mma_rate":
        return run_kernel_mma_rate(args)
    if args.kernel:
        return run_kernel(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
