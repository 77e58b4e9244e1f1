#!/usr/bin/env python3
"""Benchmark of memory-efficient biased Evoformer attention on GB300.

One step = forward + backward of O = softmax(Q Kᵀ D^-1/2 + bias1 + bias2) V
over one batch of the named workload (default: MSA column-wise attention,
B=1, N=384, L=1024, H=8, D=32, bf16, key mask only — the largest of the five
configurations), i.e. every kernel of the hot path the workload needs:
forward, delta/accumulator set-up, main backward, dQ cast, and with a pair
bias the deterministic pair-bias gradient stages.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--dtype bf16|fp16] [--micro]

Prints one JSON line (rank 0).  `value` is whole-job fwd+bwd TFLOP/s with
nominal FLOPs (forward 4·B·N·H·L²·D, backward 2.5× forward) and inputs
resident in HBM; `fwd_tflops` is the forward kernel alone; `e2e` is the same
metric through the host-buffer C-ABI step (evo_attn_step_host) with the
host↔device copies inside the timed region.  The timed steps are CUDA-graph
replays over R input replicas whose total exceeds 3× the L2 cache, so no step
reads inputs left in L2 by the previous one.  Per-kernel times come from CUDA
events that the library records around each of its launches inside the timed
replays (the per-call profiling events of evo_attn_fwd_opts / evo_attn_bwd_opts).
`--impl reference` times the fp64 CPU
oracle on bounded samples of the same workload (it is the reference arm).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Evoformer attn fwd & fwd+bwd TFLOP/s and fraction of GB300 dense tensor peak"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- helpers
def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="msa_col",
                    help="msa_col (default: the largest configuration, B=1 N=384 L=1024 H=8 D=32), msa_row, "
                         "many_head, triangle or tiny")
    ap.add_argument("--rows", type=int, default=0,
                    help="run the workload with this many rows N instead of its own (same L, H, D, masks): a "
                         "reduced instance for ncu captures; never a headline")
    ap.add_argument("--micro", action="store_true",
                    help="run the throughput microbenchmarks (exponentials, FMA, tcgen05.mma issue) instead")
    ap.add_argument("--dtype", default="bf16", choices=("bf16", "fp16"))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-masked-tiles", action="store_true",
                    help="skip key tiles whose keys are all masked (bias1 <= -1e4); the FLOP count stays "
                         "the nominal one of the full shape, so report such a line apart from the headline")
    return ap.parse_args()


def flops(w):
    fwd = 4.0 * w.B * w.N * w.H * w.L * w.L * w.D
    return {"fwd": fwd, "bwd": 2.5 * fwd, "step": 3.5 * fwd}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = sum(i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas")
        if n > 0:
            return n
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_step(inp, rows):
    """fp64 oracle forward + backward on rows n < rows of batch 0 (bias2 is shared over n)."""
    from oracle import evo_oracle as O
    sl = lambda t: None if t is None else t[:1, :rows].double().numpy()
    b2 = None if inp["bias2"] is None else inp["bias2"][:1].double().numpy()
    q, k, v, do, b1 = sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["do"]), sl(inp["bias1"])
    O.forward(q, k, v, b1, b2)
    O.backward(q, k, v, b1, b2, do)


def oracle_row_seconds(inp):
    t0 = time.perf_counter()
    oracle_step(inp, 1)
    return max(time.perf_counter() - t0, 1e-6)


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, max SM clock, power, active
    clock-event reasons); None when libnvidia-ml is not loadable."""
    HW_SLOWDOWN, SW_POWER_CAP, SW_THERMAL, HW_THERMAL, HW_POWER_BRAKE = 0x8, 0x4, 0x20, 0x40, 0x80

    def __init__(self, cuda_index):
        import ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.ct = ctypes
        self.h = ctypes.c_void_p()
        bus = None
        try:
            import torch
            p = torch.cuda.get_device_properties(cuda_index)
            bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
        except Exception:
            bus = None
        ok = bus is not None and self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")

    def sample(self):
        ct = self.ct
        sm, mx, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(sm))          # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        have_pw = self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw)) == 0
        self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, ct.byref(rs))
        r = rs.value
        act = lambda bit: "Active" if r & bit else "Not Active"
        return {"t": time.time(), "sm": float(sm.value), "max": float(mx.value),
                "power": pw.value / 1000.0 if have_pw else None,
                "hw": act(self.HW_SLOWDOWN | self.HW_POWER_BRAKE), "hw_thermal": act(self.HW_THERMAL),
                "sw_thermal": act(self.SW_THERMAL), "sw_power": act(self.SW_POWER_CAP)}


class ClockSampler:
    """SM clock and clock-event reasons sampled in the background every 10 ms
    (NVML through ctypes; nvidia-smi every 20 ms as the fallback), from before the
    warm-up to after the measurements, so that even a short timed region is spanned
    by samples."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        import threading
        self.rows, self.proc, self.nvml = [], None, None
        self.stop_flag = threading.Event()
        try:
            self.nvml = _Nvml(gpu_index)
            self.source = "nvml, 10 ms"
            self.thread = threading.Thread(target=self._poll, daemon=True)
        except Exception:
            self.nvml = None
            self.source = "nvidia-smi, 20 ms"
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            except Exception:
                self.proc = None
            self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self):
        while not self.stop_flag.is_set():
            try:
                self.rows.append(self.nvml.sample())
            except Exception:
                pass
            self.stop_flag.wait(0.01)

    def _read(self):
        if self.proc is None:
            return
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                self.rows.append({"t": time.time(), "sm": float(parts[2]), "max": float(parts[3]),
                                  "power": float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else None,
                                  "hw": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8],
                                  "sw_power": parts[9]})
            except ValueError:
                continue

    def wait_first(self, timeout=10.0):
        t0 = time.time()
        while not self.rows and time.time() - t0 < timeout:
            time.sleep(0.01)

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            import signal
            self.proc.send_signal(signal.SIGINT)
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self.thread.join(timeout=5)
        return list(self.rows)


def summarize_clocks(rows, t0, t1, source=""):
    """Samples inside [t0, t1], plus the last one before and the first one after it,
    so that a timed region shorter than the sampling interval is still spanned."""
    inside = [r for r in rows if t0 <= r["t"] <= t1]
    before = [r for r in rows if r["t"] < t0]
    after = [r for r in rows if r["t"] > t1]
    span = ([before[-1]] if before else []) + inside + ([after[0]] if after else [])
    if not span:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0,
                "source": source}
    reasons = set()
    for r in span:
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in span), "sm_max_mhz": max(r["max"] for r in span),
            "reasons": sorted(reasons), "samples": len(span), "samples_inside": len(inside),
            "window": "timed region, with the nearest sample on each side", "source": source}


def traffic_for(case, kernel):
    """ncu DRAM bytes per launch of the kernel in slot `kernel` on workload `case`
    ("<workload> <dtype>"), if measured on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(case, {}).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != d["source_sha256"]:
            return None  # kernel changed since the counters were taken
    return d["dram_bytes_per_launch"]


# --------------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def memory_versus_dense(d):
    """Peak device memory of one differentiable fwd + bwd beyond the resident inputs:
    this library (autograd wrapper, both bias gradients) against plain PyTorch
    attention that materialises the L×L scores (context for the pages' memory claim)."""
    import torch
    from memory_efficient_biased_gb300.autograd import evoformer_attention

    def dense(q, k, v, b1, b2):
        sc = torch.einsum("bnihd,bnjhd->bnhij", q, k) * (q.shape[-1] ** -0.5)
        if b1 is not None:
            sc = sc + b1
        if b2 is not None:
            sc = sc + b2
        return torch.einsum("bnhij,bnjhd->bnihd", torch.softmax(sc, dim=-1), v)

    peaks = {}
    for name in ("ours", "dense"):
        leaves = [None if d[n] is None else d[n].detach().clone().requires_grad_(True)
                  for n in ("q", "k", "v", "bias1", "bias2")]
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        try:
            q, k, v, b1, b2 = leaves
            out = evoformer_attention(q, k, v, [b1, b2]) if name == "ours" else dense(q, k, v, b1, b2)
            out.backward(d["do"])
            torch.cuda.synchronize()
            peaks[name] = torch.cuda.max_memory_allocated() - base
        except torch.cuda.OutOfMemoryError:
            peaks[name] = None
        del leaves
        out = q = k = v = b1 = b2 = None
        torch.cuda.empty_cache()
    ratio = peaks["dense"] / peaks["ours"] if peaks["dense"] and peaks["ours"] else None
    return {"ours_fwd_bwd_bytes": peaks["ours"], "dense_fwd_bwd_bytes": peaks["dense"], "dense_over_ours": ratio}


def bias2_groups(w) -> int:
    """n-groups of the two-stage pair-bias gradient: the library's rule (at least two
    waves of 152 (b, h, query tile, key tile, group) blocks; among up to four times as
    many groups, the fewest that fill the last wave to 95 %, else the fullest)."""
    qt = -(-w.L // 128)
    tiles = w.B * w.H * qt * qt
    n = max(1, w.N)
    g0 = max(1, min(n, -(-304 // tiles)))
    best, best_eff = 0, -1.0
    for g in range(g0, min(4 * g0, n) + 1):
        gs = -(-n // g)
        ge = -(-n // gs)
        ctas = tiles * ge
        eff = ctas / (-(-ctas // 152) * 152)
        if eff > best_eff + 1e-9:
            best, best_eff = ge, eff
        if eff >= 0.95:
            break
    return best


def bwd_mode(w, skip=False) -> str:
    """Which backward kernel the library runs for this shape (its TMEM-fit rule)."""
    dp = 16 if w.D <= 16 else (32 if w.D <= 32 else 64)
    qt = -(-w.L // 128)
    if dp <= 32 and 384 + 2 * dp + qt * dp <= 512:
        return "key-major"
    if dp <= 32:  # the streamed key-major kernel; with masked-tile skipping, the per-key-tile one
        return "main" if skip else "key-major, dQ streamed"
    if 320 + 2 * dp + qt * dp <= 512:
        return "slice"
    return "main"


def max_over_ranks(x: float) -> float:
    """Maximum of a per-rank float over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    from memory_efficient_biased_gb300.workload import WORKLOADS, workload_inputs
    w = WORKLOADS[args.workload]
    inp = workload_inputs(args.workload, args.dtype)
    t_row = oracle_row_seconds(inp)
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    rows = int(max(1, min(w.N, budget // t_row)))
    for _ in range(args.warmup):
        oracle_step(inp, rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(inp, rows)
        times.append(time.perf_counter() - t0)
    per_step = sum(times) / len(times)
    f = flops(w)["step"] * rows / w.N
    value = f / per_step / 1e12
    sample = f"fp64 numpy oracle fwd+bwd of rows n<{rows} of N={w.N} (batch 0) per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "N": w.N, "L": w.L, "H": w.H, "D": w.D,
                       "input_dtype": args.dtype, "rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from memory_efficient_biased_gb300 import build as _build
    _build.build()
    from memory_efficient_biased_gb300 import evo_attn as E
    from memory_efficient_biased_gb300.workload import WORKLOADS, workload_inputs

    w = WORKLOADS[args.workload]
    if args.rows:
        w = dataclasses.replace(w, N=args.rows, name=f"{w.name} (N={args.rows}, reduced for profiling)")
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[args.dtype]
    # clocks are sampled from here to the end of the measurements
    sampler = ClockSampler(local) if rank == 0 else None
    inp = workload_inputs(args.workload, args.dtype, seed=rank)
    if args.rows:  # the first rows of the full workload's inputs (bias2 is shared by the rows)
        inp = {k: (None if v is None else (v if k == "bias2" else v[:, :args.rows].contiguous()))
               for k, v in inp.items()}
    has_b1, has_b2 = inp["bias1"] is not None, inp["bias2"] is not None
    shape = (w.B, w.N, w.L, w.H, w.D)
    ws_bytes = E.evo_attn_bwd_workspace_bytes(shape, dt, has_b2)
    qkv = inp["q"].numel() * 2
    per_rep = 9 * qkv + ws_bytes + (2 * inp["bias2"].numel() * 2 if has_b2 else 0)
    R = int(min(8, max(1, math.ceil(3 * L2_BYTES / per_rep))))

    def replica():
        d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty((w.B, w.N, w.H, w.L), dtype=torch.float32, device="cuda")
        for k in ("dq", "dk", "dv"):
            d[k] = torch.empty_like(d["q"])
        d["db2"] = torch.empty_like(d["bias2"]) if has_b2 else None
        d["ws"] = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
        return d

    reps = [replica() for _ in range(R)]

    skip = dict(skip_masked_tiles=args.skip_masked_tiles, skip_threshold=-1.0e4)

    def step(d, events=None):
        E.evo_attn_fwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out=d["out"], lse=d["lse"],
                            events=events, **skip)
        E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], d["out"], d["lse"], d["do"],
                            dq=d["dq"], dk=d["dk"], dv=d["dv"], dbias2=d["db2"], workspace=d["ws"], events=events,
                            **skip)

    def status_ok():
        return E.evo_attn_device_status() == 0 and all(E.evo_attn_bwd_status(d["ws"]) == 0 for d in reps if d["ws"]
                                                       is not None)

    # peak device memory per call (outputs + workspace the call needs), before anything else is cached
    torch.cuda.synchronize()
    d0 = reps[0]
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    out, lse = E.evo_attn_fwd(d0["q"], d0["k"], d0["v"], d0["bias1"], d0["bias2"])
    torch.cuda.synchronize()
    peak_fwd = torch.cuda.max_memory_allocated() - base
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    E.evo_attn_bwd(d0["q"], d0["k"], d0["v"], d0["bias1"], d0["bias2"], out, lse, d0["do"])
    torch.cuda.synchronize()
    peak_bwd = torch.cuda.max_memory_allocated() - base
    memory = memory_versus_dense(d0) if rank == 0 else None
    del out, lse
    if not status_ok():
        raise RuntimeError("device wait timed out during set-up")

    # two graphs per replica: the timed one (the step alone) and an instrumented one with
    # the library's profiling events between its kernels, replayed after the timed region
    # for the per-kernel times (each event node adds a few microseconds to a step, so the
    # headline is never taken with them)
    n_ev = 8 if has_b2 else 6
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(R)]
    for d in reps:
        step(d)  # lazy one-time set-up outside capture
    torch.cuda.synchronize()
    graphs, igraphs = [], []
    cap_stream = torch.cuda.Stream()
    for r, d in enumerate(reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            step(d)
        graphs.append(g)
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi, stream=cap_stream):
            step(d, events=evs[r])
        igraphs.append(gi)
    torch.cuda.synchronize()

    if sampler:
        sampler.wait_first()
    for k in range(args.warmup):
        graphs[k % R].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record()
    for k in range(args.steps):
        graphs[k % R].replay()
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end))
    if not status_ok():
        raise RuntimeError("device wait timed out during the timed region")

    # per-kernel durations: the instrumented graphs, replayed as many steps as were timed
    # (at most 200), each replica's events read after its last replay
    ksteps = max(R, min(args.steps, 200))
    ti0, ti1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ti0.record()
    for k in range(ksteps):
        igraphs[k % R].replay()
    ti1.record()
    torch.cuda.synchronize()
    ms_instrumented = ti0.elapsed_time(ti1) / ksteps
    clock_rows = sampler.stop() if sampler else []
    if not status_ok():
        raise RuntimeError("device wait timed out during the instrumented replays")
    # the slots of the kernels that launch (no dQ cast kernel: every schedule writes dQ itself)
    mode = bwd_mode(w, args.skip_masked_tiles)
    names = ["fwd", "bwd_pre", "bwd_main"] + (["bwd_db2_part", "bwd_db2_sum"] if has_b2 else [])
    pairs = [(0, 1), (2, 3), (3, 4)] + ([(5, 6), (6, 7)] if has_b2 else [])
    kern_ms = {n: statistics.mean(evs[r][a].elapsed_time(evs[r][b]) for r in range(R))
               for n, (a, b) in zip(names, pairs)}

    F = flops(w)
    ms_step = ms_total / args.steps
    bwd_ms = sum(v for k, v in kern_ms.items() if k != "fwd")  # every backward kernel of the step
    value = world * F["step"] / (ms_step * 1e-3) / 1e12
    fwd_tflops = F["fwd"] / (kern_ms["fwd"] * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    # algorithmic work of each kernel per launch
    E_el = w.B * w.N * w.H * w.L * w.L
    bnhl = w.B * w.N * w.H * w.L
    b1b = w.B * w.N * w.L * 2 if has_b1 else 0
    b2b = w.B * w.H * w.L * w.L * 2 if has_b2 else 0
    work = {
        "fwd": ("tensor", F["fwd"]),
        "bwd_main": ("tensor", F["bwd"]),
        "bwd_db2_part": ("tensor", 4.0 * E_el * w.D),
        # O, dO read, delta written; plus the transposed pair-bias copy (key-major mode)
        "bwd_pre": ("hbm", 2 * qkv + bnhl * 4 + (2 * b2b if mode.startswith("key-major") else 0)),
        "bwd_db2_sum": ("hbm", bias2_groups(w) * w.B * w.H * w.L * w.L * 4 + b2b if has_b2 else 0),
    }
    # The kernels are timed in windows far shorter than the seconds-long loop of the
    # sustained figure, at full SM clock: the burst bf16 peak is the denominator.
    tpeak = peaks["bf16_tflops"]
    dom = max(kern_ms, key=kern_ms.get)
    bound, amount = work[dom]
    if bound == "tensor":
        achieved = amount / (kern_ms[dom] * 1e-3) / 1e12
        peak = tpeak
        unit = "TFLOP/s"
    else:
        achieved = amount / (kern_ms[dom] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": traffic_for(f"{w.name} {args.dtype}", dom),
                "peak_source": f"{peak_src} ({'bf16_tflops (burst)' if bound == 'tensor' else 'hbm_gbs'})"}

    # end to end through the host-buffer C-ABI step, pinned host memory
    pin = lambda t: None if t is None else t.pin_memory()
    h = {k: pin(v) for k, v in inp.items()}
    hout = {k: torch.empty_like(h["q"]).pin_memory() for k in ("out", "dq", "dk", "dv")}
    hdb2 = torch.empty_like(h["bias2"]).pin_memory() if has_b2 else None
    arena = torch.empty(E.evo_attn_step_host_arena_bytes(shape, dt, has_b1, has_b2), dtype=torch.uint8,
                        device="cuda")
    for d in reps[1:]:
        for key in list(d):
            d[key] = None
    torch.cuda.empty_cache()

    def host_step():
        E.evo_attn_step_host(h["q"], h["k"], h["v"], h["bias1"], h["bias2"], h["do"], hout["out"], None,
                             hout["dq"], hout["dk"], hout["dv"], hdb2, arena)

    for _ in range(2):
        host_step()
    torch.cuda.synchronize()
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n_e2e):
        host_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e)
    if E.evo_attn_device_status() != 0:
        raise RuntimeError("device wait timed out during the end-to-end run")
    h2d = sum(t.numel() * t.element_size() for t in (h["q"], h["k"], h["v"], h["do"], h["bias1"], h["bias2"])
              if t is not None)
    d2h = 4 * qkv + (hdb2.numel() * 2 if has_b2 else 0)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_row = oracle_row_seconds(inp)
        rows = int(max(1, min(w.N, 12.0 // t_row)))
        t0 = time.perf_counter()
        oracle_step(inp, rows)
        dt_cpu = time.perf_counter() - t0
        cpu = {"value": F["step"] * rows / w.N / dt_cpu / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
               "kind": "oracle",
               "sample": f"fp64 numpy oracle fwd+bwd of rows n<{rows} of N={w.N} (batch 0), {dt_cpu:.1f} s"}

    # forward; delta, the backward kernel, the skip bits (per-key-tile schedule with
    # skipping); the two pair-bias stages
    launches_per_step = (1 + 2 + (1 if mode == "main" and args.skip_masked_tiles and has_b1 else 0)
                         + (2 if has_b2 else 0))
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "N": w.N, "L": w.L, "H": w.H, "D": w.D,
                       "bias1": w.mask and f"{w.mask[0]} {w.mask[1]}", "bias2": has_b2, "backward": mode,
                       "masked_tile_skip": (("on: key tiles whose bias1 is all <= -1e4 are skipped; TFLOP/s "
                                             "counts the full shape's nominal FLOPs") if args.skip_masked_tiles
                                            else "off"),
                       "l2": (f"inputs larger than L2: {R} rotating replicas of {per_rep / 1e6:.0f} MB"
                              if R * per_rep >= L2_BYTES else
                              f"L2-warm: {R} replicas of {per_rep / 1e6:.1f} MB fit in L2 (small case)"),
                       "parallelism": f"{world} independent replicas" if world > 1 else "single GPU"},
            "fwd_tflops": fwd_tflops,
            "fwd_frac_of_peak": fwd_tflops / tpeak,
            "bwd_tflops": F["bwd"] / (bwd_ms * 1e-3) / 1e12,
            "bwd_frac_of_peak": F["bwd"] / (bwd_ms * 1e-3) / 1e12 / tpeak,
            "fwd_bwd_frac_of_peak": value / world / tpeak,
            "peak_used": f"bf16_tflops (burst) = {tpeak} TFLOP/s, {peak_src}",
            "kernel_ms": kern_ms,
            "kernel_ms_source": (f"CUDA events the library records between its kernels, {ksteps} replays of "
                                 f"instrumented copies of the timed graphs right after the timed region "
                                 f"({ms_instrumented:.4f} ms/step with the events; the timed steps run without them)"),
            "peak_mem_bytes": {"fwd_call": peak_fwd, "bwd_call": peak_bwd},
            "memory_vs_dense": memory,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": world * F["step"] / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": summarize_clocks(clock_rows, wall0, wall1, sampler.source if sampler else ""),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# --------------------------------------------------------------------------- microbenchmarks
# (kind, name, results per chain step): ops counted are exponentials, or fp32 FMA lane-ops
MICRO_EXP = [(0, "ex2.approx.ftz.f32", 1), (1, "ex2.approx.f16x2", 2), (2, "ex2.approx.ftz.bf16x2", 2),
             (3, "polynomial 2^x, scalar fma", 1), (4, "polynomial 2^x, fma.f32x2", 1), (5, "fma.rn.f32", 1),
             (6, "fma.rn.f32x2", 1), (7, "mix: 6 ex2.f32 + 1 packed polynomial pair", 1)]


def run_micro(args):
    """Per-SM-clock throughput of the exponential forms and of tcgen05.mma issue
    (libevo_micro.so); one JSON line per measurement."""
    import ctypes
    import torch
    from memory_efficient_biased_gb300 import build as _build
    _build.build()
    lib = ctypes.CDLL(_build.MICRO_LIB)
    torch.cuda.set_device(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    sink = torch.zeros(512, dtype=torch.float32, device="cuda")
    sampler = ClockSampler(0)
    sampler.wait_first()
    blocks, iters, threads, chains = 4 * sms, 1 << 14, 512, 8
    cyc = torch.zeros(blocks, dtype=torch.int64, device="cuda")
    for kind, name, per_instr in MICRO_EXP:
        best = None
        for rep in range(4):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            rc = lib.evo_micro_exp(kind, blocks, iters, ctypes.c_void_p(sink.data_ptr()),
                                   ctypes.c_void_p(cyc.data_ptr()), stream)
            e1.record()
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError(f"micro_exp kind {kind}: cuda error {rc}")
            cycles = statistics.median(cyc.cpu().tolist())
            if rep > 0 and (best is None or cycles < best[0]):
                best = (cycles, e0.elapsed_time(e1))
        cycles, ms = best
        ops = blocks * threads * iters * chains * per_instr
        clk = statistics.median(r["sm"] for r in sampler.rows[-20:]) if sampler.rows else None
        print(json.dumps({"micro": "exp", "op": name, "ops_per_s": ops / (ms * 1e-3),
                          "ops_per_sm_per_clock_at_sampled_clock": (ops / (ms * 1e-3) / sms / (clk * 1e6)
                                                                    if clk else None),
                          "sampled_sm_mhz": clk, "kernel_ms": ms, "blocks": blocks, "threads": threads,
                          "iters": iters, "chains": chains}), flush=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mcyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    reps = 4096
    for n in (32, 64, 128, 256):
        for ts in (0, 1):
            for accs in (1, 2, 4, 8):
                if accs * n > 256:
                    continue
                vals = []
                for rep in range(3):
                    rc = lib.evo_micro_mma(n, ts, accs, sms, reps, ctypes.c_void_p(mcyc.data_ptr()),
                                           ctypes.c_void_p(status.data_ptr()), stream)
                    torch.cuda.synchronize()
                    if rc != 0 or int(status.item()) != 0:
                        raise RuntimeError(f"micro_mma N={n} ts={ts}: rc {rc} status {int(status.item())}")
                    vals.append(statistics.median(mcyc.cpu().tolist()) / reps)
                cpi = min(vals[1:])
                print(json.dumps({"micro": "mma", "form": "TS (A in TMEM)" if ts else "SS (A, B in smem)",
                                  "M": 128, "N": n, "K": 16, "independent_accumulators": accs,
                                  "cycles_per_mma": cpi, "flop_per_sm_per_clock": 2 * 128 * n * 16 / cpi}),
                      flush=True)
    forms = ["A from TMEM, B MN-major 64B (forward P.V)", "A MN-major 128B, B MN-major 64B (backward dV, dK)",
             "A K-major 128B, B MN-major 64B (backward dQ)", "A and B K-major 64B (reference)"]
    for form, what in enumerate(forms):
        vals = []
        for rep in range(3):
            rc = lib.evo_micro_mma_form(form, sms, 4096, ctypes.c_void_p(mcyc.data_ptr()),
                                        ctypes.c_void_p(status.data_ptr()), stream)
            torch.cuda.synchronize()
            if rc != 0 or int(status.item()) != 0:
                raise RuntimeError(f"micro_mma_form {form}: rc {rc} status {int(status.item())}")
            vals.append(statistics.median(mcyc.cpu().tolist()) / 4096)
        print(json.dumps({"micro": "mma_form", "form": what, "M": 128, "N": 32, "K": 16,
                          "cycles_per_mma": min(vals[1:])}), flush=True)
    for pw in (1, 2, 4):
        vals = []
        for rep in range(3):
            rc = lib.evo_micro_tmem_ld(pw, sms, 4096, ctypes.c_void_p(mcyc.data_ptr()), ctypes.c_void_p(sink.data_ptr()),
                                       stream)
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError(f"micro_tmem_ld {pw}: rc {rc}")
            vals.append(statistics.median(mcyc.cpu().tolist()) / 4096)
        print(json.dumps({"micro": "tmem_ld", "loads_per_wait": pw, "columns_per_load": 32,
                          "cycles_per_round": min(vals[1:])}), flush=True)
    modes = ["none", "TMEM loads (4 x32 per wait)", "TMEM stores (4 x16 per wait)", "TMEM loads then stores",
             "shared-memory loads and stores", "ex2 chains", "TMEM loads (2 x64 per wait)",
             "TMEM loads (8 x16 per wait)"]
    creps = [0, 3000, 3000, 2000, 3000, 600, 3000, 3000]
    tmem_bytes = [0, 16384, 8192, 24576, 0, 0, 16384, 16384]  # per traffic warp and round
    ccyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    csink = torch.zeros(384, dtype=torch.float32, device="cuda")
    for ss in (0, 1):
        for n in (32, 48):
            for mode, what in enumerate(modes):
                if ss and n == 48:
                    continue
                vals, tcyc = [], []
                for rep in range(3):
                    rc = lib.evo_micro_contend(mode, n, ss, sms, 4096, creps[mode], ctypes.c_void_p(mcyc.data_ptr()),
                                               ctypes.c_void_p(ccyc.data_ptr()), ctypes.c_void_p(csink.data_ptr()),
                                               ctypes.c_void_p(status.data_ptr()), stream)
                    torch.cuda.synchronize()
                    if rc != 0 or int(status.item()) != 0:
                        raise RuntimeError(f"micro_contend {mode} N={n}: rc {rc} status {int(status.item())}")
                    vals.append(statistics.median(mcyc.cpu().tolist()) / 4096)
                    tcyc.append(statistics.median(ccyc.cpu().tolist()))
                form = "A K-major 128B in smem" if ss else "A from TMEM"
                rec = {"micro": "mma_contend", "form": form + ", B MN-major 64B", "N": n, "other_warps": what,
                       "cycles_per_mma": min(vals[1:])}
                if tmem_bytes[mode] and mode != 0:
                    rec["traffic_tmem_bytes_per_clock"] = 8 * tmem_bytes[mode] * creps[mode] / max(tcyc[1:])
                    rec["traffic_cycles_per_round"] = max(tcyc[1:]) / creps[mode]
                print(json.dumps(rec), flush=True)
    micro_host_link(lib, sms)
    rows = sampler.stop()
    print(json.dumps({"micro": "clocks", **summarize_clocks(rows, 0, 1e18, sampler.source)}), flush=True)
    return 0


def micro_host_link(lib, sms, nbytes=512 << 20):
    """Host <-> device bandwidth between pinned host memory and HBM: the copy engines one
    direction at a time and both at once, and copies by the SMs through mapped pinned
    memory.  These rates bound the host-buffer step (its e2e number)."""
    import ctypes
    import torch
    h_in = torch.ones(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_b = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / reps

    def duplex():
        cur = torch.cuda.current_stream()
        for st in (s_up, s_down):
            st.wait_stream(cur)
        with torch.cuda.stream(s_up):
            d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s_down):
            h_out.copy_(d_b, non_blocking=True)
        for st in (s_up, s_down):
            cur.wait_stream(st)

    rec = {"micro": "host_link", "bytes": nbytes,
           "copy_engine_h2d_gbs": nbytes / timed(lambda: d_a.copy_(h_in, non_blocking=True)) / 1e9,
           "copy_engine_d2h_gbs": nbytes / timed(lambda: h_out.copy_(d_b, non_blocking=True)) / 1e9,
           "copy_engine_both_directions_gbs": 2 * nbytes / timed(duplex) / 1e9}
    lib.evo_micro_host_ptr.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    lib.evo_micro_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    p_in, p_out = ctypes.c_void_p(), ctypes.c_void_p()
    r_in = lib.evo_micro_host_ptr(ctypes.c_void_p(h_in.data_ptr()), ctypes.byref(p_in))
    r_out = lib.evo_micro_host_ptr(ctypes.c_void_p(h_out.data_ptr()), ctypes.byref(p_out))
    if r_in == 0 and r_out == 0 and p_in.value and p_out.value:  # SM copies only through mapped memory
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

        def sm_copy(src, dst):
            rc = lib.evo_micro_copy(src, dst, nbytes, 2 * sms, st)
            if rc != 0:
                raise RuntimeError(f"micro_copy: cuda error {rc}")

        rec["sm_copy_h2d_gbs"] = nbytes / timed(lambda: sm_copy(p_in, ctypes.c_void_p(d_a.data_ptr()))) / 1e9
        rec["sm_copy_d2h_gbs"] = nbytes / timed(lambda: sm_copy(ctypes.c_void_p(d_b.data_ptr()), p_out)) / 1e9
        if not torch.equal(d_a[:4096].cpu(), h_in[:4096]):
            raise RuntimeError("micro_copy: wrong bytes")
    else:
        rec["sm_copy"] = "pinned memory not mapped into the device address space"
    print(json.dumps(rec), flush=True)


def main():
    args = parse_args()
    if args.micro:
        return run_micro(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
