"""Benchmark of the chunkwise DPLR-decay linear-attention forward on GB300.

One step = one whole forward (every row of the hot path) over one batch of the
synthetic workload, inputs resident in HBM: the fused per-head kernel for Gated
DeltaNet with bf16 inputs at d = 128, the two stages (chunk maps, then state scan)
otherwise. Prints ONE JSON line (rank 0). The default workload is Gated DeltaNet
B=8 H=16 T=8192 d=128 bf16 (the training-shaped case, T = 8K).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 0..4] [--impl ours|reference]

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica of the
workload (independent heads: no data-path collective), so the scaling is weak;
the value is the tokens of all ranks divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

DEFAULT_WORKLOAD = 2
# The headline metric: forward tokens/s (and TFLOP/s) at T = 8K-128K on one GB300, with the fraction of the roofline.
METRIC = "fwd tokens/s & TFLOP/s at T=8K\u2013128K on 1 GB300; % of roofline"
L2_BYTES = 129 * 2 ** 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ----------------------------------------------------------------------------
# Algorithmic work per token and head (the chunkwise algorithm's formula).
# ----------------------------------------------------------------------------

def folded_ranks(w):
    """GDN and HDLA fold the write term into A (K = beta k lies in span(A)), so r_kv counts as 0."""
    return (w.r_ab, 0) if w.mode in ("gdn", "hdla") else (w.r_ab, w.r_kv)


def flops_per_token(w):
    """d^2 (4r + 2p + 2) + C d (3r^2 + 2rp + 2r + 2p) + C^2 r^3 / 3 with dk = dv = d (mean of dk, dv
    otherwise), C = 64: state pass and inter-chunk readout, Gram blocks / solve applications /
    intra-chunk scores, and the Cr x Cr triangular inverse."""
    r, p = folded_ranks(w)
    d = 0.5 * (w.dk + w.dv)
    C = 64
    return d * d * (4 * r + 2 * p + 2) + C * d * (3 * r * r + 2 * r * p + 2 * r + 2 * p) + C * C * r ** 3 / 3.0


def bytes_per_token(w):
    """Compulsory HBM bytes per token and head: inputs read once, o (fp32) written once."""
    e = 2 if w.dtype == "bf16" else 4
    if w.mode in ("gdn", "hdla"):
        b = e * (2 * w.dk + w.dv) + 4 + 4 * w.dv
        b += 4 if w.mode == "gdn" else 4 * w.dk
    else:
        b = e * (w.dk + 2 * w.r_ab * w.dk + w.r_kv * (w.dk + w.dv)) + 4 * w.dk + 4 * w.dv
    return b


def step_bytes(w):
    state = 4 * w.dk * w.dv * (1 + (1 if w.nonzero_s0 else 0))
    return w.B * w.H * (w.T * bytes_per_token(w) + state)


# ----------------------------------------------------------------------------
# Clock sampling during the timed region.
# ----------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")


class ClockSampler:
    def __init__(self, gpu_index, interval_ms=100):
        """gpu_index: anything nvidia-smi --id accepts (ordinal or UUID)."""
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", f"-lms={interval_ms}"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "mem_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm, smax, mem, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
            try:
                mem.append(float(r[9]))
            except (IndexError, ValueError):
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "mem_mhz": statistics.median(mem) if mem else None, "reasons": sorted(reasons), "samples": len(sm)}


def effective_sm_mhz(dev, cycles=20_000_000):
    """SM clock cycles (clock64) per microsecond of a spin of `cycles` cycles, timed with CUDA events:
    the clock the kernels actually ran at, next to the clock nvidia-smi reports. Median of three."""
    import torch
    if not hasattr(torch.cuda, "_sleep"):
        return None
    with torch.cuda.device(dev):
        torch.cuda._sleep(cycles // 20)
        vals = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.cuda._sleep(cycles)
            e1.record()
            torch.cuda.synchronize(dev)
            vals.append(cycles / (e0.elapsed_time(e1) * 1e3))
    return round(statistics.median(vals), 1)


# ----------------------------------------------------------------------------
# Helpers.
# ----------------------------------------------------------------------------

def slowest_ms(ms, world, device):
    """The largest per-rank time of a step (all ranks call it; single process: ms itself)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as tdist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, slowest):
    """Whole-job throughput: every rank processes its own replica of the workload."""
    return world * tokens_per_rank / (slowest * 1e-3)


def smi_id(dev):
    """nvidia-smi --id for a torch device: its UUID when torch exposes it, else the ordinal."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        return str(dev.index)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def oracle_sample(w, seconds_hint=15.0):
    """Times the float64 oracle (as it stands) on a bounded sample of the workload: every head of
    the workload, a shorter sequence drawn with the same recipe. Returns (tokens/s, cores, text)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    T_s = min(w.T, 1024)
    inp = workloads.generate(w, heads=heads, T=T_s)
    t0 = time.perf_counter()
    oracle.forward_inputs(inp, threads=cores)
    dt = time.perf_counter() - t0
    # grow the sample toward the time hint (bounded by the workload's own length)
    if dt < seconds_hint / 4 and T_s < w.T:
        T_s = int(min(w.T, T_s * max(2.0, seconds_hint / max(dt, 1e-3))))
        T_s = max(64, T_s // 64 * 64)
        inp = workloads.generate(w, heads=heads, T=T_s)
        t0 = time.perf_counter()
        oracle.forward_inputs(inp, threads=cores)
        dt = time.perf_counter() - t0
    ntask = len(heads) * ((w.dv + 15) // 16)
    toks = len(heads) * T_s
    return toks / dt, min(cores, ntask), f"{len(heads)} heads x {T_s} tokens (same recipe), {dt:.1f} s", dt


def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel_name, workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel_name, {}).get(workload_name)
        if not ent:
            return None
        srcs = [os.path.join(ROOT, s) for s in ent["sources"]]
        if source_digest(srcs) != ent["source_sha"]:
            return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------
# Arms.
# ----------------------------------------------------------------------------

def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return
    steps, warm = args.steps, args.warmup
    cores = len(os.sched_getaffinity(0))
    import oracle
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    T_s = min(w.T, 1024)
    inp = workloads.generate(w, heads=heads, T=T_s)
    for _ in range(warm):
        oracle.forward_inputs(inp, threads=cores)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.forward_inputs(inp, threads=cores)
    dt = (time.perf_counter() - t0) / max(steps, 1)
    toks = len(heads) * T_s
    value = toks / dt
    sample = f"{len(heads)} heads x {T_s} tokens of the workload recipe per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "mode": w.mode, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                   "r_ab": w.r_ab, "r_kv": w.r_kv, "chunk": w.chunk, "in_dtype": w.dtype, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, len(heads) * ((w.dv + 15) // 16)),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import torch.distributed as tdist

    import structured_decay_linear_gb300 as sdl

    rank, local_rank, world = dist_env()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        tdist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            tdist.barrier()

    lib_path = sdl.LIB_PATH
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = workloads.generate(w)
    names = ["q", "k", "v", "decay", "beta", "A", "Bm", "K", "V", "S0"]
    host = {}
    for key in names:
        x = inp[key]
        if x is None:
            host[key] = None
            continue
        t = torch.from_numpy(np.ascontiguousarray(x))
        if key in ("q", "k", "v", "A", "Bm", "K", "V"):
            t = t.to(dt)
        host[key] = t.pin_memory()
    dev_in = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    f = sdl.Forward(w.mode, dt, w.B, w.H, w.T, w.dk, w.dv, w.r_ab, w.r_kv, w.chunk, device=dev)
    maps_args = {k: dev_in[k] for k in names if k != "S0"}
    S0 = dev_in["S0"]
    in_bytes = sum(int(v.numel() * v.element_size()) for v in host.values() if v is not None)

    flush = None
    if in_bytes < 4 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        if f.kernels == 1:
            f(**maps_args, S0=S0, check=False)
        else:
            f.chunk_maps(**maps_args)
            f.state_scan(S0)
    torch.cuda.synchronize(dev)

    K = args.steps
    fused = f.kernels == 1
    fwd_args = dict(maps_args, S0=S0)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(smi_id(dev))
    barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        if fused:
            f(**fwd_args, check=False)          # dplr_la_forward: one fused kernel
            ev[i][1].record(stream)
            ev[i][2].record(stream)
        else:
            f.chunk_maps(**maps_args)           # stage 1 then stage 2: the same kernels as dplr_la_forward
            ev[i][1].record(stream)
            f.state_scan(S0)
            ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    clocks["sm_mhz_effective"] = effective_sm_mhz(dev)
    k1 = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    k2 = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    step_ms = slowest_ms(sum(a + b for a, b in zip(k1, k2)) / K, world, dev)
    toks = w.B * w.H * w.T
    value = job_tokens_per_s(toks, world, step_ms)
    flops = flops_per_token(w) * w.B * w.H * w.T
    sbytes = step_bytes(w)

    # end-to-end through the public C ABI with host buffers (pinned): dplr_la_forward_host_seq copies
    # every input in, runs the forward and copies o and S_T back, all inside the timed region
    # (the sequence in segments: the copies of one segment overlap the forwards and copies of the others).
    fh = sdl.ForwardHostSeq(w.mode, dt, w.B, w.H, w.T, w.dk, w.dv, w.r_ab, w.r_kv, w.chunk, device=dev)
    o_host, s_host = fh.o, fh.S_T

    def e2e_step():
        fh(**host)

    e2e_step()
    torch.cuda.synchronize(dev)
    ke = max(1, min(K, 10))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(ke):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = slowest_ms(e0.elapsed_time(e1) / ke, world, dev)
    h2d = in_bytes
    d2h = int(o_host.numel() * 4 + s_host.numel() * 4)

    # parity spot check of this very run (sampled head vs oracle) happens in the tests; here we only
    # guard against a broken run producing non-finite output.
    finite = bool(torch.isfinite(f.o).all().item() and torch.isfinite(f.S_T).all().item())

    if rank == 0:
        peaks, peak_kind = load_peaks()
        if fused:
            kern = [("dplr_fused_head", sum(k1) / K)]
        elif f.path == "hdla_tcgen05":
            kern = [("hdla_chunk_kernel", sum(k1) / K), ("hdla_chain_kernel", sum(k2) / K)]
        elif f.path == "generic_tcgen05":
            kern = [("generic_chunk_kernel", sum(k1) / K), ("generic_chain_kernel", sum(k2) / K)]
        else:
            kern = [("dplr_chunk_maps", sum(k1) / K), ("dplr_state_scan", sum(k2) / K)]
        dom_name, dom_ms = max(kern, key=lambda x: x[1])
        achieved = sbytes / (dom_ms * 1e-3) / 1e9
        traffic = measured_traffic(dom_name, w.name)
        if world == 1 and not args.no_cpu_baseline:
            cpu_v, cpu_cores, cpu_sample, _ = oracle_sample(w)
        else:
            cpu_v, cpu_cores, cpu_sample = None, None, "not run (rank 0 at N=1 only)"
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": max(args.warmup, 3),
            "ms_per_step": step_ms,
            "ms_per_step_median": statistics.median(a + b for a, b in zip(k1, k2)),   # this rank's steps
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            # arithmetic of the path's products: bf16 tensor-core operands (fp32 accumulation and state;
            # bf16 hi + lo pairs where one term is too coarse), fp16 hi + lo pairs with power-of-two scales
            # (the generic path), or fp32 on the CUDA cores
            "dtype": {"two_stage_fp32": "f32", "generic_tcgen05": "f16"}.get(f.path, "bf16"),
            "input_dtype": w.dtype,                        # storage type of q, k, v (A, B, K, V)
            "path": f.path,
            "data": "synthetic (seeded workload recipe, resident in HBM)",
            "config": {"workload": w.name, "mode": w.mode, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                       "r_ab": w.r_ab, "r_kv": w.r_kv, "chunk": w.chunk, "in_dtype": w.dtype,
                       "global_batch": w.B * world, "seq_len": w.T, "parallelism": f"replicas x{world}",
                       "l2": ("inputs larger than L2" if flush is None else "L2 flushed between steps")},
            "tflops": flops / (step_ms * 1e-3) / 1e12,
            "flops_per_step": flops,
            "bytes_per_step": sbytes,
            "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "peak_source": f"{peak_kind} hbm_gbs"},
            "step_roofline": {"achieved_gbs": sbytes / (step_ms * 1e-3) / 1e9,
                              "frac": sbytes / (step_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                              "flop_frac_of_bf16_peak": flops / (step_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
            "kernels_ms": {n: ms for n, ms in kern},
            "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": cpu_cores, "kind": "oracle",
                             "sample": cpu_sample},
            "e2e": {"value": job_tokens_per_s(toks, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "call": "dplr_la_forward_host_seq",
                    "segments": fh.segments, "slots": fh.slots},
            "gpu_launches": K * f.kernels,
            "clocks": clocks,
            "wall_s_timed_region": t_wall,
            "output_finite": finite,
            "library": os.path.relpath(lib_path, ROOT),
            "device": {"name": torch.cuda.get_device_name(dev),
                       "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()


def run_host_overhead(args):
    """Host time of one dplr_la_forward call (argument checks, plan, cached tensor maps, launch),
    measured through the C ABI on T = 64 problems. Calls are timed in bursts of 100 that start on
    an idle GPU, so that the launch queue never fills and the host never waits for the device; the
    best of 20 bursts is kept. The ctypes overhead is measured on dplr_la_check (no launch)."""
    import torch
    import structured_decay_linear_gb300 as sdl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    lines = []
    for mode, heads in (("gdn", 1), ("gdn", 16), ("hdla", 1), ("hdla", 16)):
        w = dataclasses_replace(workloads.WORKLOADS[2 if mode == "gdn" else 4], B=1, H=heads, T=64,
                                name=f"{mode}_bf16_b1h{heads}_t64_d128")
        inp = workloads.generate(w, heads=[(0, h) for h in range(heads)], T=64)
        dt = torch.bfloat16
        t = {k: (None if inp[k] is None else torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev))
             for k in ("q", "k", "v", "decay", "beta", "S0")}
        for k in ("q", "k", "v"):
            t[k] = t[k].to(dt)
        f = sdl.Forward(mode, dt, 1, heads, 64, 128, 128, device=dev)
        ptr = lambda x: None if x is None else x.data_ptr()
        call = lambda: sdl.dplr_la_forward(f.desc, ptr(t["q"]), ptr(t["k"]), ptr(t["v"]), ptr(t["decay"]),
                                           ptr(t["beta"]), None, None, None, None, ptr(t["S0"]), ptr(f.o),
                                           ptr(f.S_T), ptr(f.workspace), f.ws_bytes, stream)
        for _ in range(50):
            assert call() == 0
        torch.cuda.synchronize(dev)
        n, best = 100, float("inf")
        for _ in range(20):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            for _ in range(n):
                call()
            best = min(best, (time.perf_counter() - t0) / n * 1e6)
        host_us = best
        torch.cuda.synchronize(dev)
        n = 5000
        t0 = time.perf_counter()
        for _ in range(n):
            sdl.dplr_la_check(f.desc)
        ctypes_us = (time.perf_counter() - t0) / n * 1e6
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(200):
            call()
        e1.record()
        torch.cuda.synchronize(dev)
        lines.append({"workload": w.name, "kernels_per_call": f.kernels,
                      "host_us_per_call": host_us, "ctypes_us_per_check_call": ctypes_us,
                      "gpu_us_per_call_back_to_back": e0.elapsed_time(e1) / 200 * 1e3})
    print(json.dumps({"mode": "host_overhead", "burst": 100, "bursts": 20, "results": lines}), flush=True)


def run_decode(args):
    """Time of one decode step (dplr_la_decode_step, one token for every head) for the head counts of
    workloads 2 (GDN, B=8 H=16) and 4 (HDLA, B=1 H=16) at d = 128, bf16 inputs. The step reads and writes
    each head's fp32 state once: 2 * dk * dv * 4 bytes per head, plus the token's inputs. Timed with CUDA
    events over 200 steps launched back to back, and over 200 steps captured in one CUDA graph (no launch
    gaps). The state (8 MB and 1 MB) stays in L2 from step to step, so the figure is an L2-resident one."""
    import torch
    import structured_decay_linear_gb300 as sdl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    lines = []
    for wid in (2, 4):
        w = workloads.WORKLOADS[wid]
        inp = workloads.generate(w, T=1)
        t = {k: (None if inp[k] is None else torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev))
             for k in ("q", "k", "v", "decay", "beta", "S0")}
        for k in ("q", "k", "v"):
            t[k] = t[k].to(torch.bfloat16)
        step = sdl.Decode(w.mode, torch.bfloat16, w.B, w.H, w.dk, w.dv, S0=t["S0"], device=dev)
        call = lambda: step(q=t["q"], k=t["k"], v=t["v"], decay=t["decay"], beta=t["beta"])
        for _ in range(20):
            call()
        torch.cuda.synchronize(dev)
        n = 200
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            call()
        e1.record()
        torch.cuda.synchronize(dev)
        us_launch = e0.elapsed_time(e1) / n * 1e3
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            call()
            with torch.cuda.graph(g, stream=s):
                for _ in range(n):
                    call()
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        us_graph = e0.elapsed_time(e1) / n * 1e3
        heads = w.B * w.H
        state_bytes = heads * 2 * w.dk * w.dv * 4
        in_bytes = heads * (2 * (2 * w.dk + w.dv) + 4 + 4 * (1 if w.mode == "gdn" else w.dk)) + heads * w.dv * 4
        gbs = (state_bytes + in_bytes) / (us_graph * 1e-6) / 1e9
        lines.append({"workload": f"{w.mode}_bf16_b{w.B}h{w.H}_d128_decode", "heads": heads,
                      "us_per_step_launched": us_launch, "us_per_step_graph": us_graph,
                      "tokens_per_s_graph": heads / (us_graph * 1e-6), "bytes_per_step": state_bytes + in_bytes,
                      "achieved_gbs_graph": gbs, "frac_of_hbm_peak": gbs / peaks["hbm_gbs"],
                      "peak": f"{peak_kind} hbm_gbs {peaks['hbm_gbs']}"})
    print(json.dumps({"mode": "decode", "steps": 200, "results": lines}), flush=True)


def dataclasses_replace(w, **kw):
    import dataclasses
    return dataclasses.replace(w, **kw)


def run_hla(args):
    """Time of dplr_hla_forward (HLA's query-gated composition of GDN chunk transitions) on a synthetic HLA
    workload: GDN inputs of the workload recipe (bf16, d = 128) at B=1 H=16 T=4096 (the HLA page's 4K context),
    chunks of L = 256 tokens, gates sigmoid(N(-1, 2)) per (query, chunk) and the page's inference threshold 0.1.
    Not a benchmark line; the JSON carries "mode": "hla"."""
    import torch
    import structured_decay_linear_gb300 as sdl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T = args.seq_len or 4096
    L, theta, H = 256, 0.1, 16
    w = workloads.Workload(98, "hla_gdn_bf16_b1h16", "gdn", "bf16", 1, H, T, 128, 128, 1, 1, 64, False)
    inp = workloads.generate(w)
    N = (T + L - 1) // L
    z = np.random.default_rng(1).standard_normal((1, H, T, N)) * 2.0 - 1.0
    W = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    d = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to(dev).to(t)
    args_t = [d(inp["q"], torch.bfloat16), d(inp["k"], torch.bfloat16), d(inp["v"], torch.bfloat16),
              d(inp["decay"], torch.float32), d(inp["beta"], torch.float32), d(W, torch.float32)]
    f = sdl.HLA(torch.bfloat16, 1, H, T, 128, 128, L, device=dev)
    call = lambda: f(*args_t, theta)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        call()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / K
    # the gated pass's products: per 64-query block and history chunk with a gate >= theta, U A_j and U B_j
    Wt = np.where(W >= theta, W, 0.0)
    pairs = 0
    for qb in range(T // 64):
        c = (qb * 64) // L
        blk = Wt[0, :, qb * 64:(qb + 1) * 64, :c]
        pairs += int((blk.max(axis=1) > 0).sum())
    flops = pairs * 2 * (2 * 64 * 128 * 128)
    fwd = sdl.Forward("gdn", torch.bfloat16, 1, H, T, 128, 128, device=dev)
    for _ in range(3):
        fwd(q=args_t[0], k=args_t[1], v=args_t[2], decay=args_t[3], beta=args_t[4])
    torch.cuda.synchronize(dev)
    e0.record()
    for _ in range(K):
        fwd(q=args_t[0], k=args_t[1], v=args_t[2], decay=args_t[3], beta=args_t[4])
    e1.record()
    torch.cuda.synchronize(dev)
    ms_fwd = e0.elapsed_time(e1) / K
    print(json.dumps({"mode": "hla", "workload": f"hla_gdn_bf16_b1h{H}_t{T}_d128_L{L}", "steps": K, "ms_per_forward": ms,
                      "tokens_per_s": H * T / (ms * 1e-3), "gate_pairs_kept": pairs,
                      "gate_pairs_total": H * sum((qb * 64) // L for qb in range(T // 64)),
                      "gated_pass_tflops_over_the_call": flops / (ms * 1e-3) / 1e12, "gdn_forward_ms": ms_fwd,
                      "output_finite": bool(torch.isfinite(f.o).all().item()), "path": f.path,
                      "arithmetic": ("block maps, chunk composition and gated composition bf16 hi + lo on tcgen05, "
                                     "f32 accumulate and inverse" if f.path == "hla_gated_tcgen05"
                                     else "f32 (CUDA cores)")}),
          flush=True)


def run_gdp(args):
    """Time of dplr_gdp_forward (stacked Householders in the Gated DeltaProduct style: per token the gate, then n_h
    erase-and-write steps) at the generic workload's shape, B=2 H=8 T=8192 d=64, fp32 inputs, for n_h = 2 (the
    tensor-core generic stages) and n_h = 3 (the fp32 stages). Synthetic inputs: unit-norm k, beta in (0, 2),
    log-gates -softplus(-(N(0, 1) + 3)). Not a benchmark line; the JSON carries "mode": "gdp"."""
    import torch
    import structured_decay_linear_gb300 as sdl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, H, T, d = 2, 8, args.seq_len or 8192, 64
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    rn = lambda *shape: torch.randn(*shape, device=dev, generator=g)
    lines = []
    for nh in (2, 3):
        k = torch.nn.functional.normalize(rn(B, H, T, nh, d), dim=-1)
        x = dict(q=rn(B, H, T, d) / d ** 0.5, k=k, v=rn(B, H, T, nh, d),
                 g=-torch.nn.functional.softplus(-(rn(B, H, T) + 3)), beta=2 * torch.sigmoid(rn(B, H, T, nh)),
                 S0=0.1 * rn(B, H, d, d))
        f = sdl.GDP(torch.float32, B, H, T, d, d, nh, device=dev)
        call = lambda: f(**x)
        for _ in range(max(args.warmup, 3)):
            call()
        torch.cuda.synchronize(dev)
        K = args.steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            call()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / K
        lines.append({"workload": f"gdp_nh{nh}_f32_b{B}h{H}_t{T}_d{d}", "n_h": nh, "path": f.path, "ms_per_forward": ms,
                      "tokens_per_s": B * H * T / (ms * 1e-3),
                      "output_finite": bool(torch.isfinite(f.o).all().item() and torch.isfinite(f.S_T).all().item())})
    print(json.dumps({"mode": "gdp", "steps": args.steps, "results": lines}), flush=True)


def run_backward(args):
    """Time of dplr_la_backward (the gradients of every input given dO and dS_T) on a workload at full size, with
    the same recipe as the forward and random upstream gradients. Reports ms per backward and tokens/s, and the
    algorithmic bytes per backward: the forward's inputs and S0 read, dO and dS_T read, every gradient written
    once in fp32 (not a benchmark line; the JSON carries "mode": "backward")."""
    import torch
    import structured_decay_linear_gb300 as sdl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    if args.seq_len:
        w = dataclasses.replace(w, T=args.seq_len)
    inp = workloads.generate(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    t = {}
    for k in ("q", "k", "v", "A", "Bm", "K", "V"):
        t[k] = None if inp[k] is None else torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev).to(dt)
    for k in ("decay", "beta", "S0"):
        t[k] = None if inp[k] is None else torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    dO = torch.randn((w.B, w.H, w.T, w.dv), device=dev, generator=g)
    dST = torch.randn((w.B, w.H, w.dk, w.dv), device=dev, generator=g)
    bw = sdl.Backward(w.mode, dt, w.B, w.H, w.T, w.dk, w.dv, w.r_ab if w.mode == "generic" else None,
                      w.r_kv if w.mode == "generic" else None, device=dev)
    call = lambda: bw(dO=dO, dST=dST, **t)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        call()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / K
    tokens = w.B * w.H * w.T
    esz = 2 if w.dtype == "bf16" else 4
    if w.mode == "generic":
        per_tok = (w.dk + 2 * w.r_ab * w.dk + w.r_kv * (w.dk + w.dv)) * (esz + 4) + w.dk * 8 + w.dv * 4
    else:
        dec = 1 if w.mode == "gdn" else w.dk
        per_tok = (2 * w.dk + w.dv) * (esz + 4) + 2 * (dec + 1) * 4 + w.dv * 4
    nbytes = tokens * per_tok + w.B * w.H * w.dk * w.dv * 4 * 3
    peaks, peak_kind = load_peaks()
    finite = all(bool(torch.isfinite(x).all().item()) for x in bw.grads.values())
    print(json.dumps({"mode": "backward", "workload": w.name, "T": w.T, "steps": K, "ms_per_backward": ms,
                      "tokens_per_s": tokens / (ms * 1e-3), "bytes_per_backward": nbytes,
                      "achieved_gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_hbm_peak": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "peak": f"{peak_kind} hbm_gbs {peaks['hbm_gbs']}", "workspace_bytes": bw.ws_bytes,
                      "gradients_finite": finite, "arithmetic": "f32 (CUDA cores)"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gdp", action="store_true",
                    help="time the stacked-Householder forward, n_h = 2 and 3 (not a benchmark line)")
    ap.add_argument("--hla", action="store_true",
                    help="time HLA's query-gated composition (dplr_hla_forward); not a benchmark line")
    ap.add_argument("--backward", action="store_true",
                    help="time dplr_la_backward on the workload (not a benchmark line)")
    ap.add_argument("--decode", action="store_true",
                    help="time the one-token decode step (not a benchmark line)")
    ap.add_argument("--host-overhead", action="store_true",
                    help="time the host side of dplr_la_forward on T = 64 problems (not a benchmark line)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override the workload's T (smaller cases for profiling; not a benchmark line)")
    args = ap.parse_args()
    if args.host_overhead:
        run_host_overhead(args)
        return
    if args.gdp:
        run_gdp(args)
        return
    if args.hla:
        run_hla(args)
        return
    if args.backward:
        run_backward(args)
        return
    if args.decode:
        run_decode(args)
        return
    w = workloads.WORKLOADS[args.workload]
    if args.seq_len > 0:
        import dataclasses
        w = dataclasses.replace(w, T=args.seq_len, name=f"{w.name}_T{args.seq_len}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
