#!/usr/bin/env python3
"""Benchmark of the chunkwise linear-attention forward (libla.so) on GB300.

One step = one la_chunk_fwd call over one batch of the workload: the whole
hot path (staging, gate prefix, local scores, WY/UT solve, state-dependent
values, output, state passing) in one fused kernel launch. Default workload:
Gated DeltaNet, B=4, H=16, T=16384, dk=dv=128, bf16, C=64.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the path shards by (batch, head) with no exchange), timing is
the max over ranks and `value` sums the tokens of all ranks.

Prints ONE JSON line (rank 0). `--impl reference` times the float64 CPU
oracle on this host's cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "tokens/sec and TFLOP/s of chunk fwd at 1 GB300; % of roofline"
UNIT = "tokens/s"
PROFILE_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
_CS = "gated_delta_rule_linear_gb300/csrc/"
_COMMON = [_CS + "la_tc_common.cuh", _CS + "la_sm100.cuh"]
# The sources each workload's dominant kernel is built from: a recorded DRAM
# traffic figure stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "gdn": [_CS + "la_chunk_delta_pair.cu", _CS + "la_chunk_delta.cu", _CS + "la_wy.cuh"] + _COMMON,
    "kda": [_CS + "la_chunk_kda_wy.cu", _CS + "la_warp_mma.cuh", _CS + "la_wy.cuh"],
    "retnet": [_CS + "la_chunk_ws.cu"] + _COMMON,
    "gla": [_CS + "la_chunk_ws.cu"] + _COMMON,
    "outer": [_CS + "la_chunk_ws.cu"] + _COMMON,
    "scalar": [_CS + "la_chunk_ws.cu", _CS + "la_chunk_mat.cu"] + _COMMON,
    "elu1": [_CS + "la_chunk_ws.cu", _CS + "la_chunk_mat.cu"] + _COMMON,
    "linear_fp32": [_CS + "la_chunk_simt.cu"],
    "noncausal": [_CS + "la_chunk_mat.cu"] + _COMMON,
    "backward": [_CS + "la_backward.cu", _CS + "la_chunk_ws.cu", _CS + "la_chunk_mat.cu"] + _COMMON,
    "backward_scalar": [_CS + "la_backward.cu", _CS + "la_chunk_ws.cu", _CS + "la_chunk_mat.cu"] + _COMMON,
    "backward_gla": [_CS + "la_backward.cu", _CS + "la_chunk_ws.cu"] + _COMMON,
    "decode": [_CS + "la_step.cu"],
    "gdelta": [_CS + "la_chunk_gdelta.cu", _CS + "la_chunk_gdelta_wy.cu", _CS + "la_warp_mma.cuh"],
    "backward_gdn": [_CS + "la_backward_delta.cu", _CS + "la_warp_mma.cuh", _CS + "la_wy.cuh", _CS + "la_tc_common.cuh"],
    "backward_kda": [_CS + "la_backward_delta.cu", _CS + "la_warp_mma.cuh", _CS + "la_wy.cuh", _CS + "la_tc_common.cuh"],
    "prologue": [_CS + "la_prologue.cu", _CS + "la_sm100.cuh"],
    "prologue_gla": [_CS + "la_prologue.cu", _CS + "la_sm100.cuh"],
}


def uses_materialised(wl, variant=None, sm_count=152) -> bool:
    """Whether la_chunk_fwd runs the materialised variant for this workload
    (the library's per-shape rule, or a forced LA_VARIANT)."""
    if variant is not None:
        return variant == "mat" and wl.mode not in ("gdn", "kda", "outer")
    if wl.C == 128:
        return True
    bh = wl.B * wl.H
    small = 4 * bh <= sm_count if wl.mode == "gla" else True if wl.mode == "elu1" else 2 * bh <= sm_count
    return wl.dtype == "bf16" and wl.mode not in ("gdn", "kda", "outer") and wl.T >= 512 and small


def mat_chunk(wl) -> int:
    """The chunk length the materialised variant runs for this workload
    (the library's rule for C = 0, else the workload's C)."""
    if wl.C:
        return wl.C
    return 128 if wl.mode != "gla" and (wl.mode in ("linear", "elu1") or wl.T >= 2048) else 64


def is_noncausal(wl) -> bool:
    return bool(wl.extra.get("noncausal"))


def parallel_state_pass(wl) -> bool:
    """Whether the materialised variant's state pass runs as every chunk's partial
    plus a prefix scan (linear and elu+1, partials up to 2 GiB, unless
    LA_MAT_STATE=serial): three launches a call instead of two."""
    part = wl.B * wl.H * ((wl.T + 63) // 64) * wl.dk * (wl.dv * 4 + (4 if wl.mode == "elu1" else 0))
    return (wl.mode in ("linear", "elu1") and part <= (2 << 30)
            and os.environ.get("LA_MAT_STATE") != "serial")


def kernel_name(wl, variant=None, sm_count=152) -> str:
    """The kernel one la_chunk_fwd launch of this workload runs."""
    if is_noncausal(wl):
        return "nc_sum_kernel+nc_finalize_kernel+nc_out_kernel"
    if uses_materialised(wl, variant, sm_count):
        out = "chunk_output128_kernel" if mat_chunk(wl) == 128 else "chunk_output_kernel"
        if parallel_state_pass(wl):
            return "nc_sum_kernel+mat_scan_kernel+" + out
        return "chunk_state_kernel+" + out
    if wl.dtype == "f32" or variant == "simt":
        return "chunk_simt_kernel"
    if wl.mode == "kda":
        fused = variant in ("tc", "nonmat") or os.environ.get("LA_KDA") == "tc"
        return "chunk_tc_kernel" if fused else "kdw_pre_kernel+kdw_chain_kernel"
    if wl.mode == "gdn":
        if wl.dk == 128 and wl.dv == 128:
            path = os.environ.get("LA_DELTA", "pair" if 2 * wl.B * wl.H <= sm_count else "single")
            if variant == "mat":
                path = "wy"
            return {"pair": "chunk_delta_pair_kernel", "single": "chunk_delta_kernel"}.get(
                path, "wy_kernel+chain_kernel")
        return "chunk_tc_kernel"
    return "chunk_ws_kernel"


# ---------------------------------------------------------------- cost model

def flops_per_token_head(mode: str, dk: int, dv: int, C: int = 64) -> float:
    """Algorithmic FLOP per token and head of the chunk form, fixed at C=64.
    Unit write: scores 2*C*dk, local output 2*C*dv, inter output 2*dk*dv,
    state update 2*dk*dv. Delta rule adds K K^T (2*C*dk), the triangular solve
    (C^2/3), the WY products (2*C*dk + 2*C*dv) and the S-dependent correction
    (2*dk*dv). elu+1 carries one extra value column (the normaliser)."""
    if mode == "elu1":
        dv = dv + 1
    if mode in ("gdn", "kda"):  # the per-channel gate of kda changes no contraction size
        return 2 * C * (3 * dk + 2 * dv) + C * C / 3.0 + 6 * dk * dv
    if mode == "noncausal":  # K^T V and Q S: no scores
        return 4 * dk * dv
    return 2 * C * (dk + dv) + 4 * dk * dv


def algorithmic_bytes(wl, has_s0: bool) -> float:
    """Minimum HBM traffic of one call: read q, k, v, gates, beta once, write o
    once, read S0 and write S_final once."""
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    e = 2 if wl.dtype == "bf16" else 4
    per_tok = e * (2 * dk + dv) + e * dv
    if wl.mode in ("scalar", "gdn"):
        per_tok += 4
    if wl.mode in ("gdn", "kda"):
        per_tok += 4
    if wl.mode in ("gla", "kda", "outer"):
        per_tok += 4 * dk
    if wl.mode == "outer":  # value-axis gates
        per_tok += 4 * dv
    W = dv + 1 if wl.mode == "elu1" else dv
    state = 4 * dk * W * (2 if has_s0 else 1)
    return float(B * H * (T * per_tok + state))


L2_BYTES = 129e6
FLUSH_NOTE = "inputs smaller than L2: a 256 MB buffer written between timed steps, outside the timed intervals"


def l2_flusher(working_set_bytes: float, dev):
    """A device buffer twice the L2 size, written between timed steps when a
    step's working set would otherwise stay in L2 from the step before; None
    when the working set is larger than L2."""
    if working_set_bytes > L2_BYTES:
        return None
    return torch.empty(256 << 20, dtype=torch.uint8, device=dev)


def time_steps(step, stream, steps: int, flush):
    """Device time of `steps` calls of step() on `stream` (CUDA events): the
    whole bracket when no flush is needed, else the sum of the per-step
    intervals with the L2 flush written between them. Returns (total_ms,
    per-step ms)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xff)
        ev[2 * i].record(stream)
        step()
        ev[2 * i + 1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    per = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)]
    total = t_start.elapsed_time(t_end) if flush is None else sum(per)
    return total, per


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of x over all ranks (the job is as slow as its slowest
    replica); x itself with a single process."""
    if not dist:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput of `world` replicas that each processed
    units_per_rank in ms milliseconds (the max over ranks)."""
    return world * units_per_rank / (ms / 1e3)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_hash(workload: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(workload, sorted({f for v in KERNEL_SOURCES.values() for f in v})):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source for this workload; else None."""
    if not os.path.exists(PROFILE_FILE):
        return None
    cur = kernel_hash(workload)
    with open(PROFILE_FILE) as f:
        for line in f:
            m = re.match(r"\s*traffic\s+workload=(\S+)\s+kernel_hash=(\S+)\s+bytes_per_launch=(\d+)", line)
            if m and m.group(1) == workload and m.group(2) == cur:
                return int(m.group(3))
    return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle

def time_oracle(wl, inp, target_s: float = 12.0, max_heads: int | None = None):
    """Time the float64 C oracle on this host on a sample of heads over the
    full sequence. Returns (tokens/s scaled to the workload's unit, cores, sample)."""
    import numpy as np
    import oracle

    cores = oracle.c_threads_default()
    BH = wl.B * wl.H
    nh = max(1, min(BH, max_heads or 4 * cores))
    heads = [(i // wl.H, i % wl.H) for i in range(nh)]

    def pick(x):
        if x is None:
            return None
        return torch.stack([x[b, h] for b, h in heads])[None].float().numpy().astype(np.float64)

    q, k, v = pick(inp["q"]), pick(inp["k"]), pick(inp["v"])
    g = inp["g"]
    if g is not None:
        g = (torch.stack([g[h] for _, h in heads]).double().numpy() if wl.mode == "retnet"
             else pick(g))
    beta, S0 = pick(inp["beta"]), pick(inp["S0"])
    t0 = time.perf_counter()
    if is_noncausal(wl):
        from oracle.noncausal import noncausal
        noncausal(q, k, v, wl.mode, S0=S0)
        cores = 1
    else:
        oracle.recurrence_c(q, k, v, wl.mode, g=g, beta=beta, S0=S0, nthreads=cores)
    dt = time.perf_counter() - t0
    # nh head-sequences of T tokens = nh/H of the workload's B*T tokens
    tokens = nh * wl.T / wl.H
    sample = (f"{nh} of {BH} (batch, head) sequences, full T={wl.T}, float64, "
              + ("numpy" if is_noncausal(wl) else f"{cores} threads"))
    return tokens / dt, cores, sample, dt


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gdn",
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.PROLOGUE_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--B", type=int, default=None, help="override batch (profiling of a smaller case)")
    ap.add_argument("--H", type=int, default=None)
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--chunk", type=int, default=None, choices=[0, 64, 128],
                    help="override the workload's chunk length C (0: the library's per-shape choice)")
    ap.add_argument("--variant", default=None, choices=["tc", "nonmat", "mat", "simt"],
                    help="force a kernel variant (default: the library's per-shape choice)")
    args = ap.parse_args()
    if args.variant:
        os.environ["LA_VARIANT"] = args.variant
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload in workloads.PROLOGUE_WORKLOADS:
        return bench_prologue(args, rank, world, local_rank)
    if workloads.WORKLOADS[args.workload].extra.get("backward"):
        return bench_backward(args, rank, world, local_rank)
    if workloads.WORKLOADS[args.workload].extra.get("decode"):
        return bench_decode(args, rank, world, local_rank)
    if workloads.WORKLOADS[args.workload].mode == "gdelta":
        return bench_gdelta(args, rank, world, local_rank)
    wl = workloads.WORKLOADS[args.workload]
    over = {k: getattr(args, k) for k in ("B", "H", "T") if getattr(args, k) is not None}
    if args.chunk is not None:
        over["C"] = args.chunk
    if over:
        wl = wl.with_sizes(**over)

    if args.impl == "reference":
        return run_reference(args, wl, rank, world)

    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build as labuild
    labuild.build()
    la.load_library()

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    inp = workloads.make_inputs(wl)
    d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    W = dv + 1 if wl.mode == "elu1" else dv
    o = torch.empty((B, H, T, dv), dtype=wl.torch_dtype, device=dev)
    S = torch.empty((B, H, dk, W), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    mode_id = la.MODE_IDS[wl.mode] | (la.CONSTANTS["LA_F32"] if wl.dtype == "f32" else 0)
    if is_noncausal(wl):
        mode_id |= la.CONSTANTS["LA_NONCAUSAL"]
    ptr = lambda t: None if t is None else t.data_ptr()

    def step():
        rc = la.la_chunk_fwd(d["q"], d["k"], d["v"], ptr(d["g"]), ptr(d["beta"]), o,
                             ptr(d["S0"]), S, B, H, T, dk, dv, wl.C, mode_id, sh)
        if rc != 0:
            raise RuntimeError(la.la_last_error())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc = la.la_stream_status(sh)
    if rc != 0:
        raise RuntimeError(f"device status after warm-up: {la.la_last_error()}")

    flush = l2_flusher(algorithmic_bytes(wl, d["S0"] is not None), dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms, launch_ms = time_steps(step, stream, args.steps, flush)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    tokens_per_step = B * T
    value = replica_throughput(tokens_per_step * args.steps, world, total_ms)
    flop_call = B * H * T * flops_per_token_head("noncausal" if is_noncausal(wl) else wl.mode, dk, dv)
    tflops = world * flop_call * args.steps / (total_ms / 1e3) / 1e12
    avg_launch_s = statistics.mean(launch_ms) / 1e3
    alg_bytes = algorithmic_bytes(wl, d["S0"] is not None)
    hbm_peak, tc_peak, peak_src = read_peaks()
    ai = flop_call / alg_bytes
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
    if ai < ridge:
        achieved = alg_bytes / avg_launch_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4)}
    else:
        achieved = flop_call / avg_launch_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(achieved / tc_peak, 4)}
    traffic = recorded_traffic(args.workload)
    roof["traffic"] = traffic
    roof["peak_source"] = peak_src
    roof["algorithmic_bytes"] = alg_bytes
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mat = uses_materialised(wl, args.variant, sms)
    roof["kernel"] = kernel_name(wl, args.variant, sms)
    roof["launch_ms_mean"] = round(statistics.mean(launch_ms), 4)

    # ---- end to end through the C ABI with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(la, wl, inp, dev, stream, mode_id, args, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, dt = time_oracle(wl, inp)
        cpu = {"value": round(v_cpu, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample, "seconds": round(dt, 2)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": wl.name, "mode": wl.mode + ("+noncausal" if is_noncausal(wl) else ""), "B": B, "H": H, "T": T, "dk": dk,
                       "dv": dv, "C": wl.C, "global_batch": B * world, "seq_len": T,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (no flush)" if flush is None else FLUSH_NOTE},
            "tflops": round(tflops, 2),
            "roofline": roof,
            "cpu_baseline": cpu,
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": args.steps * (3 if is_noncausal(wl) else
                                          ((3 if parallel_state_pass(wl) else 2) if mat else 1)),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_e2e(la, wl, inp, dev, stream, mode_id, args, world, dist):
    """Same metric through the C ABI with host buffers: every step copies the
    inputs from pinned host memory, runs the forward, and copies o and the
    final state back, all inside the timed region. The steps are pipelined the
    way a streaming caller would run them: the inputs of step i + 1 cross to the
    device (one copy stream) while step i computes (the main stream) and the
    outputs of step i - 1 cross back (a second copy stream), on two device
    buffer sets; every step's copies still lie inside the timed region."""
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    W = dv + 1 if wl.mode == "elu1" else dv
    names = [n for n in ("q", "k", "v", "g", "beta", "S0") if inp[n] is not None]
    host = {n: inp[n].pin_memory() for n in names}
    devb = [{n: torch.empty_like(inp[n], device=dev) for n in names} for _ in range(2)]
    o_h = [torch.empty((B, H, T, dv), dtype=wl.torch_dtype).pin_memory() for _ in range(2)]
    S_h = [torch.empty((B, H, dk, W), dtype=torch.float32).pin_memory() for _ in range(2)]
    o_d = [torch.empty((B, H, T, dv), dtype=wl.torch_dtype, device=dev) for _ in range(2)]
    S_d = [torch.empty((B, H, dk, W), dtype=torch.float32, device=dev) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_h[0].numel() * o_h[0].element_size() + S_h[0].numel() * S_h[0].element_size()
    sh = stream.cuda_stream
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    done, out_free = [ev(), ev()], [ev(), ev()]
    for e in in_free + out_free:
        e.record(stream)

    def copy_in(i):
        b = i % 2
        s_in.wait_event(in_free[b])
        with torch.cuda.stream(s_in):
            for n in names:
                devb[b][n].copy_(host[n], non_blocking=True)
        in_ready[b].record(s_in)

    def compute_and_copy_out(i):
        b = i % 2
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        d = devb[b]
        rc = la.la_chunk_fwd(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), o_d[b], d.get("S0"), S_d[b],
                             B, H, T, dk, dv, wl.C, mode_id, sh)
        if rc != 0:
            raise RuntimeError(la.la_last_error())
        done[b].record(stream)
        in_free[b].record(stream)
        s_out.wait_event(done[b])
        with torch.cuda.stream(s_out):
            o_h[b].copy_(o_d[b], non_blocking=True)
            S_h[b].copy_(S_d[b], non_blocking=True)
        out_free[b].record(s_out)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute_and_copy_out(i)
        stream.wait_stream(s_out)

    steps = max(3, min(args.steps, 10))
    run(3)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_stream(stream)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    ms = max_over_ranks(ms, dist, dev)
    return {"value": round(world * B * T * steps / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4), "pipelined": "copy-in of step i+1 and copy-out of step i-1 overlap step i"}


def run_reference(args, wl, rank, world):
    """Reference arm: the float64 CPU oracle, timed as it stands on this
    host's cores, each step a bounded sample of the same workload."""
    if rank != 0:
        return
    inp = workloads.make_inputs(wl)
    vals = []
    cores = sample = None
    for i in range(args.warmup + args.steps):
        v, cores, sample, _ = time_oracle(wl, inp, max_heads=None)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    B, T = wl.B, wl.T
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(B * T / value * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": wl.name, "mode": wl.mode + ("+noncausal" if is_noncausal(wl) else ""), "B": B, "H": wl.H, "T": T, "dk": wl.dk,
                   "dv": wl.dv, "C": wl.C, "global_batch": B, "seq_len": T,
                   "parallelism": "single"},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- prologue

PRO_METRIC = "tokens/sec of the prologue (short conv + L2 norm + gate/beta activations) at 1 GB300; % of roofline"


def prologue_bytes(wl) -> float:
    """Minimum HBM traffic of one la_prologue call: read the three projections,
    the gate and beta pre-activations and the weights once, write q, k, v, g
    and beta once."""
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    per_tok = 2 * 2 * (2 * dk + dv)
    if wl.gate_kind != "none":
        per_tok += 2 * 4 * wl.gate_width
    if wl.beta:
        per_tok += 2 * 4
    return float(B * H * T * per_tok + H * 4 * wl.K * (2 * dk + dv))


def _pro_args(la, d, wl, hist_out=None):
    flags = (la.CONSTANTS["LA_PRO_L2NORM_Q"] if wl.l2q else 0) | (la.CONSTANTS["LA_PRO_L2NORM_K"] if wl.l2k else 0)
    return (d["xq"], d["xk"], d["xv"], d["wq"], d["wk"], d["wv"], wl.K, None, hist_out, d.get("a_gate"),
            la.GATE_KINDS[wl.gate_kind], wl.gate_width, wl.tau, d.get("a_beta"), d["q"], d["k"], d["v"],
            d.get("g"), d.get("beta"), wl.B, wl.H, wl.T, wl.dk, wl.dv, flags)


def time_prologue_oracle(wl, inp, target_s: float = 10.0):
    """The float64 prologue oracle on this host, on a sample of heads over the
    full sequence (numpy; it uses the threads numpy's own routines use)."""
    import numpy as np
    import oracle.prologue as P
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()
    BH = wl.B * wl.H
    done, t0, tokens = 0, time.perf_counter(), 0
    while done < BH and (time.perf_counter() - t0) < target_s:
        b, h = done // wl.H, done % wl.H
        sl = lambda t: None if t is None else t[b:b + 1, h:h + 1]
        P.prologue(f64(sl(inp["xq"])), f64(sl(inp["xk"])), f64(sl(inp["xv"])),
                   f64(inp["wq"][h:h + 1]), f64(inp["wk"][h:h + 1]), f64(inp["wv"][h:h + 1]),
                   l2q=wl.l2q, l2k=wl.l2k, a_gate=f64(sl(inp["a_gate"])), gate_kind=wl.gate_kind,
                   tau=wl.tau, a_beta=f64(sl(inp["a_beta"])), K=wl.K)
        done += 1
        tokens += wl.T
    dt = time.perf_counter() - t0
    # done head-sequences of T tokens = done/H of the workload's B*T tokens
    sample = f"{done} of {BH} (batch, head) sequences, full T={wl.T}, float64 numpy"
    return (tokens / wl.H) / dt, 1, sample, dt


def bench_prologue(args, rank, world, local_rank):
    wl = workloads.PROLOGUE_WORKLOADS[args.workload]
    over = {k: getattr(args, k) for k in ("B", "H", "T") if getattr(args, k) is not None}
    if over:
        wl = wl.with_sizes(**over)
    B, H, T = wl.B, wl.H, wl.T
    if args.impl == "reference":
        if rank != 0:
            return
        inp = workloads.make_prologue_inputs(wl)
        vals = []
        for i in range(args.warmup + args.steps):
            v, cores, sample, _ = time_prologue_oracle(wl, inp, target_s=3.0)
            if i >= args.warmup:
                vals.append(v)
        value = statistics.mean(vals)
        print(json.dumps({
            "impl": "reference", "metric": PRO_METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(B * T / value * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": wl.name, "B": B, "H": H, "T": T, "dk": wl.dk, "dv": wl.dv, "K": wl.K,
                       "global_batch": B, "seq_len": T, "parallelism": "single"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return

    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build as labuild
    labuild.build()
    la.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = workloads.make_prologue_inputs(wl)
    ins = [n for n in ("xq", "xk", "xv", "wq", "wk", "wv", "a_gate", "a_beta") if inp[n] is not None]
    d = {n: inp[n].to(dev) for n in ins}
    d["q"], d["k"], d["v"] = (torch.empty_like(d["xq"]), torch.empty_like(d["xk"]), torch.empty_like(d["xv"]))
    if "a_gate" in d:
        d["g"] = torch.empty_like(d["a_gate"])
    if "a_beta" in d:
        d["beta"] = torch.empty_like(d["a_beta"])
    outs = [n for n in ("q", "k", "v", "g", "beta") if n in d]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(dd):
        rc = la.la_prologue(*_pro_args(la, dd, wl), sh)
        if rc != 0:
            raise RuntimeError(la.la_last_error())

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()
    flush = l2_flusher(prologue_bytes(wl), dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms, launch_ms = time_steps(lambda: step(d), stream, args.steps, flush)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, dist, dev)
    value = replica_throughput(B * T * args.steps, world, total_ms)
    alg = prologue_bytes(wl)
    hbm_peak, _, peak_src = read_peaks()
    achieved = alg / (statistics.mean(launch_ms) / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": recorded_traffic(wl.name),
            "peak_source": peak_src, "algorithmic_bytes": alg, "kernel": "prologue_kernel",
            "launch_ms_mean": round(statistics.mean(launch_ms), 4)}

    e2e = None
    if not args.no_e2e:
        host = {n: inp[n].pin_memory() for n in ins}
        hout = {n: torch.empty_like(d[n], device="cpu").pin_memory() for n in outs}
        dd = dict(d)
        h2d = sum(host[n].numel() * host[n].element_size() for n in ins)
        d2h = sum(hout[n].numel() * hout[n].element_size() for n in outs)

        def e2e_step():
            with torch.cuda.stream(stream):
                for n in ins:
                    dd[n].copy_(host[n], non_blocking=True)
                step(dd)
                for n in outs:
                    hout[n].copy_(dd[n], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        steps = max(3, min(args.steps, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        e2e = {"value": round(world * B * T * steps / (ms / 1e3), 1), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
               "ms_per_step": round(ms / steps, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, dt = time_prologue_oracle(wl, inp)
        cpu = {"value": round(v_cpu, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample, "seconds": round(dt, 2)}
    if rank == 0:
        print(json.dumps({
            "metric": PRO_METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": wl.name, "B": B, "H": H, "T": T, "dk": wl.dk, "dv": wl.dv, "K": wl.K,
                       "gate": wl.gate_kind, "gate_width": wl.gate_width, "l2norm_qk": [wl.l2q, wl.l2k],
                       "global_batch": B * world, "seq_len": T,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (no flush)" if flush is None else FLUSH_NOTE},
            "roofline": roof, "cpu_baseline": cpu, "clocks": clk, "e2e": e2e,
            "gpu_launches": args.steps,
        }), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- backward

BWD_METRIC = "tokens/sec of the chunk backward (dq, dk, dv, dS0; dg, dbeta where the mode has them) at 1 GB300; % of roofline"


def backward_inputs(wl):
    """The forward workload's inputs plus dO ~ N(0,1)/sqrt(dv) and dS_final ~ N(0, 0.01)."""
    inp = workloads.make_inputs(wl)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed + 1000)
    inp["dO"] = (torch.randn(wl.B, wl.H, wl.T, wl.dv, generator=gen) / math.sqrt(wl.dv)).to(wl.torch_dtype)
    inp["dS"] = torch.randn(wl.B, wl.H, wl.dk, wl.dv, generator=gen) * 0.1
    return inp


def backward_bytes(wl) -> float:
    """Minimum HBM traffic of one backward call: read q, k, v, dO, write dq, dk, dv
    once, read dS_final and write dS0."""
    e = 2 if wl.dtype == "bf16" else 4
    per_tok = e * (2 * wl.dk + 2 * wl.dv) + e * (2 * wl.dk + wl.dv)
    if wl.mode == "scalar":  # read g, write dg
        per_tok += 8
    elif wl.mode == "gla":
        per_tok += 8 * wl.dk
    elif wl.mode == "gdn":  # read g and beta, write dg and dbeta; also read S0
        per_tok += 16
        return float(wl.B * wl.H * (wl.T * per_tok + 3 * 4 * wl.dk * wl.dv))
    elif wl.mode == "kda":  # read the per-channel g and beta, write dg and dbeta; also read S0
        per_tok += 8 * wl.dk + 8
        return float(wl.B * wl.H * (wl.T * per_tok + 3 * 4 * wl.dk * wl.dv))
    return float(wl.B * wl.H * (wl.T * per_tok + 2 * 4 * wl.dk * wl.dv))


def time_backward_oracle(wl, inp, target_s: float = 10.0):
    from oracle.backward import backward, backward_gla, backward_scalar
    from oracle.backward_delta import backward_delta
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()
    BH = wl.B * wl.H
    done, t0 = 0, time.perf_counter()
    while done < BH and (time.perf_counter() - t0) < target_s:
        b, h = done // wl.H, done % wl.H
        sl = lambda t: None if t is None else f64(t[b:b + 1, h:h + 1])
        if wl.mode in ("gdn", "kda"):  # one full-length head per iteration (the token recurrence, reversed)
            backward_delta(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dO"]), wl.mode, g=sl(inp["g"]),
                           beta=sl(inp["beta"]), S0=sl(inp["S0"]), dS=sl(inp["dS"]))
            done += 1
            continue
        if wl.mode == "gla":  # quadratic in T: a 512-token prefix of one head
            pre = lambda t: t[..., :512, :]
            backward_gla(pre(sl(inp["q"])), pre(sl(inp["k"])), pre(sl(inp["v"])), pre(sl(inp["dO"])),
                         pre(sl(inp["g"])), dS=sl(inp["dS"]))
            dt = time.perf_counter() - t0
            return 512 / wl.H / dt, 1, ("the first 512 tokens of 1 (batch, head) sequence, float64 numpy "
                                        "(explicit pair sums: quadratic in T, so faster per token than at T=4096)"), dt
        if wl.mode == "scalar":
            backward_scalar(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dO"]), sl(inp["g"]), dS=sl(inp["dS"]))
        else:
            backward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["dO"]), wl.mode,
                     g=None if inp["g"] is None else f64(inp["g"])[h:h + 1], dS=sl(inp["dS"]))
        done += 1
    dt = time.perf_counter() - t0
    return (done * wl.T / wl.H) / dt, 1, f"{done} of {BH} (batch, head) sequences, full T={wl.T}, float64 numpy", dt


def bench_backward(args, rank, world, local_rank):
    wl = workloads.WORKLOADS[args.workload]
    over = {k: getattr(args, k) for k in ("B", "H", "T") if getattr(args, k) is not None}
    if over:
        wl = wl.with_sizes(**over)
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    cfg = {"workload": wl.name, "mode": wl.mode + "+backward", "B": B, "H": H, "T": T, "dk": dk, "dv": dv, "C": wl.C,
           "global_batch": B * world, "seq_len": T, "parallelism": "replicas" if world > 1 else "single"}
    if args.impl == "reference":
        if rank != 0:
            return
        inp = backward_inputs(wl)
        vals = []
        for i in range(args.warmup + args.steps):
            v, cores, sample, _ = time_backward_oracle(wl, inp, target_s=3.0)
            if i >= args.warmup:
                vals.append(v)
        value = statistics.mean(vals)
        print(json.dumps({
            "impl": "reference", "metric": BWD_METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(B * T / value * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)", "config": cfg,
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build as labuild
    labuild.build()
    la.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = backward_inputs(wl)
    delta = wl.mode in ("gdn", "kda")
    names = [n for n in ("q", "k", "v", "g", "dO", "dS") + (("beta", "S0") if delta else ()) if inp[n] is not None]
    d = {n: inp[n].to(dev) for n in names}
    outs = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"]),
            "dS0": torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)}
    if wl.mode in ("scalar", "gdn"):
        outs["dg"] = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    if delta:
        outs["dbeta"] = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    if wl.mode in ("gla", "kda"):
        outs["dg"] = torch.empty(B, H, T, dk, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    mode_id = la.MODE_IDS[wl.mode] | (la.CONSTANTS["LA_F32"] if wl.dtype == "f32" else 0)

    def step(dd, oo):
        if delta:
            rc = la.la_chunk_bwd_delta(dd["q"], dd["k"], dd["v"], dd.get("g"), dd.get("beta"), dd["dO"], dd["dS"],
                                       dd.get("S0"), oo["dq"], oo["dk"], oo["dv"], oo["dbeta"], oo["dg"], oo["dS0"],
                                       B, H, T, dk, dv, wl.C, mode_id, sh)
        else:
            rc = la.la_chunk_bwd(dd["q"], dd["k"], dd["v"], dd.get("g"), dd["dO"], dd["dS"], None, oo["dq"],
                                 oo["dk"], oo["dv"], oo["dS0"], oo.get("dg"), B, H, T, dk, dv, wl.C, mode_id, sh)
        if rc != 0:
            raise RuntimeError(la.la_last_error())

    for _ in range(args.warmup):
        step(d, outs)
    torch.cuda.synchronize()
    if la.la_stream_status(sh) != 0:
        raise RuntimeError(la.la_last_error())
    flush = l2_flusher(backward_bytes(wl), dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms, launch_ms = time_steps(lambda: step(d, outs), stream, args.steps, flush)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, dist, dev)
    value = replica_throughput(B * T * args.steps, world, total_ms)
    flop = 3 * B * H * T * flops_per_token_head(wl.mode, dk, dv)
    alg = backward_bytes(wl)
    hbm_peak, _, peak_src = read_peaks()
    achieved = alg / (statistics.mean(launch_ms) / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": recorded_traffic(wl.name), "peak_source": peak_src,
            "algorithmic_bytes": alg, "kernel": "bd_pre_kernel + bd_fwd_kernel + bd_bwd_kernel + bd_grad_kernel"
            if wl.mode == "gdn" else "bk_pre_kernel + bd_fwd_kernel + bd_bwd_kernel + bk_grad_kernel (per-channel gates)"
            if wl.mode == "kda" else "3 x chunk_ws_kernel (dq causal; dk and dv reversed runs)"
            + (" + forward for S_final + dg_tile_kernel + dg_carry_kernel" if wl.mode == "scalar" else
               " + forward for S_final + dgc_tile_kernel + dgc_carry_kernel (dq, dk: outer-product-gate passes)"
               if wl.mode == "gla" else ""),
            "launch_ms_mean": round(statistics.mean(launch_ms), 4)}
    e2e = None
    if not args.no_e2e:
        host = {n: inp[n].pin_memory() for n in names}
        hout = {n: torch.empty_like(outs[n], device="cpu").pin_memory() for n in outs}
        dd, oo = dict(d), dict(outs)
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = sum(hout[n].numel() * hout[n].element_size() for n in outs)

        def e2e_step():
            with torch.cuda.stream(stream):
                for n in names:
                    dd[n].copy_(host[n], non_blocking=True)
                step(dd, oo)
                for n in outs:
                    hout[n].copy_(oo[n], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        steps = max(3, min(args.steps, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        e2e = {"value": round(world * B * T * steps / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": round(ms / steps, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, dt = time_backward_oracle(wl, inp)
        cpu = {"value": round(v_cpu, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2)}
    if rank == 0:
        cfg["l2"] = "inputs larger than L2 (no flush)" if flush is None else FLUSH_NOTE
        print(json.dumps({
            "metric": BWD_METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded; shapes and distributions of the workload)", "config": cfg,
            "tflops": round(world * flop * args.steps / (total_ms / 1e3) / 1e12, 2), "roofline": roof,
            "cpu_baseline": cpu, "clocks": clk, "e2e": e2e,
            # state prep, 3 passes, dS0 scaling (+ the forward for S_final and the two dg launches)
            "gpu_launches": args.steps * {"scalar": 8, "gla": 8, "gdn": 4, "kda": 4}.get(wl.mode, 5),
        }), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------- decode

DEC_METRIC = "tokens/sec of one decode step (la_recurrent_step, states resident) at 1 GB300; % of roofline"


def decode_bytes(wl) -> float:
    """Minimum HBM traffic of one step: read and write every head's state once,
    read q, k, v and the gates, write o."""
    e = 2 if wl.dtype == "bf16" else 4
    W = wl.dv + 1 if wl.mode == "elu1" else wl.dv
    per_head = 2 * 4 * wl.dk * W + e * (2 * wl.dk + 2 * wl.dv) + 8
    return float(wl.B * wl.H * per_head)


GD_METRIC = "tokens/sec of the generalised-delta-rule chunk forward (la_chunk_fwd_gdelta) at 1 GB300; % of roofline"


def gdelta_flops_per_token_head(dk: int, dv: int, C: int = 64) -> float:
    """Chunk form at C = 64: the four C x C products Q K^T, A B^T, A K^T, Q B^T
    (half each under the masks, counted whole), A S and Q S (2 dk dv each),
    L_ak V, T R, M(Q K^T) V and M(Q B^T) U (2 C dv each, counted whole), the
    triangular solve (C^2 / 3) and the state update K^T V - B^T U (4 dk dv)."""
    return 8 * C * dk + 8 * C * dv + C * C / 3.0 + 8 * dk * dv


def time_gdelta_oracle(wl, inp, target_s: float = 10.0):
    from oracle.gdelta import recurrence_gdelta
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()
    BH = wl.B * wl.H
    done, t0 = 0, time.perf_counter()
    while done < BH and (time.perf_counter() - t0) < target_s:
        b, h = done // wl.H, done % wl.H
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        recurrence_gdelta(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["a"]), sl(inp["b"]),
                          S0=None if inp["S0"] is None else sl(inp["S0"]))
        done += 1
    dt = time.perf_counter() - t0
    return (done * wl.T / wl.H) / dt, 1, f"{done} of {BH} (batch, head) sequences, full T={wl.T}, float64 numpy", dt


def bench_gdelta(args, rank, world, local_rank):
    wl = workloads.WORKLOADS[args.workload]
    over = {k: getattr(args, k) for k in ("B", "H", "T") if getattr(args, k) is not None}
    if over:
        wl = wl.with_sizes(**over)
    B, H, T, dk, dv = wl.B, wl.H, wl.T, wl.dk, wl.dv
    cfg = {"workload": wl.name, "mode": "gdelta", "B": B, "H": H, "T": T, "dk": dk, "dv": dv, "C": wl.C,
           "global_batch": B * world, "seq_len": T, "parallelism": "replicas" if world > 1 else "single"}
    inp = workloads.make_inputs(wl)
    if args.impl == "reference":
        if rank != 0:
            return
        vals = []
        for i in range(args.warmup + args.steps):
            v, cores, sample, _ = time_gdelta_oracle(wl, inp, target_s=3.0)
            if i >= args.warmup:
                vals.append(v)
        value = statistics.mean(vals)
        print(json.dumps({
            "impl": "reference", "metric": GD_METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(B * T / value * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)", "config": cfg,
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build as labuild
    labuild.build()
    la.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    names = [n for n in ("q", "k", "v", "a", "b", "S0") if inp[n] is not None]
    d = {n: inp[n].to(dev) for n in names}
    outs = {"o": torch.empty((B, H, T, dv), dtype=wl.torch_dtype, device=dev),
            "S": torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)}
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    mode = la.CONSTANTS["LA_F32"] if wl.dtype == "f32" else 0

    def step(dd, oo):
        rc = la.la_chunk_fwd_gdelta(dd["q"], dd["k"], dd["v"], dd["a"], dd["b"], oo["o"], dd.get("S0"), oo["S"],
                                    B, H, T, dk, dv, wl.C, mode, sh)
        if rc != 0:
            raise RuntimeError(la.la_last_error())

    for _ in range(args.warmup):
        step(d, outs)
    torch.cuda.synchronize()
    flush = l2_flusher(float(B * H * (T * (2 if wl.dtype == "bf16" else 4) * (4 * dk + 2 * dv) + 4 * dk * dv * (2 if inp["S0"] is not None else 1))), dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms, launch_ms = time_steps(lambda: step(d, outs), stream, args.steps, flush)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, dist, dev)
    value = replica_throughput(B * T * args.steps, world, total_ms)
    flop = B * H * T * gdelta_flops_per_token_head(dk, dv)
    e = 2 if wl.dtype == "bf16" else 4
    alg = float(B * H * (T * e * (4 * dk + 2 * dv) + 4 * dk * dv * (2 if inp["S0"] is not None else 1)))
    hbm_peak, tc_peak, peak_src = read_peaks()
    t_launch = statistics.mean(launch_ms) / 1e3
    # the arithmetic intensity (~100 FLOP/byte at d = 64) sits below the bf16 ridge: an HBM roofline
    roof = {"bound": "hbm", "achieved": round(alg / t_launch / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(alg / t_launch / 1e9 / hbm_peak, 4), "traffic": recorded_traffic(wl.name),
            "peak_source": peak_src, "algorithmic_bytes": alg, "kernel": "gdw_pre_kernel + gdw_chain_kernel (bf16 warp MMAs)"
            if wl.dtype == "bf16" else "chunk_gdelta_kernel (CUDA cores, fp32)",
            "launch_ms_mean": round(statistics.mean(launch_ms), 4)}
    e2e = None
    if not args.no_e2e:
        host = {n: inp[n].pin_memory() for n in names}
        hout = {n: torch.empty_like(outs[n], device="cpu").pin_memory() for n in outs}
        dd, oo = dict(d), dict(outs)
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = sum(hout[n].numel() * hout[n].element_size() for n in outs)

        def e2e_step():
            with torch.cuda.stream(stream):
                for n in names:
                    dd[n].copy_(host[n], non_blocking=True)
                step(dd, oo)
                for n in outs:
                    hout[n].copy_(oo[n], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        steps = max(3, min(args.steps, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        e2e = {"value": round(world * B * T * steps / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": round(ms / steps, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, dt = time_gdelta_oracle(wl, inp)
        cpu = {"value": round(v_cpu, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2)}
    if rank == 0:
        cfg["l2"] = "inputs larger than L2 (no flush)" if flush is None else FLUSH_NOTE
        print(json.dumps({
            "metric": GD_METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded; shapes and distributions of the workload)", "config": cfg,
            "tflops": round(world * flop * args.steps / (total_ms / 1e3) / 1e12, 2), "roofline": roof,
            "cpu_baseline": cpu, "clocks": clk, "e2e": e2e, "gpu_launches": args.steps,
        }), flush=True)
    if dist:
        dist.destroy_process_group()


def bench_decode(args, rank, world, local_rank):
    wl = workloads.WORKLOADS[args.workload]
    over = {k: getattr(args, k) for k in ("B", "H") if getattr(args, k) is not None}
    if over:
        wl = wl.with_sizes(**over)
    B, H, dk, dv = wl.B, wl.H, wl.dk, wl.dv
    inp = workloads.make_inputs(wl)
    sq = lambda t: None if t is None else t[:, :, 0].contiguous() if t.dim() >= 3 else t
    step_in = {"q": sq(inp["q"]), "k": sq(inp["k"]), "v": sq(inp["v"]),
               "g": None if inp["g"] is None else inp["g"][:, :, 0].contiguous(),
               "beta": None if inp["beta"] is None else inp["beta"][:, :, 0].contiguous()}
    cfg = {"workload": wl.name, "mode": wl.mode + "+decode", "B": B, "H": H, "dk": dk, "dv": dv,
           "global_batch": B * world, "seq_len": 1, "parallelism": "replicas" if world > 1 else "single"}

    def time_cpu(target_s):
        import numpy as np
        from oracle import recurrence
        f64 = lambda t: None if t is None else t.to(torch.float64).numpy()
        BH, done, t0 = B * H, 0, time.perf_counter()
        while done < BH and time.perf_counter() - t0 < target_s:
            b, h = done // H, done % H
            sl = lambda t: None if t is None else f64(t[b:b + 1, h:h + 1])
            recurrence(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), wl.mode, g=sl(inp["g"]), beta=sl(inp["beta"]),
                       S0=sl(inp["S0"]))
            done += 1
        dt = time.perf_counter() - t0
        return (done / H) / dt, 1, f"{done} of {BH} (batch, head) one-token steps, float64 numpy", dt

    if args.impl == "reference":
        if rank != 0:
            return
        vals = []
        for i in range(args.warmup + args.steps):
            v, cores, sample, _ = time_cpu(1.0)
            if i >= args.warmup:
                vals.append(v)
        value = statistics.mean(vals)
        print(json.dumps({
            "impl": "reference", "metric": DEC_METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(B / value * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)", "config": cfg,
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return
    import gated_delta_rule_linear_gb300 as la
    from gated_delta_rule_linear_gb300 import build as labuild
    labuild.build()
    la.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    names = [n for n in ("q", "k", "v", "g", "beta") if step_in[n] is not None]
    d = {n: step_in[n].to(dev) for n in names}
    S = inp["S0"].to(dev).contiguous()
    o = torch.empty(B, H, dv, dtype=wl.torch_dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    mode_id = la.MODE_IDS[wl.mode] | (la.CONSTANTS["LA_F32"] if wl.dtype == "f32" else 0)

    def step(dd, oo):
        rc = la.la_recurrent_step(dd["q"], dd["k"], dd["v"], dd.get("g"), dd.get("beta"), oo, S, B, H, dk, dv,
                                  mode_id, sh)
        if rc != 0:
            raise RuntimeError(la.la_last_error())

    for _ in range(args.warmup):
        step(d, o)
    torch.cuda.synchronize()
    flush = l2_flusher(decode_bytes(wl), dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    steps = max(args.steps, 50)  # a step is ~20 us: enough of them to time
    total_ms, launch_ms = time_steps(lambda: step(d, o), stream, steps, flush)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(total_ms, dist, dev)
    value = replica_throughput(B * steps, world, total_ms)
    alg = decode_bytes(wl)
    hbm_peak, _, peak_src = read_peaks()
    achieved = alg / (statistics.mean(launch_ms) / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "traffic": recorded_traffic(wl.name), "peak_source": peak_src,
            "algorithmic_bytes": alg, "kernel": "step_kernel", "launch_ms_mean": round(statistics.mean(launch_ms), 4)}
    e2e = None
    if not args.no_e2e:
        host = {n: step_in[n].pin_memory() for n in names}
        o_h = torch.empty(B, H, dv, dtype=wl.torch_dtype).pin_memory()
        dd = dict(d)
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = o_h.numel() * o_h.element_size()

        def e2e_step():
            with torch.cuda.stream(stream):
                for n in names:
                    dd[n].copy_(host[n], non_blocking=True)
                step(dd, o)
                o_h.copy_(o, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        e2e = {"value": round(world * B * steps / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": round(ms / steps, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, dt = time_cpu(10.0)
        cpu = {"value": round(v_cpu, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2)}
    if rank == 0:
        cfg["l2"] = ("state larger than L2 (no flush)" if flush is None else
                     "state smaller than L2: a 256 MB buffer written between timed steps, outside the timed intervals")
        print(json.dumps({
            "metric": DEC_METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded; shapes and distributions of the workload)", "config": cfg,
            "roofline": roof, "cpu_baseline": cpu, "clocks": clk, "e2e": e2e, "gpu_launches": steps,
        }), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
