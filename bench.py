#!/usr/bin/env python
"""Benchmark: LSTM / GRU forward + backward-through-time on GB300.

One step = rnn_forward (training) + rnn_backward_data + rnn_backward_weights
over one batch of seeded synthetic sequences, inputs resident in HBM.  The
default workload is the largest configuration of the problem statement that
fits one GPU: the 2-layer bidirectional LSTM, bf16 storage / fp32
accumulation, seq 512, batch 128, input 1024 (layer 2: 2048), hidden 1024 per
direction.  The other workloads run with --workload NAME.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     (the fp64 oracle on host cores)

Without --steps the number of timed steps is chosen after the warm-up so that
the timed region lasts at least 2.5 s (at least 10 steps).

Multi-GPU: one process per GPU under torchrun; the sequences of a step are
independent, so each rank runs its own replica on its own batch (weak
scaling, no data-path collective); timing takes the max over ranks.  A plain
``python bench.py --gpus N`` (no WORLD_SIZE in the environment) starts its N
ranks itself through torch.distributed.run on 127.0.0.1.

Prints one JSON line (rank 0).  ``value`` is timestep*batch per second over
all ranks; ``roofline`` covers the kernel class with the largest share of the
step, timed live with CUDA events on its launching stream.  ``e2e`` is the
same step through the C ABI with the inputs uploaded from pinned host memory
and the result (dw; y for forward-only workloads) read back inside the timed
region; dy's upload runs on a copy stream during the forward.
``us_per_timestep`` is the step time over the sequence length (the per-step
latency of the forward-only workloads).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "lstm2bi_bf16_T512_B128_H1024"
MIN_TIMED_S = 2.5
L2_POLICY = "flushed (256 MiB write) before every timed GPU step"
L2_BYTES = 129 * 1024 * 1024
METRIC = "LSTM/GRU fwd+bwd timestep*batch/s"
UNIT = "timestep*batch/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--probe-ranks", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--seq-len", type=int, default=None,
                    help="run the workload on a shorter sequence (profiling captures of a smaller case); "
                         "the workload name then carries the length")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# fp64 oracle on the host cores (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
def _oracle_sample_cols(wl, target_s: float) -> int:
    """Batch columns per oracle sample so that one sample takes ~target_s."""
    # fp64 numpy on the host: rough rate for sizing only
    flops_per_col = wl.flops() / wl.batch
    est_rate = 5e9
    cols = max(1, min(wl.batch, int(target_s * est_rate / max(flops_per_col, 1.0))))
    return cols


def oracle_worker(spec: str) -> None:
    """Internal mode, run in a fresh process: time the oracle on a bounded
    sample, at least ``reps`` times and until ``budget`` seconds have passed;
    print {"times": [seconds per repeat], "units_per_rep": ...}."""
    import numpy as np
    import synth
    from oracle import rnn_oracle
    name, cols, budget, reps = spec.split(":")
    base, _, tlen = name.partition("@T")
    wl = synth.WORKLOADS[base]
    if tlen:
        import dataclasses
        wl = dataclasses.replace(wl, name=name, seq_len=int(tlen))
    cols, budget, reps = int(cols), float(budget), int(reps)
    inp = synth.make_inputs(wl, batch_subset=list(range(cols)))
    times = []
    while len(times) < reps or sum(times) < budget:
        t0 = time.perf_counter()
        rnn_oracle.run_inputs(inp, with_backward=not wl.forward_only)
        times.append(time.perf_counter() - t0)
    units = wl.seq_len * cols if inp.lengths is None else int(np.sum(inp.lengths))
    print(json.dumps({"times": times, "units_per_rep": units}))


def run_oracle_subprocess(wl, budget_s: float, cols: int, reps: int = 1, threads: int = 0):
    """Time the oracle in a fresh process on ``threads`` host threads (0: all cores)."""
    cores = threads or os.cpu_count() or 1
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample",
                        f"{wl.name}:{cols}:{budget_s}:{reps}"], capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed: {r.stderr[-2000:]}")
    out = json.loads(r.stdout.strip().splitlines()[-1])
    return out, cores


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu_index), "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.path) as f:
            out = parse_clock_lines(f)
        os.unlink(self.path)
        return out


def parse_clock_lines(lines):
    """Summarise nvidia-smi samples of ClockSampler.QUERY (csv, no header, no
    units): median SM clock, the highest max clock, and every throttle reason
    seen active in any sample."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            smax.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower().startswith("active"):
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: one per GPU, no data-path collective)
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's time: the job is done when every replica is."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the max-over-ranks time."""
    return units_per_rank * world / (ms / 1e3)


# ---------------------------------------------------------------------------
# algorithmic flop counts per kernel class (per whole step)
# ---------------------------------------------------------------------------
def class_flops(wl):
    G, H, B, T, D = wl.gates, wl.hidden_size, wl.batch, wl.seq_len, wl.dirs
    rec = sum(D * 2.0 * G * H * H * B * T for _ in range(wl.num_layers))
    proj = sum(D * 2.0 * G * H * wl.layer_input(l) * B * T for l in range(wl.num_layers))
    return {"persist_fwd": rec, "persist_bwd": rec, "gemm_proj": proj, "gemm_dx": proj,
            "gemm_dw": proj + rec, "layout_seq": 0.0, "layout_pack": 0.0, "recompute_cells": 0.0}


LAYOUT_CLASSES = ("layout_seq", "layout_pack", "recompute_cells")


def layout_report(names, cls_ms, cls_n, cls_bytes, steps: int, hbm_gbs: float):
    """Per layout class: time, launches and algorithmic bytes per step, and
    the achieved bandwidth against the measured HBM copy rate."""
    out = {}
    for i, n in enumerate(names):
        if n not in LAYOUT_CLASSES or cls_n[i] == 0:
            continue
        gbs = cls_bytes[i] / (cls_ms[i] / 1e3) / 1e9 if cls_ms[i] > 0 else None
        out[n] = {"ms_per_step": cls_ms[i] / steps, "launches_per_step": cls_n[i] / steps,
                  "bytes_per_step": cls_bytes[i] / steps, "achieved_gbs": gbs,
                  "frac_of_hbm": gbs / hbm_gbs if gbs is not None else None}
    return out


PROFILE_FOR_CLASS = {
    "persist_bwd": "profiles/persist_bwd_tc_{workload}.md",
    "persist_fwd": "profiles/persist_fwd_tc_{workload}.md",
}
KERNEL_SOURCES = ["bwd_persistent_cta_gb300/csrc/persist_tc_kernels.cuh", "bwd_persistent_cta_gb300/csrc/persist_tc.cu",
                  "bwd_persistent_cta_gb300/csrc/common.cuh"]


def code_only(text: str) -> str:
    """C++ source without its comments and whitespace: what a profile's
    counters depend on."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def kernel_sources_sha() -> str:
    """Hash of the code (comments and whitespace removed) of the sources that
    make the profiled kernels."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(open(os.path.join(ROOT, f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(cls: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel code has changed since
    the counters were taken (a comment edit does not count)."""
    path = PROFILE_FOR_CLASS.get(cls)
    if not path:
        return None
    path = os.path.join(ROOT, path.format(workload=workload))
    if not os.path.exists(path):
        return None
    sha = kernel_sources_sha()
    fields = {}
    for line in open(path):
        if ":" in line and line.split(":", 1)[0].strip() in ("traffic-bytes-per-launch", "kernel-source-sha256"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel-source-sha256") != sha:
        return None
    try:
        return int(fields["traffic-bytes-per-launch"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d.get("bf16_tflops"), "hbm_gbs": d.get("hbm_gbs"), "sm_max_mhz": d.get("sm_max_mhz"),
                "src": "measured"}
    return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "src": "fallback"}


def fp32_fma_tflops(sms: int, sm_mhz: float) -> float:
    """FP32 peak of the SIMT pipes: 128 FP32 lanes per SM, one FMA (2 flops)
    per lane per clock."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def workload_config(wl, lengths, world: int) -> dict:
    """The ``config`` keys that name the workload; both arms report them."""
    cfg = {"workload": wl.name, "mode": wl.mode, "reset_after": wl.reset_after, "layers": wl.num_layers,
           "bidirectional": wl.bidirectional, "seq_len": wl.seq_len, "batch_per_gpu": wl.batch,
           "input": wl.input_size, "hidden": wl.hidden_size, "seed": wl.seed, "parallelism": f"replicas{world}",
           "recompute_cell_states": wl.recompute, "l2": L2_POLICY}
    if lengths is not None:
        cfg["seq_lengths"] = {"min": int(min(lengths)), "max": int(max(lengths)),
                              "valid_frac": float(sum(int(v) for v in lengths)) / (wl.seq_len * wl.batch),
                              "units": "valid timesteps (sum of sequence lengths) x 1"}
    return cfg


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def pick_workload(args):
    """The named workload, or a copy of it on --seq-len timesteps (same seed,
    shapes and draws otherwise; the name records the length)."""
    import dataclasses
    import synth
    wl = synth.WORKLOADS[args.workload]
    if args.seq_len is not None and args.seq_len != wl.seq_len:
        wl = dataclasses.replace(wl, name=f"{wl.name}@T{args.seq_len}", seq_len=int(args.seq_len))
    return wl


def run_ours(args):
    import numpy as np
    import torch
    import synth
    import bwd_persistent_cta_gb300 as R
    from bwd_persistent_cta_gb300 import build as B

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        B.build()
    if dist is not None:
        dist.barrier()
    B.build()

    wl = pick_workload(args)
    inp = synth.make_inputs(wl)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    dev = torch.device("cuda", local)

    def dt(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev, tdt)

    rnn = R.RNN(wl.mode, wl.input_size, wl.hidden_size, wl.seq_len, wl.batch, wl.num_layers, wl.bidirectional,
                wl.reset_after, wl.dtype, wl.gate_order, wl.batch_first, device=dev, recompute=wl.recompute)
    # variable-length workloads: the work is the valid steps (sum of lengths)
    valid_frac = 1.0
    if inp.lengths is not None:
        rnn.set_seq_lengths([int(v) for v in inp.lengths])
        valid_frac = float(np.sum(inp.lengths)) / (wl.seq_len * wl.batch)
    w = dt(synth.flatten_params(wl, inp.params))
    x, dy, hx, cx = dt(inp.x), dt(inp.dy), dt(inp.h0), dt(inp.c0)
    D = wl.dirs
    y = torch.empty(wl.seq_len, wl.batch, D * wl.hidden_size, dtype=tdt, device=dev)
    S = (wl.num_layers * D, wl.batch, wl.hidden_size)
    hy = torch.empty(S, dtype=tdt, device=dev)
    cy = torch.empty(S, dtype=tdt, device=dev) if wl.mode == "lstm" else None
    dx = torch.empty_like(x)
    dhx = torch.empty(S, dtype=tdt, device=dev)
    dcx = torch.empty(S, dtype=tdt, device=dev) if wl.mode == "lstm" else None
    dw = torch.empty(rnn.weight_count, dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    def step():
        rnn.forward(x, w, hx, cx, train=not wl.forward_only, y=y, hy=hy, cy=cy)
        if not wl.forward_only:
            rnn.backward_data(dy, w, None, None, dx=dx, dhx=dhx, dcx=dcx, cx=cx)
            rnn.backward_weights(x, dw=dw)

    for _ in range(args.warmup):
        step()
    rnn.sync()

    K = args.steps
    if K is None:
        # enough steps for a timed region of at least MIN_TIMED_S (the same K on every rank)
        t0 = time.perf_counter()
        step()
        rnn.sync()
        K = max(10, int(MIN_TIMED_S / max(time.perf_counter() - t0, 1e-4)) + 1)
        if dist is not None:
            kt = torch.tensor([K], dtype=torch.int64, device=dev)
            dist.all_reduce(kt, op=dist.ReduceOp.MAX)
            K = int(kt.item())
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0] or local)
                           if os.environ.get("CUDA_VISIBLE_DEVICES") else local)
    R.rnn_get_timing(rnn.handle)
    R.rnn_set_timing(rnn.handle, True)
    launches0 = rnn.launches()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall0 = time.perf_counter()
    for k in range(K):
        flush.zero_()
        starts[k].record()
        step()
        ends[k].record()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    if dist is not None:
        dist.barrier()
    rnn.sync()
    R.rnn_set_timing(rnn.handle, False)
    launches = rnn.launches() - launches0
    cls_ms, cls_n, cls_bytes = R.rnn_get_timing_ex(rnn.handle)
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K, dist, dev)

    # --- end to end through the C ABI with host buffers --------------------
    xh = x.cpu().pin_memory()
    dyh = dy.cpu().pin_memory()
    res = y if wl.forward_only else dw            # the step's result read back to the host
    resh = torch.empty(res.shape, dtype=res.dtype).pin_memory()
    for _ in range(2):
        x.copy_(xh, non_blocking=True); dy.copy_(dyh, non_blocking=True); step(); resh.copy_(res, non_blocking=True)
    torch.cuda.synchronize()
    Ke = max(3, K // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # dy is needed only by the backward: its upload runs on a copy stream
    # during the forward (started once x is in, so the two uploads do not share
    # the host link; waited for before the backward)
    copy_stream = torch.cuda.Stream(device=dev)
    started, dy_in = torch.cuda.Event(), torch.cuda.Event()
    main = torch.cuda.current_stream()
    e_ms = 0.0
    for _ in range(Ke):
        flush.zero_()
        e0.record()
        x.copy_(xh, non_blocking=True)
        started.record()
        if wl.forward_only:
            step()
        else:
            copy_stream.wait_event(started)
            with torch.cuda.stream(copy_stream):
                dy.copy_(dyh, non_blocking=True)
                dy_in.record()
            rnn.forward(x, w, hx, cx, train=True, y=y, hy=hy, cy=cy)
            main.wait_event(dy_in)
            rnn.backward_data(dy, w, None, None, dx=dx, dhx=dhx, dcx=dcx, cx=cx)
            rnn.backward_weights(x, dw=dw)
        resh.copy_(res, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        e_ms += e0.elapsed_time(e1)
    e_ms = max_over_ranks(e_ms / Ke, dist, dev)
    rnn.sync()

    units = wl.seq_len * wl.batch * world * valid_frac
    value = job_throughput(wl.seq_len * wl.batch * valid_frac, world, ms)
    tflops = wl.flops() * valid_frac * world / (ms / 1e3) / 1e12
    peaks = load_peaks()
    names = R.TIMING_CLASS_NAMES
    per_step = {n: cls_ms[i] / K for i, n in enumerate(names)}
    dom = max(range(len(names)), key=lambda i: cls_ms[i])
    fl = class_flops(wl)
    per_launch_ms = cls_ms[dom] / max(cls_n[dom], 1)
    launches_per_step = cls_n[dom] / K
    flops_per_launch = fl[names[dom]] / max(launches_per_step, 1)
    achieved = flops_per_launch / (per_launch_ms / 1e3) / 1e12
    if wl.dtype == "bf16":
        bound, peak, peak_src = "tensor", peaks["bf16_tflops"], peaks["src"] + " bf16 burst"
    else:
        # the fp32 path runs on the FP32 pipes (FMA), not the tensor cores
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = fp32_fma_tflops(sms, peaks.get("sm_max_mhz") or 2070.0)
        bound, peak_src = "alu", f"derived: {sms} SMs x 128 FP32 lanes x 2 flops x {peaks.get('sm_max_mhz') or 2070.0:.0f} MHz"
    layout = layout_report(names, cls_ms, cls_n, cls_bytes, K, peaks["hbm_gbs"])
    roofline = {"kernel": names[dom], "bound": bound, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": profiled_traffic(names[dom], wl.name),
                "peak_src": peak_src, "share": cls_ms[dom] / max(sum(cls_ms), 1e-9),
                "per_launch_ms": per_launch_ms, "per_class_ms_per_step": per_step}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cols = _oracle_sample_cols(wl, 3.0)
        out, cores = run_oracle_subprocess(wl, 12.0, cols, reps=2)
        times = out["times"][1:]          # the first repeat warms the process up
        cpu = {"value": out["units_per_rep"] * len(times) / sum(times), "unit": UNIT, "cores": cores,
               "kind": "oracle",
               "sample": f"{wl.name} with {cols} of {wl.batch} batch columns, "
                         f"{'fwd' if wl.forward_only else 'fwd+bwd'}, {len(times)} timed repeats in "
                         f"{sum(times):.1f} s after one warm-up (fp64 numpy, all host cores)"}
        # the same sample on one host thread
        out1, _ = run_oracle_subprocess(wl, 6.0, cols, reps=2, threads=1)
        t1 = out1["times"][1:]
        cpu["single_thread"] = {"value": out1["units_per_rep"] * len(t1) / sum(t1), "cores": 1,
                                "timed_s": sum(t1)}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms, "us_per_timestep": ms * 1e3 / wl.seq_len, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
            "config": workload_config(wl, inp.lengths, world),
            "reserve_bytes": rnn.reserve_bytes,
            "tflops": tflops,
            "tflops_unit": "TFLOP/s (algorithmic, sum over layers/dirs of "
                           f"{'' if wl.forward_only else '3*'}2*G*H*(I+H)*B*T)",
            "e2e": {"value": job_throughput(wl.seq_len * wl.batch * valid_frac, world, e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": int(x.numel() * x.element_size() +
                                              (0 if wl.forward_only else dy.numel() * dy.element_size())),
                    "d2h_bytes_per_step": int(res.numel() * res.element_size())},
            "gpu_launches": int(launches), "gpu_launches_per_step": launches / K,
            "roofline": roofline, "layout": layout, "layout_peak_src": peaks["src"] + " HBM copy",
            "clocks": clocks, "cpu_baseline": cpu,
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line))
    rnn.close()
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = pick_workload(args)
    cols = _oracle_sample_cols(wl, 2.0)
    steps = args.steps if args.steps is not None else 10
    out, cores = run_oracle_subprocess(wl, 0.0, cols, reps=args.warmup + steps)
    per_step = out["times"][args.warmup:args.warmup + steps]
    units = out["units_per_rep"] * len(per_step)
    secs = sum(per_step)
    value = units / secs
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(wl, synth.make_lengths(wl), args.gpus),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{wl.name} with {cols} of {wl.batch} batch columns per step, "
                                       f"{'fwd' if wl.forward_only else 'fwd+bwd'}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def self_launch(args) -> int:
    """``--gpus N`` without WORLD_SIZE in the environment: run this script as
    N ranks under torch.distributed.run (one node, rendezvous on 127.0.0.1)
    and return its exit code."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.run(cmd, cwd=ROOT).returncode


def probe_ranks(args) -> None:
    """The launch and aggregation path alone, without a kernel: every rank
    joins the process group (nccl with GPUs, else gloo), the ranks' numbers
    are summed, and rank 0 prints how many ranks took part."""
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    t = torch.tensor([1.0 + rank], dtype=torch.float64)
    if world > 1:
        dist.all_reduce(t)
    slowest = max_over_ranks(float(rank), dist if world > 1 else None, "cpu")
    if rank == 0:
        print(json.dumps({"probe": "ranks", "n_gpus": world, "gpus_requested": args.gpus,
                          "rank_sum": float(t.item()), "max_rank": slowest}))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.oracle_sample:
        oracle_worker(args.oracle_sample)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(self_launch(args))
    if args.probe_ranks:
        probe_ranks(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
