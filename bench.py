#!/usr/bin/env python3
"""Benchmark: sparse MLA (DSA) forward + backward on one GB300.

One step is one pass of the whole hot path on one batch of synthetic input:
dsa_fwd, then the three stages of dsa_bwd.  All calls go through the C ABI.

Workload: DeepSeek-V4 "flash" layout at T=8192, H=128.  Each token has a
128-row sliding window and 512 compressed causal top-k rows (width 640,
non-compact).  KV holds 8192 + 2048 rows of 576 (V = the first 512
columns).  Inputs are bf16 N(0,1) values from a seeded generator.

Metrics:
  - value: fwd+bwd TFLOPS.  fwd FLOPs = 2*H*sum_t K_t*(576+512), with K_t the
    valid gathered slots; bwd = 2.5x fwd.
  - gathered-KV TB/s = sum_t K_t * 1152 B * 2 passes / step time.
  - roofline: the dominant kernel (k_bwd_dq, the dsa_bwd_main stage) against
    the measured bf16 peak.

`--impl reference` times the fp64 CPU oracle on the host cores.  Each step is
a bounded sample of the same workload, scaled to the same unit.

Launch: python bench.py [--gpus N --steps K --warmup W] (torchrun for N > 1:
each rank runs an independent replica, "replicas only").
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FWD_FLOPS_PER_SLOT_HEAD = 2 * (576 + 512)
BWD_DQ_FLOPS_PER_SLOT_HEAD = 2 * (576 + 512 + 576)   # k_bwd_dq: S, dP, dQ
BWD_DKV_FLOPS_PER_SLOT_HEAD = 2 * (576 + 512)        # k_bwd_dkv: dK, dV
ROW_BYTES = 576 * 2
WORKLOAD = dict(name="flash_t8k", T=8192, H=128, topk=512, window=128, W=640, S_kv=8192 + 2048,
                compact=False)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = None

    def _launch(self, interval_ms: int, wait_s: float) -> bool:
        """Start nvidia-smi polling every interval_ms; True once it has
        written a sample (the timed region must not start before that)."""
        fd, self.path = tempfile.mkstemp(prefix="dsa_clocks_", suffix=".csv")
        self.fh = os.fdopen(fd, "w")
        self.proc = subprocess.Popen(
            ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
             "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
            stdout=self.fh, stderr=subprocess.DEVNULL)
        t0 = time.time()
        while time.time() - t0 < wait_s and os.path.getsize(self.path) == 0:
            time.sleep(0.01)
        return os.path.getsize(self.path) > 0

    def start(self):
        # Every 10 ms, so that a timed region of a fraction of a second still
        # holds a dozen samples; every 50 ms if that interval yields nothing.
        try:
            if not self._launch(10, 2.0):
                self._discard()
                self._launch(50, 10.0)
        except Exception:
            self.proc = None

    def _discard(self):
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        try:
            os.remove(self.path)
        except OSError:
            pass

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_workload(device):
    from sparse_top_attention_gb300 import workloads as WL
    return WL.dsv4(T=WORKLOAD["T"], H=WORKLOAD["H"], topk=WORKLOAD["topk"],
                   compact=WORKLOAD["compact"], seed=1005, name=WORKLOAD["name"],
                   value_device=device)


def valid_counts(w):
    from sparse_top_attention_gb300 import workloads as WL
    return WL.valid_slot_count_formula(w.T, WORKLOAD["topk"])


def cpu_oracle_sample(w, budget_s: float, rng_seed: int = 0):
    """Time the fp64 oracle (fwd + bwd) on tokens drawn from the workload
    until `budget_s` seconds of CPU work are done.  Returns (TFLOPS, tokens,
    seconds)."""
    from oracle import dsa_oracle as O
    rng = np.random.default_rng(rng_seed)
    counts = valid_counts(w)
    # the host copies cover only the sampled tokens
    kv = w.kv.cpu()
    sink = w.sink.cpu()
    toks_done, flops, t_used = 0, 0.0, 0.0
    while t_used < budget_s:
        toks = sorted(rng.choice(w.T, size=4, replace=False).tolist())
        idx = w.topk_idxs[toks].cpu()
        q = w.q[toks].cpu()
        dout = w.dout[toks].cpu()
        t0 = time.perf_counter()
        O.forward(q, kv, idx, None, sink, w.scale)
        O.backward(q, kv, idx, None, sink, w.scale, dout)
        t_used += time.perf_counter() - t0
        toks_done += len(toks)
        flops += 3.5 * FWD_FLOPS_PER_SLOT_HEAD * w.H * float(np.sum(counts[toks]))
    return flops / t_used / 1e12, toks_done, t_used


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, rank, world):
    """The oracle arm: fp64 numpy on the host cores, same metric and config."""
    if rank != 0:
        return
    w = make_workload("cuda" if torch.cuda.is_available() else "cpu")
    per_step = []
    # bound the whole reference run to a few minutes whatever K and W are
    step_s = max(0.5, min(args.ref_step_seconds, 150.0 / (args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        tf, n, s = cpu_oracle_sample(w, budget_s=step_s, rng_seed=i)
        if i >= args.warmup:
            per_step.append((tf, n, s))
    value = float(np.mean([x[0] for x in per_step]))
    secs = float(np.mean([x[2] for x in per_step]))
    toks = int(np.mean([x[1] for x in per_step]))
    line = {
        "impl": "reference", "metric": "sparse-MLA fwd+bwd TFLOPS", "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, DeepSeek-V4 flash layout)",
        "config": {"workload": "flash_t8k: T=8192 H=128 window 128 + top-k 512 (W=640), "
                               "S_kv=10240, D_qk=576 D_v=512, non-compact",
                   "sample": f"{toks} random tokens per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
                         "sample": f"fp64 numpy oracle fwd+bwd of {toks} random tokens per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    from sparse_top_attention_gb300 import dsa
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dsa.library()
    w = make_workload(str(dev))
    counts = valid_counts(w)
    sum_k = float(np.sum(counts))
    T, H, S_kv, W = w.T, w.H, w.S_kv, w.W
    fwd_flops = FWD_FLOPS_PER_SLOT_HEAD * H * sum_k
    step_flops = 3.5 * fwd_flops
    bwd_main_flops = BWD_DQ_FLOPS_PER_SLOT_HEAD * H * sum_k
    bwd_dkv_flops = BWD_DKV_FLOPS_PER_SLOT_HEAD * H * sum_k
    gathered_bytes = 2 * ROW_BYTES * sum_k  # one gather list per token, fwd + bwd

    out = torch.empty(T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    dq = torch.empty(T, H, 576, dtype=torch.bfloat16, device=dev)
    dkv = torch.empty(S_kv, 576, dtype=torch.bfloat16, device=dev)
    dsink = torch.empty(H, dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.bwd_workspace_bytes(T, H, S_kv, W), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dsa.fwd(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale, out=out, lse=lse)
        if ev is not None:
            ev[1].record(stream)
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws, entry="dsa_bwd_preprocess")
        if ev is not None:
            ev[2].record(stream)
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws, entry="dsa_bwd_main")
        if ev is not None:
            ev[3].record(stream)
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws, entry="dsa_bwd_finalize")
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dsa.device_status() != 0:
        raise RuntimeError("device status not ok after warm-up")

    # Kernel launches per step: fwd 1; preprocess 1 (k_compact, plus a driver
    # memset); main 1 (k_bwd_dq); finalize 3 (k_bwd_dkv, k_dkv_cast, k_dsink).
    launches_per_step = 1 + 1 + 1 + 3
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    pre_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    main_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    fin_ms = float(np.mean([e[3].elapsed_time(e[4]) for e in evs]))
    assert dsa.device_status() == 0

    value = world * step_flops / (ms_step * 1e-3) / 1e12
    peaks, peak_kind = read_peaks()
    # The kernels are timed in a sub-second loop at full clocks: the burst peak.
    peak = float(peaks["bf16_tflops"])
    main_tflops = bwd_main_flops / (main_ms * 1e-3) / 1e12
    fwd_tflops = fwd_flops / (fwd_ms * 1e-3) / 1e12
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        traffic = json.load(open(tpath)).get("k_bwd_dq")

    # The backward again with DSA_FLAG_DETERMINISTIC (bitwise reproducible
    # dkv), all three stages, for the same steps.
    ws_det = torch.empty(dsa.bwd_workspace_bytes(T, H, S_kv, W, deterministic=True),
                         dtype=torch.uint8, device=dev)

    def bwd_det():
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws_det, deterministic=True)

    for _ in range(args.warmup):
        bwd_det()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    d0.record(stream)
    for _ in range(args.steps):
        bwd_det()
    d1.record(stream)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    bwd_det_ms = d0.elapsed_time(d1) / args.steps
    del ws_det

    graph_leg = run_graph_leg(args, w, dev, out, lse, dq, dkv, dsink, ws, fwd_flops)
    varlen_leg = run_varlen_leg(args, dev, stream)
    d512_leg = run_d512_leg(args, dev, stream)
    small_h_leg = run_small_h_leg(args, dev, stream)

    # End to end through the public API: pinned host inputs -> device, fwd + bwd,
    # outputs -> pinned host, every step.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, dev, stream, step_flops, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, n, s = cpu_oracle_sample(w, budget_s=args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
               "sample": f"fp64 numpy oracle fwd+bwd of {n} random tokens of the workload ({s:.1f} s)"}

    if rank == 0:
        line = {
            "metric": "sparse-MLA fwd+bwd TFLOPS", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded bf16 N(0,1), DeepSeek-V4 flash layout)",
            "config": {"workload": f"{WORKLOAD['name']}: T={w.T} H=128 window 128 + top-k 512 "
                                   f"(W=640), S_kv={w.S_kv}, D_qk=576 D_v=512, non-compact, B=1",
                       "valid_slots": int(sum_k), "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (q 1.2 GB, dout 1.07 GB per step)"},
            "gathered_kv_tbps": world * gathered_bytes / (ms_step * 1e-3) / 1e12,
            "gathered_kv_frac_of_hbm": (gathered_bytes / (ms_step * 1e-3) / 1e9) / float(peaks["hbm_gbs"]),
            "frac_of_bf16_peak": value / world / peak,
            "kernels_ms": {"fwd": fwd_ms, "bwd_preprocess": pre_ms, "bwd_main (k_bwd_dq)": main_ms,
                           "bwd_finalize (k_bwd_dkv + cast + d_sink)": fin_ms},
            "bwd_ms": pre_ms + main_ms + fin_ms,
            "bwd_deterministic_ms": bwd_det_ms,
            "graph_medians": graph_leg,
            "varlen": varlen_leg,
            "d512": d512_leg,
            "small_h": small_h_leg,
            "fwd_tflops": fwd_tflops,
            "bwd_finalize_tflops": bwd_dkv_flops / (fin_ms * 1e-3) / 1e12,
            "roofline": {"kernel": "k_bwd_dq", "bound": "tensor", "achieved": main_tflops,
                         "peak": peak, "unit": "TFLOP/s", "frac": main_tflops / peak,
                         "traffic": traffic, "peak_kind": f"bf16 burst ({peak_kind})",
                         "flops_per_launch": bwd_main_flops},
            "clocks": clk,
            "gpu_launches": launches_per_step * args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_graph_leg(args, w, dev, out, lse, dq, dkv, dsink, ws, fwd_flops, warm=10, replays=50):
    """The timing protocol of the pages' table (flash-attention "[CuTe, SM100]
    Support 1..128 Q heads in sparse MLA via in-kernel TMA padding",
    "Performance at DeepSeek-V4 shapes": medians over CUDA-graph replays):
    dsa_fwd and the whole dsa_bwd are each captured once into a CUDA graph,
    replayed `warm` times, then timed replay by replay with CUDA events on
    the replay stream; the medians are reported.  The KV tensor stays in L2
    between replays (warm, as on the pages); q and dout do not fit."""
    from sparse_top_attention_gb300 import dsa
    s = torch.cuda.Stream(dev)

    def fwd():
        dsa.fwd(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale, out=out, lse=lse)

    def bwd():
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):          # the library's per-device set-up is done by now
        fwd()
        bwd()
    torch.cuda.synchronize()
    g_f, g_b = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_f, stream=s):
        fwd()
    with torch.cuda.graph(g_b, stream=s):
        bwd()
    n = max(replays, args.steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    with torch.cuda.stream(s):
        for _ in range(warm):
            g_f.replay()
            g_b.replay()
        for e in ev:
            e[0].record(s)
            g_f.replay()
            e[1].record(s)
            g_b.replay()
            e[2].record(s)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    fwd_ms = float(np.median([e[0].elapsed_time(e[1]) for e in ev]))
    bwd_ms = float(np.median([e[1].elapsed_time(e[2]) for e in ev]))
    return {"protocol": f"CUDA-graph replays: {warm} warm-up, median of {n}",
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_plus_bwd_ms": fwd_ms + bwd_ms,
            "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
            "bwd_tflops": 2.5 * fwd_flops / (bwd_ms * 1e-3) / 1e12,
            "step_tflops": 3.5 * fwd_flops / ((fwd_ms + bwd_ms) * 1e-3) / 1e12}


def run_varlen_leg(args, dev, stream):
    """fwd + bwd through dsa_fwd_varlen / dsa_bwd_varlen on four packed
    2048-token sequences (the same 8192 tokens as the headline workload, each
    sequence with its own window and compressed rows)."""
    from sparse_top_attention_gb300 import dsa
    from sparse_top_attention_gb300 import workloads as WL
    lengths = [2048] * 4
    w = WL.varlen(lengths, H=WORKLOAD["H"], topk=WORKLOAD["topk"], compact=False, seed=1006,
                  value_device=str(dev))
    sum_k = float(sum(WL.valid_slot_count_formula(n, WORKLOAD["topk"]).sum() for n in lengths))
    flops = 3.5 * FWD_FLOPS_PER_SLOT_HEAD * w.H * sum_k
    vl = (w.cu_seqlens_q, w.cu_seqlens_kv)
    out = torch.empty(w.T, w.H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.T, w.H, dtype=torch.float32, device=dev)
    dq = torch.empty(w.T, w.H, 576, dtype=torch.bfloat16, device=dev)
    dkv = torch.empty(w.S_kv, 576, dtype=torch.bfloat16, device=dev)
    dsink = torch.empty(w.H, dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.bwd_workspace_bytes(w.T, w.H, w.S_kv, w.W), dtype=torch.uint8,
                     device=dev)

    def step():
        dsa.fwd(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale, out=out, lse=lse, varlen=vl)
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws, varlen=vl)

    for _ in range(args.warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    ms = e0.elapsed_time(e1) / args.steps
    return {"workload": "4 packed sequences x 2048 tokens, H=128, window 128 + top-k 512",
            "valid_slots": int(sum_k), "ms_per_step": ms,
            "tflops": flops / (ms * 1e-3) / 1e12}


def run_d512_leg(args, dev, stream):
    """The same layout with D_qk = D_v = 512 (no rope part), the row width of
    the DeepSeek-V4 performance table on the flash-attention page: fwd and
    bwd timed separately, FLOPs by valid slots (2 * H * (512 + 512) each)."""
    from sparse_top_attention_gb300 import dsa
    from sparse_top_attention_gb300 import workloads as WL
    w = WL.dsv4(T=WORKLOAD["T"], H=WORKLOAD["H"], topk=WORKLOAD["topk"], compact=False,
                seed=1007, name="flash_t8k_d512", value_device=str(dev), d_qk=512)
    sum_k = float(WL.valid_slot_count_formula(w.T, WORKLOAD["topk"]).sum())
    fwd_flops = 2 * (512 + 512) * w.H * sum_k
    out = torch.empty(w.T, w.H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.T, w.H, dtype=torch.float32, device=dev)
    dq = torch.empty(w.T, w.H, 512, dtype=torch.bfloat16, device=dev)
    dkv = torch.empty(w.S_kv, 512, dtype=torch.bfloat16, device=dev)
    dsink = torch.empty(w.H, dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.bwd_workspace_bytes(w.T, w.H, w.S_kv, w.W, d_qk=512),
                     dtype=torch.uint8, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]

    def step(e=None):
        if e:
            e[0].record(stream)
        dsa.fwd(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale, out=out, lse=lse)
        if e:
            e[1].record(stream)
        dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, dq=dq, dkv=dkv,
                dsink=dsink, workspace=ws)
        if e:
            e[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for e in ev:
        step(e)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    return {"workload": "flash layout T=8192 H=128, window 128 + top-k 512, D_qk=D_v=512",
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
            "bwd_tflops": 2.5 * fwd_flops / (bwd_ms * 1e-3) / 1e12}


def run_small_h_leg(args, dev, stream):
    """The headline layout at fewer heads (H = 16, 64): fwd + bwd per step.
    The kernels put heads on the MMA N side, so a gathered block costs about
    the same at any H up to the head group; the time per token, not per
    head, is what stays put."""
    from sparse_top_attention_gb300 import dsa
    from sparse_top_attention_gb300 import workloads as WL
    res = {}
    for H in (16, 64):
        w = WL.dsv4(T=WORKLOAD["T"], H=H, topk=WORKLOAD["topk"], compact=False, seed=1008,
                    name=f"flash_t8k_h{H}", value_device=str(dev))
        sum_k = float(WL.valid_slot_count_formula(w.T, WORKLOAD["topk"]).sum())
        flops = 3.5 * FWD_FLOPS_PER_SLOT_HEAD * H * sum_k
        out = torch.empty(w.T, H, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(w.T, H, dtype=torch.float32, device=dev)
        ws = torch.empty(dsa.bwd_workspace_bytes(w.T, H, w.S_kv, w.W), dtype=torch.uint8,
                         device=dev)

        def step():
            dsa.fwd(w.q, w.kv, w.topk_idxs, None, w.sink, w.scale, out=out, lse=lse)
            dsa.bwd(w.q, w.kv, w.topk_idxs, None, w.sink, out, lse, w.dout, w.scale, workspace=ws)

        for _ in range(args.warmup):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        assert dsa.device_status() == 0
        ms = e0.elapsed_time(e1) / args.steps
        res[f"H{H}"] = {"ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                        "us_per_token": ms * 1e3 / w.T}
        del w, out, lse, ws
    return res


def run_e2e(args, w, dev, stream, step_flops, world):
    """Every step copies its inputs in from pinned host memory, runs fwd + bwd
    and copies every output back out, as a training loop would.  The copies
    of step i + 1 (in) and step i - 1 (out) overlap the compute of step i:
    three streams, double-buffered device inputs and outputs, and events so
    that no buffer is overwritten while a copy or kernel still uses it."""
    from sparse_top_attention_gb300 import dsa
    host = {k: getattr(w, k).cpu().pin_memory() for k in ("q", "kv", "topk_idxs", "sink", "dout")}
    T, H, S_kv, W = w.T, w.H, w.S_kv, w.W

    def outputs():
        return {"out": torch.empty(T, H, 512, dtype=torch.bfloat16, device=dev),
                "lse": torch.empty(T, H, dtype=torch.float32, device=dev),
                "dq": torch.empty(T, H, 576, dtype=torch.bfloat16, device=dev),
                "dkv": torch.empty(S_kv, 576, dtype=torch.bfloat16, device=dev),
                "dsink": torch.empty(H, dtype=torch.float32, device=dev)}

    d = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    outs = [outputs() for _ in range(2)]
    hout = [{k: torch.empty_like(v, device="cpu").pin_memory() for k, v in outs[0].items()}
            for _ in range(2)]
    ws = torch.empty(dsa.bwd_workspace_bytes(T, H, S_kv, W), dtype=torch.uint8, device=dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in hout[0].values())
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp = stream
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, comp_done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in comp_done + out_free:      # both buffer sets start free
        e.record(comp)

    def step(i):
        u = i & 1
        with torch.cuda.stream(s_in):   # inputs of step i (set u is free once step i-2 is done)
            s_in.wait_event(comp_done[u])
            for k in host:
                d[u][k].copy_(host[k], non_blocking=True)
            in_ready[u].record(s_in)
        comp.wait_event(in_ready[u])
        comp.wait_event(out_free[u])    # step i-2's outputs have been copied out
        x, o = d[u], outs[u]
        dsa.fwd(x["q"], x["kv"], x["topk_idxs"], None, x["sink"], w.scale, out=o["out"],
                lse=o["lse"], stream=comp)
        dsa.bwd(x["q"], x["kv"], x["topk_idxs"], None, x["sink"], o["out"], o["lse"], x["dout"],
                w.scale, dq=o["dq"], dkv=o["dkv"], dsink=o["dsink"], workspace=ws, stream=comp)
        comp_done[u].record(comp)
        with torch.cuda.stream(s_out):  # outputs of step i
            s_out.wait_event(comp_done[u])
            for k in hout[u]:
                hout[u][k].copy_(o[k], non_blocking=True)
            out_free[u].record(s_out)

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 10))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(s_in)                     # before the first input copy
    for i in range(steps):
        step(i)
    e1.record(s_out)                    # after the last output copy (it follows all other work)
    torch.cuda.synchronize()
    assert dsa.device_status() == 0
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    return {"value": world * step_flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "steps": steps, "overlap": "copies of neighbouring steps overlap the compute"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=6.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=int, default=WORKLOAD["T"],
                    help="tokens (smaller values only for profiling captures)")
    args = ap.parse_args()
    if args.T != WORKLOAD["T"]:
        WORKLOAD["T"] = args.T
        WORKLOAD["S_kv"] = args.T + args.T // 4
        WORKLOAD["name"] = f"flash_T{args.T}"
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
