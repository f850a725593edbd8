#!/usr/bin/env python
"""Throughput of the attention core (forward + backward) on one GB300.

A step is one xt_attn_fwd + xt_attn_bwd (all kernels of the path) over one
batch of synthetic inputs resident in HBM. Metric: causal GQA attention
fwd+bwd TFLOP/s, FLOPs counted as 2*B*H*S^2*D forward and 2.5x that
backward. The L2 is flushed (a 512 MB write) between timed steps, outside the
per-step CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle timed on host cores
  python bench.py --mode decode ...      # one decode step against a full KV cache
  python bench.py --mode varlen ...      # fwd+bwd over a packed batch of unequal samples

In decode mode a step is one xt_attn_decode call: every sequence's next token
against a cache that holds its whole capacity (the largest cache read), and
the metric is the cache bytes read per second (K-hat and V rows, the algorithmic
bytes of the step); the cache is larger than L2, so no flush is needed.

In varlen mode a step is xt_attn_fwd_varlen + xt_attn_bwd_varlen over 16384
packed rows (samples of 256..4096 rows, seeded), FLOPs counted per sample as
2*H*len^2*D forward and 2.5x that backward; otherwise as the default mode.

Under torchrun (N > 1) every rank runs its own shard of independent batch
units on its own GPU (weak scaling, no collective on the data path); rank 0
prints one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal GQA attention fwd+bwd TFLOP/s at 1 GB300 and % of dense BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "qwen3_like_bf16"
DECODE_METRIC = ("GQA decode step (each sequence's next token against its full KV cache): "
                 "cache bytes read per second at 1 GB300")
DECODE_WORKLOAD = "qwen3_like_decode_bf16"
VARLEN_METRIC = ("packed variable-length causal GQA attention fwd+bwd TFLOP/s (block-causal, "
                 "FLOPs counted per sample) at 1 GB300")
VARLEN_WORKLOAD = "qwen3_like_varlen_bf16"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(tflops=float(p["bf16_tflops"]), tflops_sustained=float(p["bf16_tflops_sustained"]),
                    hbm_gbs=float(p["hbm_gbs"]), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(tflops=1900.0, tflops_sustained=1700.0, hbm_gbs=6800.0, source="fallback")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch of independent units (weak scaling)."""
    return base_seed + rank


def reduce_max(values, device=None):
    """Element-wise max over ranks of a list of floats (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
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
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_pci_id(torch):
    try:
        p = torch.cuda.get_device_properties(torch.cuda.current_device())
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(w, s_len, cores):
    """A bounded sample of workload w for the CPU oracle: batch element 0, as
    many kv groups as give one query head per core, sequence cut to s_len.
    Returns (sub-workload, inputs as float64, description)."""
    import numpy as np  # noqa: F401
    from causal_gqa_attention_xt_gb300.inputs import make_inputs, to_f64
    n_groups = max(1, min(w.G, cores // w.group))
    sub = w.with_(B=1, S=s_len, H=n_groups * w.group, G=n_groups)
    x = to_f64(make_inputs(sub))
    desc = (f"B=1, S={s_len}, {sub.H} query heads / {sub.G} kv heads (group {w.group}), "
            f"D={w.D}: oracle fwd + bwd, fp64, {min(cores, sub.H)} threads")
    return sub, x, desc


def run_oracle_step(sub, x, threads):
    import oracle
    oracle.attn_fwd(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], sub.eps, sub.theta,
                    nthreads=threads)
    oracle.attn_bwd(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], x["dout"], sub.eps,
                    sub.theta, nthreads=threads)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds_target=20.0):
    import oracle
    oracle.build()
    cores = host_cores()
    sub, x, desc = oracle_sample(w, w.S, cores)
    threads = min(cores, sub.H)
    t0 = time.perf_counter()
    run_oracle_step(sub, x, threads)
    dt = time.perf_counter() - t0
    flops = sub.fwd_flops + sub.bwd_flops
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc, "seconds": dt}


def oracle_configs():
    """The CPU oracle (fwd + bwd, fp64) timed on every configured workload on
    this host's cores. The tiny fp32 and GQA bring-up shapes run whole, on one
    thread and on all threads; the larger ones run a sample of one batch
    element with as many query heads as there are threads (one head per
    thread, whole kv groups, full sequence), and the whole config's time is
    estimated from it by the number of such head waves. One JSON line per
    workload."""
    import math
    import oracle
    from causal_gqa_attention_xt_gb300.inputs import WORKLOADS, make_inputs, to_f64
    oracle.build()
    cores = host_cores()
    for name in CONFIG_WORKLOADS:
        w = WORKLOADS[name]
        runs = []
        if name in ("tiny_mha_f32", "gqa_bf16"):
            x = to_f64(make_inputs(w))
            for req in sorted({1, cores}):
                threads = oracle.head_threads(req, w.S, 2, w.B * w.H)
                t0 = time.perf_counter()
                run_oracle_step(w, x, threads)
                dt = time.perf_counter() - t0
                runs.append({"threads": threads, "sample": "whole workload", "seconds": dt,
                             "tflops": (w.fwd_flops + w.bwd_flops) / dt / 1e12,
                             "est_full_seconds": dt})
        else:
            n_groups = max(1, min(w.G, cores // w.group))
            sub = w.with_(B=1, H=n_groups * w.group, G=n_groups)
            x = to_f64(make_inputs(sub))
            threads = oracle.head_threads(min(cores, sub.H), sub.S, 2, sub.H)
            t0 = time.perf_counter()
            run_oracle_step(sub, x, threads)
            dt = time.perf_counter() - t0
            waves_sub = math.ceil(sub.H / threads)
            waves_full = w.B * math.ceil(w.H / threads)
            runs.append({"threads": threads,
                         "sample": f"B=1, {sub.H} query heads / {sub.G} kv heads, S={w.S}",
                         "seconds": dt, "tflops": (sub.fwd_flops + sub.bwd_flops) / dt / 1e12,
                         "est_full_seconds": dt * waves_full / waves_sub})
        print(json.dumps({"oracle_config": name, "B": w.B, "S": w.S, "n_heads": w.H,
                          "n_kv_heads": w.G, "head_dim": w.D, "dtype_in": w.dtype,
                          "arith": "f64", "host_cores": cores, "runs": runs}), flush=True)
    return 0


def longest_sample(w):
    """The longest sample of a packed batch as a one-element batched workload
    (what the oracle times for the packed mode's CPU numbers)."""
    from causal_gqa_attention_xt_gb300.inputs import Workload
    return Workload(w.name + "_longest", 1, w.max_len, w.H, w.G, w.D, w.theta, w.eps, w.dtype,
                    w.seed)


def bench_reference(args, w, metric=None, workload_name=None):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = host_cores()
    s_len = min(w.S, args.ref_seq)
    sub, x, desc = oracle_sample(w, s_len, cores)
    threads = min(cores, sub.H)
    for _ in range(args.warmup):
        run_oracle_step(sub, x, threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run_oracle_step(sub, x, threads)
        times.append(time.perf_counter() - t0)
    flops = sub.fwd_flops + sub.bwd_flops
    value = flops * len(times) / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": metric or METRIC, "value": value, "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name or w.name, "B": w.B, "S": w.S, "n_heads": w.H,
                   "n_kv_heads": w.G, "head_dim": w.D, "theta": w.theta, "eps": w.eps,
                   "sample_per_step": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def bench_ours(args, w):
    import torch
    import torch.distributed as dist

    from causal_gqa_attention_xt_gb300 import build as xbuild
    from causal_gqa_attention_xt_gb300 import xt
    from causal_gqa_attention_xt_gb300.inputs import PackedWorkload, make_inputs, make_packed_inputs

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    xbuild.build()
    xt.lib()
    packed = isinstance(w, PackedWorkload)
    code = 1 if w.dtype == "bf16" else 0

    # each rank owns its own shard of batch units (weak scaling)
    if packed:
        wr = dataclasses.replace(w, seed=shard_seed(w.seed, rank))
        cpu = make_packed_inputs(wr)
        d = {k: v.to(dev) for k, v in cpu.items()}

        def fwd(dd, **kw):
            return xt.xt_attn_fwd_varlen(dd["q"], dd["k"], dd["v"], dd["gamma_q"], dd["gamma_k"],
                                         dd["cu_seqlens"], w.max_len, w.eps, w.theta, **kw)

        def bwd(dd, saved_, **kw):
            return xt.xt_attn_bwd_varlen(dd["q"], dd["k"], dd["v"], dd["gamma_q"], dd["gamma_k"],
                                         dd["cu_seqlens"], w.max_len, saved_, dd["dout"], w.eps,
                                         w.theta, **kw)

        ws_bytes = xt.xt_attn_varlen_workspace_bytes(w.T, len(w.lens), w.max_len, w.H, w.G, w.D, code,
                                                     True)
    else:
        wr = w.with_(seed=shard_seed(w.seed, rank))
        cpu = make_inputs(wr)
        d = {k: v.to(dev) for k, v in cpu.items()}

        def fwd(dd, **kw):
            return xt.xt_attn_fwd(dd["q"], dd["k"], dd["v"], dd["gamma_q"], dd["gamma_k"], w.eps,
                                  w.theta, **kw)

        def bwd(dd, saved_, **kw):
            return xt.xt_attn_bwd(dd["q"], dd["k"], dd["v"], dd["gamma_q"], dd["gamma_k"], saved_,
                                  dd["dout"], w.eps, w.theta, **kw)

        ws_bytes = xt.xt_attn_workspace_bytes(w.B, w.S, w.H, w.G, w.D, code, True)
    saved = fwd(d)
    grads = bwd(d, saved)
    ws = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    flush = torch.empty(512 * 1024 * 1024, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def fwd_only(dd=d, sv=saved):
        fwd(dd, out=sv["out"], lse=sv["lse"], q_hat=sv["q_hat"], k_hat=sv["k_hat"],
            rstd_q=sv["rstd_q"], rstd_k=sv["rstd_k"], workspace=ws)

    def bwd_only(dd=d, sv=saved, gr=grads):
        bwd(dd, sv, dq=gr["dq"], dk=gr["dk"], dv=gr["dv"], dgamma_q=gr["dgamma_q"],
            dgamma_k=gr["dgamma_k"], workspace=ws)

    def step():
        fwd_only()
        bwd_only()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if xt.xt_attn_check() != xt.XT_OK:
        raise RuntimeError("device error flag raised during warm-up")

    # ---- timed region: K steps, events per step, L2 flushed between steps
    clocks = ClockSampler(gpu_pci_id(torch))
    clocks.start()
    time.sleep(0.4)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        fwd_only()
        ev[i][1].record(stream)
        bwd_only()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    # the same K steps again with the library's per-launch events on (kernel
    # times for the roofline), outside the timed region so they add nothing to it
    xt.xt_timing_reset()
    xt.xt_timing_enable(True)
    for i in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    xt.xt_timing_enable(False)
    per_kernel = xt.xt_timing_query()
    clk = clocks.stop()
    if xt.xt_attn_check() != xt.XT_OK:
        raise RuntimeError("device error flag raised during the timed steps")
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    step_ms_local = sum(fwd_ms + bwd_ms) / args.steps
    fwd_ms_local = sum(fwd_ms) / args.steps
    bwd_ms_local = sum(bwd_ms) / args.steps
    step_ms, fwd_ms_m, bwd_ms_m = reduce_max([step_ms_local, fwd_ms_local, bwd_ms_local], dev)

    # ---- end to end through the public API: pinned host buffers in and out
    pin = {k: v.pin_memory() for k, v in cpu.items()}
    sets = [(d, saved, grads)]
    d1 = {k: v.clone() for k, v in d.items()}
    s1 = fwd(d1)
    sets.append((d1, s1, bwd(d1, s1)))
    out_keys = ("dq", "dk", "dv", "dgamma_q", "dgamma_k")
    dev_outs = [dict(out=sv["out"], **{k: gr[k] for k in out_keys}) for _, sv, gr in sets]
    host_outs = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()}
                 for o in dev_outs]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(v.numel() * v.element_size() for v in host_outs[0].values())

    def compute(k):
        dd, sv, gr = sets[k]
        fwd_only(dd, sv)
        bwd_only(dd, sv, gr)

    e2e_ms = reduce_max([pipelined_e2e(torch, args.steps, pin, [x[0] for x in sets], compute,
                                       dev_outs, host_outs)], dev)[0]
    if xt.xt_attn_check() != xt.XT_OK:
        raise RuntimeError("device error flag raised during the end-to-end steps")

    flops_step = w.fwd_flops + w.bwd_flops
    value = world * flops_step / (step_ms * 1e-3) / 1e12
    peaks = load_peaks()

    # ---- roofline of the dominant kernel (largest share of the timed region)
    fwd_f, D = w.fwd_flops, w.D
    algo_flops = {  # algorithmic FLOPs per launch
        "fwd_tcgen05_bf16": fwd_f, "fwd_simt_f32": fwd_f,
        "bwd_dkdv_tcgen05_bf16": 2.0 * fwd_f, "bwd_dkdv_simt_f32": 2.0 * fwd_f,
        "bwd_dq_tcgen05_bf16": 0.5 * fwd_f, "bwd_dq_simt_f32": 0.5 * fwd_f,
    }
    top = max(per_kernel.items(), key=lambda kv: kv[1][0]) if per_kernel else None
    roofline = None
    if top is not None:
        name, (tot_ms, n) = top
        avg_s = tot_ms / n * 1e-3
        esz = 2 if w.dtype == "bf16" else 4
        if name in algo_flops:
            ach = algo_flops[name] / avg_s / 1e12
            roofline = {"kernel": name, "bound": "tensor", "achieved": ach,
                        "peak": peaks["tflops"], "unit": "TFLOP/s", "frac": ach / peaks["tflops"],
                        "peak_source": f"{peaks['source']} bf16 burst",
                        "frac_of_sustained": ach / peaks["tflops_sustained"],
                        "traffic": None, "avg_launch_ms": tot_ms / n}
        else:
            rows = w.T if packed else w.B * w.S
            rows_q, rows_k = rows * w.H, rows * w.G
            algo_bytes = {
                "prologue_qknorm_rope": 2 * esz * D * (rows_q + rows_k) + 4 * (rows_q + rows_k),
                "bwd_epilogue_rope_norm": (4 + 2 * esz) * D * (rows_q + rows_k) + 4 * (rows_q + rows_k),
                "bwd_pre_dlt": 2 * esz * D * rows_q + 4 * rows_q,
            }.get(name, 0)
            ach = algo_bytes / avg_s / 1e9
            roofline = {"kernel": name, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                        "peak_source": f"{peaks['source']} copy", "traffic": None,
                        "avg_launch_ms": tot_ms / n}
    traffic_file = os.path.join(ROOT, "profiles", "traffic.json")
    if roofline is not None and os.path.exists(traffic_file):
        try:
            with open(traffic_file) as f:
                tr = json.load(f)
            ent = tr.get(roofline["kernel"], {})
            if (ent.get("workload") == w.name and roofline["kernel"] in KERNEL_SOURCES
                    and ent.get("source_hash") == source_hash(roofline["kernel"])):
                roofline["traffic"] = ent.get("bytes_per_launch")
        except (OSError, ValueError):
            pass

    launches = sum(n for _, n in per_kernel.values())
    if packed:
        config = {"workload": w.name, "total_rows": w.T, "samples": len(w.lens),
                  "lengths": list(w.lens), "max_seqlen": w.max_len, "n_heads": w.H,
                  "n_kv_heads": w.G, "head_dim": w.D, "theta": w.theta, "eps": w.eps,
                  "length_mix": "uniform 256..4096 rows per sample (seeded), last takes the rest"}
    else:
        config = {"workload": w.name, "B": w.B, "S": w.S, "n_heads": w.H, "n_kv_heads": w.G,
                  "head_dim": w.D, "theta": w.theta, "eps": w.eps, "per_rank_batch": w.B}
    config["l2"] = "flushed between timed steps (512 MB write, outside the step events)"
    config["e2e"] = ("pinned host -> device copy of q/k/v/dout/gammas and device -> pinned host "
                     "copy of out/dq/dk/dv/dgammas every step, on copy streams overlapping the "
                     "neighbouring steps' compute (two buffer sets); inputs larger than L2, no flush")
    config["inputs"] = "N(0,1) q/k/v/dout rounded to bf16, gammas 1+0.1*N(0,1) fp32, seed 0+rank"
    line = {
        "metric": VARLEN_METRIC if packed else METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config,
        "fwd": {"ms": fwd_ms_m, "tflops": w.fwd_flops / (fwd_ms_m * 1e-3) / 1e12,
                "frac_of_peak": w.fwd_flops / (fwd_ms_m * 1e-3) / 1e12 / peaks["tflops"]},
        "bwd": {"ms": bwd_ms_m, "tflops": w.bwd_flops / (bwd_ms_m * 1e-3) / 1e12,
                "frac_of_peak": w.bwd_flops / (bwd_ms_m * 1e-3) / 1e12 / peaks["tflops"]},
        "frac_of_peak": value / world / peaks["tflops"],
        "roofline": roofline,
        "kernels": {k: {"total_ms": v[0], "launches": v[1], "share": v[0] / max(1e-9, sum(x[0] for x in per_kernel.values()))}
                    for k, v in per_kernel.items()},
        "e2e": {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if world == 1 and not packed and not args.no_configs:
        # every configured workload, timed after the headline (outside its timed region)
        line["configs"] = bench_configs(torch, xt, dev, flush, min(args.steps, 10),
                                        max(3, min(args.warmup, 5)), peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(longest_sample(w) if packed else w)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# The workloads the attention core is specified on, timed beside the headline
# (the tiny fp32 shape, GQA bring-up, dim768 MHA and GQA, Qwen3-like, long MQA)
# plus the pages' own dim768 run (24 heads x 32 at S = 256).
CONFIG_WORKLOADS = ("tiny_mha_f32", "gqa_bf16", "dim768_mha_bf16", "dim768_gqa_bf16",
                    "qwen3_like_bf16", "mqa_long_bf16", "dim768_hd32_bf16")


def bench_configs(torch, xt, dev, flush, steps, warmup, peaks):
    """fwd / bwd / step times of every configured workload in this process: the
    same calls, CUDA events on the launch stream and L2 flush between steps as
    the headline; then a second pass with the library's per-launch events for
    the per-kernel times (ms per launch). Inputs are seeded like the headline's."""
    from causal_gqa_attention_xt_gb300.inputs import WORKLOADS, make_inputs
    stream = torch.cuda.current_stream()
    res = {}
    for name in CONFIG_WORKLOADS:
        w = WORKLOADS[name]
        d = {k: v.to(dev) for k, v in make_inputs(w).items()}
        code = 1 if w.dtype == "bf16" else 0
        ws = torch.empty(max(16, xt.xt_attn_workspace_bytes(w.B, w.S, w.H, w.G, w.D, code, True)),
                         device=dev, dtype=torch.uint8)
        sv = xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], w.eps, w.theta,
                            workspace=ws)
        gr = xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], sv, d["dout"],
                            w.eps, w.theta, workspace=ws)

        def fwd():
            xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], w.eps, w.theta,
                           workspace=ws, **sv)

        def bwd():
            xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], sv, d["dout"],
                           w.eps, w.theta, workspace=ws, **gr)

        for _ in range(warmup):
            flush.zero_()
            fwd()
            bwd()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        xt.xt_timing_reset()
        xt.xt_timing_enable(True)
        for i in range(steps):
            flush.zero_()
            fwd()
            bwd()
        torch.cuda.synchronize()
        xt.xt_timing_enable(False)
        kern = {k: round(v[0] / v[1], 5) for k, v in xt.xt_timing_query().items() if v[1]}
        if xt.xt_attn_check() != xt.XT_OK:
            raise RuntimeError(f"device error flag raised while timing {name}")
        f_ms = sum(a.elapsed_time(b) for a, b, _ in ev) / steps
        b_ms = sum(b.elapsed_time(c) for _, b, c in ev) / steps

        def rate(fl, ms):
            return fl / (ms * 1e-3) / 1e12

        res[name] = {
            "B": w.B, "S": w.S, "n_heads": w.H, "n_kv_heads": w.G, "head_dim": w.D,
            "dtype": w.dtype, "fwd_ms": f_ms, "bwd_ms": b_ms, "step_ms": f_ms + b_ms,
            "fwd_tflops": rate(w.fwd_flops, f_ms), "bwd_tflops": rate(w.bwd_flops, b_ms),
            "step_tflops": rate(w.fwd_flops + w.bwd_flops, f_ms + b_ms),
            "step_frac_of_peak": rate(w.fwd_flops + w.bwd_flops, f_ms + b_ms) / peaks["tflops"],
            "kernel_ms_per_launch": kern,
        }
        del d, ws, sv, gr
    torch.cuda.empty_cache()
    return {"steps": steps, "warmup": warmup,
            "timing": "CUDA events per fwd / bwd call on the launch stream, L2 flushed between "
                      "steps (512 MB write), inputs seeded like the headline's (seed 0)",
            "peak_tflops": peaks["tflops"], "workloads": res}


def pipelined_e2e(torch, steps, pin_in, dev_ins, compute, dev_outs, host_outs):
    """ms per end-to-end step over `steps` steps: each step copies its inputs
    from pinned host memory (pin_in) into one of two device buffer sets, runs
    compute(set) on the current stream, and copies its outputs back into pinned
    host memory. Copies run on their own streams, so step i's compute overlaps
    step i+1's inputs coming in and step i-1's outputs going out; a set is
    reused only after its previous step's outputs have left. Timed from the
    first copy in to the last copy out."""
    cs = torch.cuda.current_stream()
    hs, ds = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def run(n, timed):
        torch.cuda.synchronize()
        if timed:
            start.record(cs)
        hs.wait_stream(cs)
        ds.wait_stream(cs)
        for i in range(n):
            k = i % 2
            with torch.cuda.stream(hs):
                if i >= 2:
                    hs.wait_event(comp_done[k])
                for name, src in pin_in.items():
                    dev_ins[k][name].copy_(src, non_blocking=True)
                h2d_done[k].record(hs)
            cs.wait_event(h2d_done[k])
            if i >= 2:
                cs.wait_event(d2h_done[k])
            compute(k)
            comp_done[k].record(cs)
            with torch.cuda.stream(ds):
                ds.wait_event(comp_done[k])
                for name, dst in host_outs[k].items():
                    dst.copy_(dev_outs[k][name], non_blocking=True)
                d2h_done[k].record(ds)
        cs.wait_stream(hs)
        cs.wait_stream(ds)
        if timed:
            end.record(cs)
        torch.cuda.synchronize()

    run(2, False)   # warm: both sets once
    run(steps, True)
    return start.elapsed_time(end) / steps


def decode_bytes(w):
    """Algorithmic bytes of one decode step with every cache full: the K-hat and V
    rows of every (sequence, kv head) read once."""
    esz = 2 if w.dtype == "bf16" else 4
    return 2 * w.B * w.G * w.S * w.D * esz


def decode_oracle_sample(w):
    """The oracle on one sequence of the decode workload: every query head of the
    last position over the whole prefix (raw q, k, v; norm and RoPE inside)."""
    from causal_gqa_attention_xt_gb300.inputs import make_inputs, to_f64
    sub = w.with_(B=1)
    x = to_f64(make_inputs(sub))
    rows = [(0, h, w.S - 1) for h in range(w.H)]
    return sub, x, rows


def run_decode_oracle(sub, x, rows, threads, reps):
    """reps decode steps of one sequence each (the same synthetic sequence)."""
    import oracle
    for _ in range(reps):
        oracle.attn_fwd_rows(x["q"], x["k"], x["v"], x["gamma_q"], x["gamma_k"], sub.eps,
                             sub.theta, rows, nthreads=threads)


def decode_sample_desc(w, reps):
    return (f"{reps} sequence-steps of {w.S} cached positions each (the {w.H} query heads of "
            f"the last position, G={w.G}, D={w.D}): oracle single-row attention in fp64, "
            f"bytes counted as the GPU step's per sequence")


def decode_cpu_baseline(w, seconds_target=10.0):
    import oracle
    oracle.build()
    cores = host_cores()
    sub, x, rows = decode_oracle_sample(w)
    t0 = time.perf_counter()
    run_decode_oracle(sub, x, rows, cores, 1)
    one = max(time.perf_counter() - t0, 1e-4)
    reps = max(1, int(seconds_target / one))
    t0 = time.perf_counter()
    run_decode_oracle(sub, x, rows, cores, reps)
    dt_s = time.perf_counter() - t0
    return {"value": reps * decode_bytes(w) / w.B / dt_s / 1e9, "unit": "GB/s",
            "cores": min(cores, len(rows)), "kind": "oracle", "sample": decode_sample_desc(w, reps),
            "seconds": dt_s}


def bench_decode(args, w):
    import torch
    import torch.distributed as dist

    from causal_gqa_attention_xt_gb300 import build as xbuild
    from causal_gqa_attention_xt_gb300 import xt

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    xbuild.build()
    xt.lib()
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    seed = shard_seed(w.seed, rank)
    gen_dev = torch.Generator(device=dev).manual_seed(seed)
    gen = torch.Generator().manual_seed(seed)
    # a full cache of synthetic rows (N(0,1); the step's cost does not depend on the values)
    kc = torch.randn(w.B, w.G, w.S, w.D, generator=gen_dev, device=dev).to(dt)
    vc = torch.randn(w.B, w.G, w.S, w.D, generator=gen_dev, device=dev).to(dt)
    host = {"q": torch.randn(w.B, w.H, w.D, generator=gen).to(dt),
            "k": torch.randn(w.B, w.G, w.D, generator=gen).to(dt),
            "v": torch.randn(w.B, w.G, w.D, generator=gen).to(dt)}
    gq = (1 + 0.1 * torch.randn(w.D, generator=gen)).to(dev)
    gk = (1 + 0.1 * torch.randn(w.D, generator=gen)).to(dev)
    d = {k_: v_.to(dev) for k_, v_ in host.items()}
    pos = torch.full((w.B,), w.S - 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty(w.B, w.H, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, xt.xt_attn_decode_workspace_bytes(w.B, w.S, w.H, w.G, w.D,
                                                                1 if w.dtype == "bf16" else 0)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        xt.xt_attn_decode(pos, d["q"], d["k"], d["v"], gq, gk, kc, vc, w.eps, w.theta, out=out,
                          lse=lse, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if xt.xt_attn_check() != xt.XT_OK:
        raise RuntimeError("device error flag raised during warm-up")
    clocks = ClockSampler(gpu_pci_id(torch))
    clocks.start()
    time.sleep(0.4)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    # per-launch kernel times for the roofline, from a second pass of K steps
    xt.xt_timing_reset()
    xt.xt_timing_enable(True)
    for i in range(args.steps):
        step()
    torch.cuda.synchronize()
    xt.xt_timing_enable(False)
    per_kernel = xt.xt_timing_query()
    clk = clocks.stop()
    if xt.xt_attn_check() != xt.XT_OK:
        raise RuntimeError("device error flag raised during the timed steps")
    step_ms = reduce_max([sum(a.elapsed_time(b) for a, b in ev) / args.steps], dev)[0]

    # end to end: the new rows in from pinned host memory, out and lse back
    pin = {k_: v_.pin_memory() for k_, v_ in host.items()}
    h2d = sum(v_.numel() * v_.element_size() for v_ in pin.values())
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

    d1 = {k_: v_.clone() for k_, v_ in d.items()}
    sets = [(d, out, lse), (d1, torch.empty_like(out), torch.empty_like(lse))]
    host_outs = [dict(out=torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
                      lse=torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True))
                 for _ in range(2)]

    def compute(k):
        dd, o_, l_ = sets[k]
        xt.xt_attn_decode(pos, dd["q"], dd["k"], dd["v"], gq, gk, kc, vc, w.eps, w.theta, out=o_,
                          lse=l_, workspace=ws)

    e2e_ms = reduce_max([pipelined_e2e(torch, args.steps, pin, [s_[0] for s_ in sets], compute,
                                       [dict(out=s_[1], lse=s_[2]) for s_ in sets],
                                       host_outs)], dev)[0]
    if xt.xt_attn_check() != xt.XT_OK:
        raise RuntimeError("device error flag raised during the end-to-end steps")

    nbytes = decode_bytes(w)
    value = world * nbytes / (step_ms * 1e-3) / 1e9
    peaks = load_peaks()
    roofline = None
    if "decode_attn" in per_kernel:
        tot_ms, n = per_kernel["decode_attn"]
        ach = nbytes / (tot_ms / n * 1e-3) / 1e9
        roofline = {"kernel": "decode_attn", "bound": "hbm", "achieved": ach,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                    "peak_source": f"{peaks['source']} copy", "traffic": None,
                    "avg_launch_ms": tot_ms / n}
        traffic_file = os.path.join(ROOT, "profiles", "traffic.json")
        try:
            with open(traffic_file) as f:
                ent = json.load(f).get("decode_attn", {})
            if ent.get("workload") == w.name and ent.get("source_hash") == source_hash("decode_attn"):
                roofline["traffic"] = ent.get("bytes_per_launch")
        except (OSError, ValueError):
            pass
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "sequences": w.B, "cache_rows": w.S, "position": w.S - 1,
                   "n_heads": w.H, "n_kv_heads": w.G, "head_dim": w.D, "theta": w.theta,
                   "eps": w.eps, "cache_bytes_read_per_step": nbytes,
                   "l2": "not flushed: the caches are larger than L2",
                   "inputs": "N(0,1) cache rows and new rows, gammas 1+0.1*N(0,1), seed 0+rank"},
        "tokens_per_s": world * w.B / (step_ms * 1e-3),
        "roofline": roofline,
        "kernels": {k_: {"total_ms": v_[0], "launches": v_[1]} for k_, v_ in per_kernel.items()},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sum(n for _, n in per_kernel.values()),
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(w)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def bench_decode_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = host_cores()
    sub, x, rows = decode_oracle_sample(w)
    reps = 8   # sequence-steps per timed step, about half a second of oracle work
    for _ in range(args.warmup):
        run_decode_oracle(sub, x, rows, cores, reps)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run_decode_oracle(sub, x, rows, cores, reps)
        times.append(time.perf_counter() - t0)
    value = reps * decode_bytes(w) / w.B * len(times) / sum(times) / 1e9
    desc = decode_sample_desc(w, reps)
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sequences": w.B, "cache_rows": w.S, "n_heads": w.H,
                   "n_kv_heads": w.G, "head_dim": w.D, "sample_per_step": desc},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": min(cores, len(rows)),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def profile_run(w):
    """One warm-up and one measured-shape fwd+bwd step (launch order: prologue,
    fwd, bwd_pre, dkdv, dq, epilogue, dgamma_reduce, twice), for ncu."""
    import torch

    from causal_gqa_attention_xt_gb300 import build as xbuild
    from causal_gqa_attention_xt_gb300 import xt
    from causal_gqa_attention_xt_gb300.inputs import make_inputs
    xbuild.build()
    d = {k: v.cuda() for k, v in make_inputs(w).items()}
    for _ in range(2):
        f = xt.xt_attn_fwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], w.eps, w.theta)
        xt.xt_attn_bwd(d["q"], d["k"], d["v"], d["gamma_q"], d["gamma_k"], f, d["dout"], w.eps,
                       w.theta)
    torch.cuda.synchronize()
    st = xt.xt_attn_check()
    print(f"profile run {w.name}: status {xt.xt_status_str(st)}")
    return 0 if st == xt.XT_OK else 1


# The sources each timed kernel is built from (its file, the shared device
# helpers): stored ncu traffic stays valid while these are unchanged.
KERNEL_SOURCES = {
    "fwd_tcgen05_bf16": ["xt_fwd_tc.cu"],
    "bwd_dkdv_tcgen05_bf16": ["xt_bwd_tc.cu"],
    "bwd_dq_tcgen05_bf16": ["xt_bwd_tc.cu"],
    "prologue_qknorm_rope": ["xt_normrope.cu", "xt_rope.cuh"],
    "bwd_pre_dlt": ["xt_normrope.cu", "xt_rope.cuh"],
    "bwd_epilogue_rope_norm": ["xt_normrope.cu", "xt_rope.cuh"],
    "decode_attn": ["xt_decode.cu", "xt_rope.cuh"],
}
SHARED_DEVICE_SOURCES = ["xt_common.cuh", "xt_tc.cuh"]


def code_text(src: str) -> str:
    """CUDA source without its comments and blank lines: what source_hash covers,
    so that comment edits keep stored traffic valid. (// inside a string literal
    does not occur in these files.)"""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in src.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def source_hash(kernel: str, read=None) -> str:
    """Hash of the code of a kernel's CUDA sources (comments left out), to tie
    stored ncu traffic to the code it measured. read(name) -> text overrides
    reading the working tree's files."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel] + SHARED_DEVICE_SOURCES:
        if read is not None:
            text = read(name)
        else:
            with open(os.path.join(ROOT, "causal_gqa_attention_xt_gb300", "csrc", name)) as f:
                text = f.read()
        h.update(code_text(text).encode())
    return h.hexdigest()[:16]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["train", "decode", "varlen"], default="train",
                    help="train: fwd+bwd step (the headline); decode: one KV-cache decode step; "
                         "varlen: fwd+bwd over a packed batch of unequal samples")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload timings that follow the headline (train mode)")
    ap.add_argument("--ref-seq", type=int, default=1024,
                    help="sequence length of the oracle's per-step sample (reference arm)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="time the CPU oracle on every configured workload (host cores only)")
    ap.add_argument("--profile-run", action="store_true",
                    help="one warm-up and one fwd+bwd step, no timing (for ncu captures)")
    args = ap.parse_args(argv)
    if args.oracle_configs:
        return oracle_configs()
    from causal_gqa_attention_xt_gb300.inputs import PACKED_WORKLOADS, WORKLOADS
    if args.mode == "varlen":
        w = PACKED_WORKLOADS[args.workload or VARLEN_WORKLOAD]
        if args.warmup < 3:
            ap.error("--warmup must be >= 3")
        if args.impl == "reference":
            return bench_reference(args, longest_sample(w), metric=VARLEN_METRIC,
                                   workload_name=w.name)
        return bench_ours(args, w)
    w = WORKLOADS[args.workload or (DECODE_WORKLOAD if args.mode == "decode" else DEFAULT_WORKLOAD)]
    if args.batch is not None:
        w = w.with_(B=args.batch, name=f"{w.name}_B{args.batch}")
    if args.profile_run:
        return profile_run(w)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.mode == "decode":
        return bench_decode_reference(args, w) if args.impl == "reference" else bench_decode(args, w)
    if args.impl == "reference":
        return bench_reference(args, w)
    return bench_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
