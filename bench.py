#!/usr/bin/env python3
"""Benchmark of the selective KV-cache refresh (packed, layer-major) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama8b]

One step = one whole refresh: kvr_select (upload and pack the 282 selected
positions, gather their embedding rows) + all 32 layers through kvr_refresh
+ the metadata commit, on the Llama-3-8B-shaped workload (N = 7680 after a
512-token deletion, 5 % of the 5632-token retained suffix in units of 32-64
tokens).  Weights (14 GB) and cache stay resident; every step streams all
weights, far more than the 129 MB L2, so no explicit flush is needed.

Prints ONE JSON line (rank 0).  With --gpus N > 1 (torchrun) every rank runs
an independent replica of the same refresh (one sequence does not shard
without tensor parallelism); `value` is the total over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "refreshed tokens/sec & refresh latency/edit; HBM and tensor-pipe % of peak"
UNIT = "tokens/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p:
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "selective_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_class, sha):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    if it was taken on the current source (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        m = re.match(r"\s*(\S+)\s+sha=(\S+)\s+dram_bytes_per_launch=(\d+)", line)
        if m and m.group(1) == kernel_class and m.group(2) == sha:
            return int(m.group(3))
    return None


# per-kernel algorithmic work at the workload: bytes and FLOPs per launch from the model shape
def algorithmic(shape, R, M_pairs_per_head, u_max):
    """Algorithmic FLOPs and bytes per launch of each kernel class for R packed
    rows: a projection reads its weights once and the rows once and writes
    fp32 partials; attention reads each K/V row up to the last selected
    position once per K/V head, reads Q and writes O, and spends
    4 d_h FLOPs per causal query-key pair per query head."""
    d, Hq, Hkv, dh, F = shape.d_model, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim
    qkv = (Hq + 2 * Hkv) * dh

    def gemm(n_out, K, out_bytes=4.0):
        return dict(flops=2.0 * R * n_out * K, bytes=2.0 * n_out * K + 2.0 * R * K + out_bytes * R * n_out)

    return {
        "gemm_qkv": gemm(qkv, d),
        "gemm_o": gemm(d, Hq * dh),
        # SwiGLU is fused: the output is silu(g) * u in bf16, half as many features
        "gemm_gate_up": gemm(2 * F, d, out_bytes=1.0),
        "gemm_down": gemm(d, F),
        "attention": dict(flops=4.0 * dh * Hq * M_pairs_per_head,
                          bytes=2.0 * 2 * Hkv * dh * (u_max + 1) + 2.0 * 2 * R * Hq * dh),
    }


def roofline_entry(kernel_class, wk, t_s, hbm_gbs, tflops, peak_source):
    """Roofline of one kernel class from its algorithmic work per call and its
    measured time per call t_s: the bound is the larger of the HBM time
    (bytes / copy peak) and the tensor time (FLOPs / burst bf16 peak), and the
    fraction is that bound's time over the measured time.  Achieved HBM GB/s
    and tensor TFLOP/s are reported beside it."""
    t_hbm = wk["bytes"] / (hbm_gbs * 1e9)
    t_tc = wk["flops"] / (tflops * 1e12)
    gbs = wk["bytes"] / t_s / 1e9
    tfs = wk["flops"] / t_s / 1e12
    if t_hbm >= t_tc:
        e = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_gbs, "unit": "GB/s", "frac": round(t_hbm / t_s, 4)}
    else:
        e = {"bound": "tensor", "achieved": round(tfs, 1), "peak": tflops, "unit": "TFLOP/s",
             "frac": round(t_tc / t_s, 4)}
    e.update({"kernel": kernel_class, "avg_call_us": round(t_s * 1e6, 2),
              "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_gbs, 4),
              "tensor_tflops": round(tfs, 1), "tensor_frac": round(tfs / tflops, 4),
              "algorithmic_bytes": int(wk["bytes"]), "algorithmic_flops": int(wk["flops"]),
              "peak_source": f"{peak_source} (copy {hbm_gbs} GB/s, burst bf16 {tflops} TFLOP/s; max of the two bounds)",
              "traffic": ncu_traffic(kernel_class, kernel_source_sha(source_files(kernel_class)))})
    return e


def source_files(kernel_class):
    if kernel_class.startswith("gemm"):
        return ["gemm.cu", "kvr_internal.h", "ptx.cuh"]
    if kernel_class == "attention":
        return sorted(f for f in os.listdir(os.path.join(ROOT, "selective_kv_cache_gb300", "csrc"))
                      if f.startswith("attn") or f in ("ptx.cuh", "kvr_internal.h"))
    return ["elementwise.cu", "kvr_internal.h"]


def job_throughput(local_time, units_per_rank, world, device=None):
    """Whole-job throughput of N independent replicas: the slowest rank's
    time (max over ranks) bounds the job, and every rank processed
    units_per_rank units.  Works on any process-group backend (NCCL on GPUs,
    gloo on CPU); returns (max time, units per second)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_time)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    t_max = float(t.item())
    return t_max, units_per_rank * world / t_max


def sharded_throughput(local_time, local_units, world, device=None):
    """Whole-job throughput of a sharded run: the ranks hold different shares
    of one job, so the job's time is the slowest rank's (max over ranks) and
    its work is the sum of the ranks' units.  Any process-group backend
    (NCCL on GPUs, gloo on CPU); returns (max time, total units, units per
    second)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_time)], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
    t_max, total = float(t.item()), float(u.item())
    return t_max, total, total / t_max


def gather_shards(lo, hi, world, device=None):
    """Every rank's sequence shard [lo, hi), in rank order."""
    import torch
    import torch.distributed as dist

    mine = torch.tensor([lo, hi], dtype=torch.int64, device=device)
    if world == 1:
        return [(lo, hi)]
    parts = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine)
    return [tuple(int(x) for x in p.tolist()) for p in parts]


def run_drift(args, w, world, rank):
    """The adapter-drift repair (CacheReforge, Bounded Recovery) sharded by
    sequence: the batch's sequences are independent (own cache, selection and
    boundary states), so rank r owns sequences shard_sequences(batch, N, r)
    with a replica of the weights, and no data crosses between ranks.  One
    step = one whole repair of the rank's sequences (kvr_refresh_range: the
    selected rows through layers [0, r0), the whole suffix through [r0, r1),
    the selected rows through the rest, the commit).  value = row-layers of
    all ranks / the slowest rank's time (strong scaling: the batch is fixed)."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from selective_kv_cache_gb300 import kvr
    from selective_kv_cache_gb300.harness import Setup, shard_sequences

    lo, hi = shard_sequences(w.batch, world, rank)
    if hi <= lo:
        raise SystemExit(f"{world} ranks for a batch of {w.batch}: rank {rank} would own no sequence")
    s = Setup(w, seqs=(lo, hi))
    m = w.model
    g = torch.Generator(device="cuda").manual_seed(w.seed(11))
    boundary = torch.randn((w.batch, w.capacity, m.d_model), device="cuda", generator=g).to(m.torch_dtype)
    boundary = boundary[lo:hi].contiguous()
    r0, r1 = w.range_layers
    stream = torch.cuda.current_stream()

    def step():
        s.refresh_range(boundary, r0, r1, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    s.sync()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with Clocks(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    s.sync()
    S = w.n_tokens - w.suffix_start
    rows = int(np.sum(s.counts))
    units = rows * (m.n_layers - (r1 - r0)) + (hi - lo) * S * (r1 - r0)
    t_max, total, value = sharded_throughput(ms / 1e3, units * args.steps, world, device="cuda")

    # end to end with host buffers: token ids in, refreshed rows out
    ids_host = s.ids.cpu().pin_memory()
    out_host = torch.empty((rows, m.d_model), dtype=s.hidden.dtype).pin_memory()
    h2d = ids_host.numel() * ids_host.element_size() + s.pos_host.nbytes + s.counts.nbytes
    d2h = out_host.numel() * out_host.element_size()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.ids.copy_(ids_host, non_blocking=True)
        step()
        out_host.copy_(s.hidden[:rows], non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    _, _, e2e_value = sharded_throughput(e2e_s, units * args.steps, world, device="cuda")
    shards = gather_shards(lo, hi, world, device="cuda")
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "row-layers/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random weights, token ids, embeddings, boundary states and stale cache)",
        "config": {"workload": describe(w, int(w.n_select * w.batch)) +
                   f"; layers [{r0},{r1}) over all {w.batch * S} suffix rows",
                   "layers": m.n_layers, "batch": w.batch,
                   "parallelism": f"sequence shards over {world} rank(s), weights replicated, no exchange"},
        "shards": shards,
        "latency": {"repair_ms": round(t_max * 1e3 / args.steps, 3)},
        "e2e": {"value": round(e2e_value, 1), "unit": "row-layers/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    s.close()
    if world > 1:
        dist.destroy_process_group()


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from selective_kv_cache_gb300 import kvr, workloads as wl
    from selective_kv_cache_gb300.harness import Setup

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    w = wl.WORKLOADS[args.workload]
    if w.range_layers:
        return run_drift(args, w, world, rank)
    s = Setup(w)
    m = w.model
    stream = torch.cuda.current_stream()

    def step():
        s.select(stream=stream)
        s.refresh(stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    s.sync()

    # ---- timed region: device-resident inputs
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with Clocks(local_rank) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    s.sync()
    rows = s.n_rows
    sec_total, value = job_throughput(ms / 1e3, rows * args.steps, world, device="cuda")
    ms_total = sec_total * 1e3

    # ---- per-kernel breakdown: the same K steps again with CUDA events around every launch
    kvr.kvr_profile_read(s.handle)
    kvr.kvr_profile_enable(s.handle, True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = kvr.kvr_profile_read(s.handle)
    kvr.kvr_profile_enable(s.handle, False)
    launches_per_step = sum(n for n, _ in prof.values()) / args.steps

    # ---- end to end through the C ABI with host buffers: token ids in, refreshed rows out
    ids_host = s.ids.cpu().pin_memory()
    out_host = torch.empty(s.hidden.shape, dtype=s.hidden.dtype).pin_memory()
    h2d = ids_host.numel() * ids_host.element_size() + s.pos_host.nbytes + s.counts.nbytes
    d2h = out_host.numel() * out_host.element_size()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.ids.copy_(ids_host, non_blocking=True)
        step()
        out_host.copy_(s.hidden, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    _, e2e_value = job_throughput(e2e_s, rows * args.steps, world, device="cuda")

    # ---- rooflines: every projection class and the attention, and the dominant kernel
    hbm, tf_burst, tf_sust, src = peaks()
    per_kernel = {k: (n, v) for k, (n, v) in prof.items() if n}
    U = np.sort(np.concatenate(s.positions))
    M = float(np.sum(U + 1))
    work = algorithmic(m, rows, M, int(U.max()))
    roofs = {}
    for k, wk in work.items():
        if k not in per_kernel:
            continue
        calls = args.steps * m.n_layers          # one call per layer and step
        roofs[k] = roofline_entry(k, wk, per_kernel[k][1] / calls / 1e3, hbm, tf_burst, src)
    dom = max(per_kernel, key=lambda k: per_kernel[k][1])
    roof = dict(roofs[dom]) if dom in roofs else None
    breakdown = {k: {"launches_per_step": n / args.steps, "us_per_step": round(v * 1e3 / args.steps, 1)}
                 for k, (n, v) in per_kernel.items()}

    # ---- packed vs interval-wise on the fragmented workload (same model and cache)
    cmp = None
    if not args.no_compare and args.workload == "llama8b":
        cmp = compare_schedules(s, args)

    # ---- Shift of the same edit (the step before the refresh), on its own cache,
    # and the Semantic-Unit Refresh selection that picks positions for it
    shift = sur = None
    if args.workload == "llama8b":
        shift = measure_shift(w, hbm)
        sur = measure_sur(s, hbm)

    # ---- the pages' matched-work benchmark at their shape (Qwen3-8B-like)
    mw = None
    if args.workload == "llama8b" and not args.no_matched:
        mw = matched_work()

    # ---- the other configurations (block seams, adapter drift)
    oc = None
    if not args.no_other_configs and args.workload == "llama8b":
        oc = other_configs(hbm, tf_burst, src)

    # ---- CPU oracle baseline: one whole refresh of the same workload (rank 0 only)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(s, w)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded random weights, "
        "token ids, embeddings and stale cache)",
        "config": workload_config(w, rows, world),
        "latency": {"refresh_ms": round(ms_total / args.steps, 4),
                    "per_layer_us": round(ms_total / args.steps / m.n_layers * 1e3, 2)},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "roofline": roof,
        "rooflines": roofs,
        "kernels": breakdown,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "packed_vs_interval": cmp,
        "shift": shift,
        "sur_select": sur,
        "matched_work": mw,
        "other_configs": oc,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    s.close()
    if world > 1:
        dist.destroy_process_group()


def workload_config(w, rows, world):
    """The `config` object of the JSON line: what the workload is (both arms
    print the same one)."""
    m = w.model
    return {"workload": describe(w, rows), "rows": rows, "n_tokens": w.n_tokens, "layers": m.n_layers,
            "l2": f"no flush: each step streams {weight_gb(m):.1f} GB of weights (> 129 MB L2)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


FAMILY = {(4096, 32, 8, 14336): "Llama-3-8B-shaped", (3584, 28, 4, 18944): "Qwen2.5-7B-shaped",
          (1536, 12, 2, 8960): "Qwen2.5-1.5B-shaped", (4096, 32, 8, 12288): "Qwen3-8B-shaped"}


def describe(w, rows):
    """The workload in words: model shape, cache, selection."""
    m = w.model
    kind = {"units": "in units of 32-64", "isolated": "isolated", "seams": "in seam windows",
            "matched": "in matched intervals"}.get(w.selection, w.selection)
    fam = FAMILY.get((m.d_model, m.n_q_heads, m.n_kv_heads, m.ffn_dim), "random-init")
    return (f"{w.name}: {fam} stack, {m.n_layers} L, d {m.d_model}, {m.n_q_heads}/{m.n_kv_heads} heads x {m.head_dim}, "
            f"FFN {m.ffn_dim}, RoPE theta {m.rope_theta:g}{', q/k/v bias' if m.qkv_bias else ''}, "
            f"batch {w.batch}, N={w.n_tokens}, suffix [{w.suffix_start},{w.n_tokens}), "
            f"{rows} refreshed positions {kind}, alpha {w.alpha:g}, beta {w.beta:g}")


def weight_gb(m):
    """Weight bytes of the whole stack in GB."""
    per_layer = (m.qkv_out + m.n_q_heads * m.head_dim) * m.d_model + 3 * m.ffn_dim * m.d_model
    return per_layer * m.n_layers * (4 if m.dtype == "f32" else 2) / 1e9


def other_configs(hbm, tflops, peak_source):
    """The block-seam repair (Qwen2.5-7B shape, 896 seam rows over 8
    independently prefilled blocks of 2048, alpha -2, beta -4) and the
    adapter-drift repair (Qwen2.5-1.5B shape, batch 4 x 32768, layers 10-14
    over the whole 24576-token affected suffix from stored boundary states,
    492 isolated rows per sequence elsewhere): CUDA events around select +
    refresh on device-resident inputs, 5 and 3 repetitions after 2 and 1
    warm-ups; then one more pass with events around every launch for the
    per-kernel breakdown, and for the seam repair the rooflines of its
    projections and of the biased attention."""
    import numpy as np
    import torch

    from selective_kv_cache_gb300 import kvr, workloads as wl
    from selective_kv_cache_gb300.harness import Setup

    def timed(fn, reps, warm):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def profiled(s, fn, reps):
        kvr.kvr_profile_read(s.handle)
        kvr.kvr_profile_enable(s.handle, True)
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        prof = kvr.kvr_profile_read(s.handle)
        kvr.kvr_profile_enable(s.handle, False)
        return {k: (n, v) for k, (n, v) in prof.items() if n}

    out = {}
    w = wl.WORKLOADS["qwen7b_seam"]
    s = Setup(w)
    rows, _ = s.select()

    def seam():
        s.select()
        s.refresh()

    ms = timed(seam, 5, 2)
    prof = profiled(s, seam, 3)
    s.sync()
    m = w.model
    U = np.sort(np.concatenate(s.positions))
    work = algorithmic(m, rows, float(np.sum(U + 1)), int(U.max()))
    roofs = {k: roofline_entry(k, wk, prof[k][1] / (3 * m.n_layers) / 1e3, hbm, tflops, peak_source)
             for k, wk in work.items() if k in prof}
    for e in roofs.values():
        e["traffic"] = None      # the committed DRAM records are for the Llama-shaped workload
    out["qwen7b_seam"] = {"workload": describe(w, rows), "ms_per_refresh": round(ms, 3),
                          "refreshed_tokens_per_s": round(rows / ms * 1e3, 1),
                          "per_layer_us": round(ms / m.n_layers * 1e3, 2),
                          "rooflines": roofs,
                          "kernels": {k: {"launches_per_refresh": n / 3, "us_per_refresh": round(v * 1e3 / 3, 1)}
                                      for k, (n, v) in prof.items()}}
    s.close()
    del s
    torch.cuda.empty_cache()
    w = wl.WORKLOADS["qwen1p5b_drift"]
    s = Setup(w)
    g = torch.Generator(device="cuda").manual_seed(w.seed(11))
    boundary = torch.randn((w.batch, w.capacity, w.model.d_model), device="cuda", generator=g).to(
        w.model.torch_dtype)
    r0, r1 = w.range_layers
    drift = lambda: s.refresh_range(boundary, r0, r1)
    ms = timed(drift, 3, 1)
    prof = profiled(s, drift, 1)
    s.sync()
    rows = int(np.sum(s.counts))
    full = w.batch * (w.n_tokens - w.suffix_start)
    row_layers = rows * (w.model.n_layers - (r1 - r0)) + full * (r1 - r0)
    out["qwen1p5b_drift"] = {"workload": describe(w, rows) + f"; layers [{r0},{r1}) over all {full} suffix rows",
                             "ms_per_repair": round(ms, 2), "row_layers_per_s": round(row_layers / ms * 1e3, 1),
                             "kernels": {k: {"launches_per_repair": n, "us_per_repair": round(v * 1e3, 1)}
                                         for k, (n, v) in prof.items()}}
    s.close()
    del s
    torch.cuda.empty_cache()
    return out


def measure_shift(w, hbm_peak, reps=10):
    """Shift for the Llama-shaped edit: an 8192-token cache (32 layers, 8 K/V
    heads x 128, bf16) loses the 512-token span at 2048, so 5632 rows per
    (layer, head) move down with their keys re-rotated.  One fresh cache per
    repetition (the shift changes the cache's length); CUDA events around the
    kvr_shift call.  The cache (1.07 GB) is larger than L2."""
    import torch

    from selective_kv_cache_gb300 import kvr

    m = w.model
    cap, start, d = 8192, 2048, 512
    shape = (1, m.n_layers, m.n_kv_heads, cap, m.head_dim)
    K = torch.randn(shape, device="cuda").to(torch.bfloat16)
    V = torch.randn(shape, device="cuda").to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    times = []
    for i in range(reps + 2):
        h = kvr.kvr_create_cache(kvr.model_desc(m), 1, cap, K, V, cap, start)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kvr.kvr_shift(h, start, d, stream=stream)
        e1.record(stream)
        kvr.kvr_sync_status(h, stream)
        kvr.kvr_destroy_cache(h)
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    moved = cap - start - d
    nbytes = 2 * 2 * m.n_layers * m.n_kv_heads * moved * m.head_dim * 2   # K and V, read and write
    us = sorted(times)[len(times) // 2] * 1e3
    gbs = nbytes / (us / 1e6) / 1e9
    return {"workload": f"delete [{start},{start + d}) of a {cap}-token Llama-3-8B-shaped cache "
                        f"({m.n_layers} L x {m.n_kv_heads} K/V heads x {m.head_dim}, bf16)",
            "us_median": round(us, 1), "bytes": int(nbytes), "achieved_gbs": round(gbs, 1), "peak_gbs": hbm_peak,
            "frac": round(gbs / hbm_peak, 4), "reps": reps}


def measure_sur(s, hbm_peak, reps=10):
    """Semantic-Unit Refresh selection for the same edit: the 5632-token
    retained suffix of the timed workload, a 64-token query, units of 8-128
    tokens, the 5 % budget; CUDA events around kvr_sur_select.  Its
    algorithmic floor is reading the suffix's embedding rows once (2 S d
    bytes); the fp32 scoring contraction (2 S Q d FLOPs, on the tensor cores
    as three exact bf16 terms of the query) is a few microseconds beside it."""
    import numpy as np
    import torch

    from selective_kv_cache_gb300 import kvr, workloads as wl

    w = s.w
    S = w.n_tokens - w.suffix_start
    Q = 64
    d = w.model.d_model
    sids = s.ids[0, w.suffix_start:w.n_tokens].contiguous()
    qids = torch.from_numpy(wl.make_query_ids(w.model.vocab, Q, 21, sids.cpu().numpy(), overlap=4)).cuda()
    bounds = torch.from_numpy(wl.make_unit_bounds(S, 22)).cuda()
    ws = torch.empty(kvr.kvr_sur_workspace_bytes(S, Q, d, bounds.numel() - 1), dtype=torch.uint8, device="cuda")
    pos = torch.empty(S, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    times = []
    for i in range(reps + 3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        B = kvr.kvr_sur_select(s.embed, sids, qids, bounds, 5, w.suffix_start, ws, pos, stream=stream)
        e1.record(stream)
        kvr.kvr_sur_status(ws, stream)
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    us = float(np.median(times)) * 1e3
    nbytes = 2.0 * S * d
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"{S}-token suffix, {Q}-token query, {bounds.numel() - 1} units of 8-128 tokens, "
                        f"{w.model.vocab} x {d} bf16 embeddings, 5 % budget ({B} positions)",
            "us_median": round(us, 1), "bound": "hbm", "bytes": int(nbytes), "achieved_gbs": round(gbs, 1),
            "peak_gbs": hbm_peak, "frac": round(gbs / hbm_peak, 4),
            "fp32_scoring_tflops": round(2.0 * S * Q * d / (us * 1e-6) / 1e12, 2)}


# Table 18 of "Budgeted KV-Cache Repair for Evolving Contexts" (Sec. 13.3):
# Qwen3-8B on one H100, B = 64, medians in ms.  Context only (other hardware).
PAGES_TABLE18_H100 = {(2048, 1): (31.465, 32.389), (2048, 4): (121.456, 32.470), (2048, 16): (485.378, 32.775),
                      (8192, 1): (32.571, 33.372), (8192, 4): (120.679, 32.235), (8192, 16): (494.826, 33.375)}


def matched_work():
    """The pages' matched-work benchmark at their shape (Sec. 13.3, Table 18):
    a Qwen3-8B-shaped stack (36 layers, 4096, 32/8 heads x 128, FFN 12288),
    a random-token prompt of N + 8 tokens that loses 8 tokens at 64 (Shift,
    untimed), B = 64 refreshed positions in R = 1, 4, 16 intervals with the
    same M(U).  Timed like the pages: synchronised wall time per refresh,
    host planning and upload included, medians of 20 after 10 warm-ups for the
    packed refresh; the interval-wise comparator (the pages' direct
    sequential control) takes 10 after 3."""
    import dataclasses

    import numpy as np
    import torch

    from selective_kv_cache_gb300 import kvr, workloads as wl
    from selective_kv_cache_gb300.harness import Setup

    w0 = wl.WORKLOADS["qwen3_matched"]
    layers = wl.make_layer_weights(w0, "cuda")
    embed = wl.make_embeddings(w0, "cuda")

    def wall(fn, warm, reps):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append((time.perf_counter() - t0) * 1e3)
        return float(np.median(ts))

    rows = []
    for N in (2048, 8192):
        w = dataclasses.replace(w0, capacity=N + 8, n_tokens=N + 8, suffix_start=64)
        for R in (1, 4, 16):
            pos = wl.matched_positions(N, 64, R)
            s = Setup(w, weights=layers, positions=[pos], embed=embed)
            kvr.kvr_shift(s.handle, 64, 8)            # the edit: 8 tokens deleted at 64
            assert kvr.kvr_cache_info(s.handle) == (N, 64)
            m_u = int(np.sum(pos.astype(np.int64) + 1))

            def packed():
                s.select()
                s.refresh()

            t_p = wall(packed, 10, 20)
            t_i = wall(lambda: s.refresh_interval_wise(), 3, 10)
            s.sync()
            s.close()
            seq_h100, custom_h100 = PAGES_TABLE18_H100[(N, R)]
            rows.append({"N": N, "R": R, "B": 64, "M_U": m_u, "packed_ms": round(t_p, 3),
                         "interval_wise_ms": round(t_i, 3), "speedup": round(t_i / t_p, 2),
                         "pages_h100_direct_seq_ms": seq_h100, "pages_h100_custom_ms": custom_h100})
    del layers, embed
    torch.cuda.empty_cache()
    return {"workload": "Qwen3-8B-shaped stack (36 L, d 4096, 32/8 heads x 128, FFN 12288, bf16, Q/K RMSNorm), "
                        "B = 64, 8 tokens deleted at 64, synchronised wall time with host planning",
            "rows": rows}


def compare_schedules(s1, args):
    """The fragmented workload (282 isolated positions of the same 5632-token
    suffix, same model and cache): layer-major packed refresh against the
    interval-major schedule, CUDA events around whole refreshes."""
    import torch

    from selective_kv_cache_gb300 import workloads as wl
    from selective_kv_cache_gb300.harness import Setup

    w = wl.WORKLOADS["llama8b_frag"]
    s = Setup(w, weights=s1.layers, cache=(s1.K, s1.V))
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def packed():
        s.select(stream=stream)
        s.refresh(stream=stream)

    for _ in range(args.warmup):
        packed()
    t_packed = timed(packed, args.steps)
    n_iv = s.refresh_interval_wise(stream=stream)   # warm-up
    s.sync()
    t_iv = timed(lambda: s.refresh_interval_wise(stream=stream), max(1, min(2, args.steps)))
    s.sync()
    s.close()
    return {"workload": f"{w.name}: same model, N={w.n_tokens}, {w.n_select} isolated positions in "
                        f"[{w.suffix_start},{w.n_tokens}) ({n_iv} intervals)",
            "packed_ms": round(t_packed, 3), "interval_wise_ms": round(t_iv, 3),
            "speedup": round(t_iv / t_packed, 2), "intervals": n_iv,
            "packed_tokens_per_s": round(w.n_select / (t_packed / 1e3), 1)}


class _TimedWeights:
    """Per-layer float64 weights for the oracle, converted from the device
    tensors when the oracle asks for a layer; the conversion (input
    preparation, not the oracle's work) is timed apart."""

    def __init__(self, layers):
        self.layers = layers
        self.convert_s = 0.0

    def __len__(self):
        return len(self.layers)

    def __getitem__(self, l):
        import torch
        t0 = time.perf_counter()
        d = {k: (v.to(torch.float64).cpu().numpy() if v is not None else None) for k, v in self.layers[l].items()}
        self.convert_s += time.perf_counter() - t0
        return d


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def _oracle_inputs(s, w):
    """Host float64 inputs of the oracle for sequence 0 of a Setup: sorted
    positions, per-position layer-0 rows, and the layer bias."""
    import numpy as np
    import torch

    import oracle

    U = oracle.sorted_positions(s.positions[0])
    ids = s.ids[0].cpu().numpy()
    X_src = np.zeros((w.capacity, w.model.d_model))
    X_src[U] = s.embed[torch.from_numpy(ids[U].astype(np.int64)).to(s.embed.device)].to(torch.float64).cpu().numpy()
    return U, X_src


def cpu_baseline(s, w):
    """The float64 oracle as it stands, timed end to end on the host cores:
    one whole refresh of the same workload (every layer, all selected rows,
    write-back into its own copy of the cache).  The bf16 -> float64
    conversion of the weights is left out of the time."""
    import numpy as np
    import torch

    import oracle

    spec = oracle.Spec.of(w.model)
    U, X_src = _oracle_inputs(s, w)
    K = s.K[0].to(torch.float64).cpu().numpy()
    V = s.V[0].to(torch.float64).cpu().numpy()
    W = _TimedWeights(s.layers)
    t0 = time.perf_counter()
    oracle.refresh_packed(spec, W, K, V, s.local_mask[0], s.sink_mask[0], U, X_src, w.alpha, w.beta)
    dt = time.perf_counter() - t0 - W.convert_s
    return {"value": round(len(U) / dt, 3), "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"one whole refresh: all {w.model.n_layers} layers for all {len(U)} rows in float64 numpy, "
                      f"end to end ({dt:.1f} s; the {W.convert_s:.1f} s of weight conversion to float64 left out)"}


def run_reference(args):
    """Reference arm: the CPU oracle, timed on the host cores.  One step is
    one layer of the refresh for all selected rows (the float64 oracle's
    layer_rows, with the write-back into that layer's cache); consecutive
    steps walk the layers in order, each taking the rows the previous step
    produced, so every L consecutive steps are one whole refresh.  Per-step
    inputs (that layer's weights and cache converted to float64) are
    prepared outside the step's time.  value = rows / (L x mean step time)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from selective_kv_cache_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"

    class S:
        pass

    s = S()
    s.layers = wl.make_layer_weights(w, dev)
    s.K, s.V = wl.make_random_cache(w, dev)
    s.embed = wl.make_embeddings(w, dev)
    s.ids = wl.make_token_ids(w, dev)
    s.positions = wl.make_positions(w)
    s.local_mask, s.sink_mask = wl.make_metadata(w)
    spec = oracle.Spec.of(w.model)
    U, X_src = _oracle_inputs(s, w)
    sel = np.zeros(w.capacity, bool)
    sel[U] = True
    loc, snk = oracle.effective_masks(s.local_mask[0], s.sink_mask[0], sel)
    bias = w.alpha * loc + w.beta * snk
    X = oracle.round_store(X_src[U], spec.dtype)
    L = w.model.n_layers
    W = _TimedWeights(s.layers)
    times = []
    for i in range(args.warmup + args.steps):
        l = i % L
        Wl = W[l]
        Kl = s.K[0, l].to(torch.float64).cpu().numpy()
        Vl = s.V[0, l].to(torch.float64).cpu().numpy()
        t0 = time.perf_counter()
        X = oracle.layer_rows(spec, Wl, X, Kl, Vl, U, bias)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    step_s = sum(times) / len(times)
    v = round(len(U) / (L * step_s), 3)
    rows = len(U)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded random weights, "
        "token ids, embeddings and stale cache)",
        "config": workload_config(w, rows, 1),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": f"one step = one layer of the refresh for all {rows} rows in float64 numpy "
                                   f"(layers walked in order, each step's rows from the previous one); "
                                   f"{args.steps} timed steps after {args.warmup}, value = rows / "
                                   f"({L} x mean step time)"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-compare", action="store_true", help="skip the packed vs interval-wise comparison")
    ap.add_argument("--no-matched", action="store_true", help="skip the matched-work benchmark (Qwen3-8B shape)")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the block-seam and adapter-drift repairs (key other_configs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
