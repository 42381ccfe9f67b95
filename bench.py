#!/usr/bin/env python3
"""Benchmark of the paged-KV-cache hot path on GB300 (one JSON line on rank 0).

Default workload: the full decode step at batch 256 -- pa_reshape_and_cache of 256 new
K/V rows (bf16, 8 KV heads x 128, 10% of slots padded with -1) followed by pa_decode
(16 q / 8 KV heads, block size 16, context lengths uniform in [100, 2048]).  A "step" is
that write plus that decode over resident inputs.

  value   = algorithmic bytes of the step (K/V read over all contexts + q + out + block
            tables + context lengths, plus the write's rows read and written and its slot
            map) / device time of the step, summed over ranks (weak scaling)
  e2e     = the same bytes / time of a step through the C ABI that also copies the step's
            inputs host->device (pinned) and its output back
  roofline: the dominant kernel (decode) against the measured HBM copy bandwidth

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20


# ----------------------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
           "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return out

    def find(obj, names):
        if isinstance(obj, dict):
            for k, v in obj.items():
                if k in names and isinstance(v, (int, float)):
                    return float(v)
                r = find(v, names)
                if r is not None:
                    return r
        return None

    h = find(d, ("hbm_gbs", "hbm_GBps", "copy_gbs"))
    b = find(d, ("bf16_tflops", "bf16_tflops_burst"))
    bs = find(d, ("bf16_tflops_sustained",))
    if h:
        out.update(hbm_gbs=h, source="measured")
    if b:
        out["bf16_tflops"] = b
    if bs:
        out["bf16_tflops_sustained"] = bs
    return out


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


def nbytes(a):
    return int(a.nbytes)


# ----------------------------------------------------------------------------- workloads


def decode_bytes(b, pool):
    """Algorithmic bytes of one decode call: K/V over all contexts + q + out + block-table
    entries used + context lengths."""
    hkv, d = pool.n_kv_heads, pool.head_dim
    L = b.context_lens.astype(np.int64)
    kv = int(L.sum()) * 2 * hkv * d * 2
    q = nbytes(b.q)
    tables = int(np.ceil(L / pool.block_size).sum()) * 4
    return kv + 2 * q + tables + nbytes(b.context_lens)


def write_bytes(wr, pool):
    valid = int((wr.slot_mapping >= 0).sum())
    row = pool.n_kv_heads * pool.head_dim * 2
    return 2 * valid * row * 2 + nbytes(wr.slot_mapping)  # K and V rows read + written, slots read


WORKLOADS = {
    "step256": 4,
    "single": 1,
    "decode64": 2,
    "long4": 3,
}


# ----------------------------------------------------------------------------- our arm


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_232_gb300 as pa
    import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    k = WORKLOADS[args.workload]
    w = wl.make_workload(k)     # every rank gets its own copy of the same batch (weak scaling)
    p, b, wr = w.pool, w.decode, w.write
    dt = torch.bfloat16 if p.dtype == wl.BF16 else torch.float16

    def dev_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt).to(dev)

    kc, vc = dev_bits(p.k_cache), dev_bits(p.v_cache)
    q = dev_bits(b.q)
    bt = torch.from_numpy(b.block_tables).to(dev)
    cl = torch.from_numpy(b.context_lens).to(dev)
    out = torch.empty_like(q)
    S, hq, D = b.q.shape
    maxL = int(b.context_lens.max())
    ws_bytes = pa.pa_decode_workspace_size(S, hq, D, maxL, 0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    which, part = pa.pa_decode_plan(S, p.n_kv_heads, maxL)
    if wr is not None:
        key, val = dev_bits(wr.key), dev_bits(wr.value)
        sm = torch.from_numpy(wr.slot_mapping).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if wr is not None:
            if ev:
                ev[0].record(stream)
            pa.pa_reshape_and_cache(key, val, kc, vc, sm)
        if ev:
            ev[1].record(stream)
        pa.pa_decode(out, q, kc, vc, bt, cl, maxL, b.scale, ws)
        if ev:
            ev[2].record(stream)

    launches_per_step = (1 if wr is not None else 0) + (1 if which == 1 else 2)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with ClockSampler(local_rank) as clocks:
        for i in range(args.steps):
            flush.zero_()                       # L2 flush between steps, outside the timed events
            step(evs[i])
        torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall0
    w_ms = [e[0].elapsed_time(e[1]) if wr is not None else 0.0 for e in evs]
    d_ms = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = float(np.sum(w_ms) + np.sum(d_ms)) / args.steps
    step_ms = max_over_ranks(step_ms, world)

    dbytes = decode_bytes(b, p)
    wbytes = write_bytes(wr, p) if wr is not None else 0
    step_bytes = dbytes + wbytes
    value = world * step_bytes / (step_ms * 1e-3) / 1e9
    peaks = measured_peaks()
    dec_ms = float(np.mean(d_ms))
    achieved = dbytes / (dec_ms * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: inputs up, result down, every step
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_bt, h_cl = pin(q), pin(bt), pin(cl)
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    h2d = nbytes(b.q) + nbytes(b.block_tables) + nbytes(b.context_lens)
    if wr is not None:
        h_key, h_val, h_sm = pin(key), pin(val), pin(sm)
        h2d += nbytes(wr.key) + nbytes(wr.value) + nbytes(wr.slot_mapping)
    d2h = nbytes(b.q)

    def e2e_step():
        q.copy_(h_q, non_blocking=True)
        bt.copy_(h_bt, non_blocking=True)
        cl.copy_(h_cl, non_blocking=True)
        if wr is not None:
            key.copy_(h_key, non_blocking=True)
            val.copy_(h_val, non_blocking=True)
            sm.copy_(h_sm, non_blocking=True)
            pa.pa_reshape_and_cache(key, val, kc, vc, sm)
        pa.pa_decode(out, q, kc, vc, bt, cl, maxL, b.scale, ws)
        h_out.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(float(np.mean([a.elapsed_time(c) for a, c in e2e_ev])), world)

    res = {
        "metric": "paged decode attn us/step & achieved HBM GB/s (% of GB300 peak); KV-write GB/s",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "us_per_step": round(step_ms * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if p.dtype == wl.BF16 else "f16",
        "data": "synthetic (seeded SplitMix64/Box-Muller N(0,1), bf16 RNE)",
        "config": {
            "workload": wl.WORKLOAD_NAMES[k],
            "num_seqs": int(S), "n_q_heads": int(hq), "n_kv_heads": p.n_kv_heads, "head_dim": p.head_dim,
            "block_size": p.block_size, "total_context_tokens": int(b.context_lens.sum()),
            "write_rows": int(wr.slot_mapping.size) if wr is not None else 0,
            "padded_rows": int((wr.slot_mapping < 0).sum()) if wr is not None else 0,
            "decode_path": "one-pass" if which == 1 else f"split-K/{part}",
            "l2": "512 MiB memset between timed steps (outside the events); working set > L2",
            "parallelism": f"replicas x{world} (independent batches, no collective)",
        },
        "breakdown": {
            "write_us": round(float(np.mean(w_ms)) * 1e3, 2),
            "write_gbs": round(wbytes / (np.mean(w_ms) * 1e-3) / 1e9, 1) if wr is not None else None,
            "decode_us": round(dec_ms * 1e3, 2),
            "decode_gbs": round(achieved, 1),
            "step_bytes": step_bytes,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "decode_kernel (pa_decode)",
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "peak_source": peaks["source"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": args.traffic,
            "algorithmic_bytes": dbytes,
        },
        "e2e": {
            "value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
        },
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": round(t_wall, 4),
    }
    cs = clocks.summary()
    if cs:
        res["clocks"] = cs
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, k, budget_s=args.cpu_seconds)
    return res


# ----------------------------------------------------------------------------- oracle arm


def oracle_sample_step(w, n_seqs):
    """One bounded step of the oracle: the write of the sample's rows, then decode of the
    first n_seqs sequences.  Returns (bytes, seconds)."""
    import oracle
    p, b, wr = w.pool, w.decode, w.write
    t0 = time.perf_counter()
    nbytes_done = 0
    k_cache, v_cache = p.k_cache, p.v_cache
    if wr is not None:
        sl = slice(0, n_seqs)
        k_cache, v_cache, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key[sl], wr.value[sl],
                                              wr.slot_mapping[sl], p.block_size)
        valid = int((wr.slot_mapping[sl] >= 0).sum())
        nbytes_done += 2 * valid * p.n_kv_heads * p.head_dim * 2 * 2 + 8 * n_seqs
    out = oracle.decode(b.q[:n_seqs], k_cache, v_cache, b.block_tables[:n_seqs], b.context_lens[:n_seqs], b.scale,
                        p.dtype)
    dt = time.perf_counter() - t0
    sub = type(b)(b.q[:n_seqs], b.block_tables[:n_seqs], b.context_lens[:n_seqs], b.n_q_heads, b.scale)
    nbytes_done += decode_bytes(sub, p)
    assert np.isfinite(out).all()
    return nbytes_done, dt


def _sample_size(w, budget_s):
    n = 1
    nb, dt = oracle_sample_step(w, n)
    S = w.decode.num_seqs
    while dt < budget_s / 4 and n < S:
        n = min(S, n * 2)
        nb, dt = oracle_sample_step(w, n)
    return n, nb, dt


def cpu_baseline(w, k, budget_s=10.0):
    import oracle
    n, nb, dt = _sample_size(w, budget_s)
    # time enough repetitions of the sample to fill roughly the budget
    reps = max(1, int(budget_s / max(dt, 1e-3)))
    t0 = time.perf_counter()
    tot = 0
    for _ in range(reps):
        b_, _ = oracle_sample_step(w, n)
        tot += b_
    el = time.perf_counter() - t0
    return {"value": round(tot / el / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {w.decode.num_seqs} sequences (their write rows + decode), {reps} reps, {el:.1f} s"}


def run_reference(args, rank, world):
    import oracle
    import workloads as wl
    if rank != 0:
        return None
    k = WORKLOADS[args.workload]
    w = wl.make_workload(k)
    n, _, dt = _sample_size(w, budget_s=min(5.0, args.cpu_seconds))
    for _ in range(args.warmup):
        oracle_sample_step(w, n)
    tot, el = 0, 0.0
    for _ in range(args.steps):
        b_, t_ = oracle_sample_step(w, n)
        tot += b_
        el += t_
    value = tot / el / 1e9
    p, b = w.pool, w.decode
    return {
        "impl": "reference",
        "metric": "paged decode attn us/step & achieved HBM GB/s (% of GB300 peak); KV-write GB/s",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": {"workload": wl.WORKLOAD_NAMES[k], "num_seqs": int(b.num_seqs), "sampled_seqs": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{n} of {b.num_seqs} sequences per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- distributed glue


_PG = None


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="step256")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of this workload (reported as-is)")
    args = ap.parse_args(argv)
    assert args.warmup >= 3, "at least 3 warm-up steps"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
