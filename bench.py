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
            inputs host->device (one copy from a pinned buffer holding all of them) and its
            output back, inside the step's events
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
L2_CLEAN_BYTES = 256 << 20


class L2Flush:
    """Between timed steps (outside the events): write a buffer four times the L2 (129 MB) and
    then read another twice its size, so that a step starts with nothing of its own data in L2
    and with no dirty lines from the flush still to be written back during it."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


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
    "mixed": 5,
    "write64k": "write64k",   # bandwidth-scale KV write: 65,536 rows (10% padded) to random slots
    "rope64k": "rope64k",     # the same write with rotary embedding fused in (keys, and 16 query heads per row)
    "rope256": "rope256",     # the batch-256 decode step with the fused RoPE write in place of the plain one
}
ROPE_THETA, ROPE_MAX_POS = 1.0e6, 32768   # Qwen3-shaped: rotary base 1e6


def make_bench_workload(k, wl):
    if k in ("write64k", "rope64k"):
        w = wl.write_rows_case(232_104, 65536)
        if k == "rope64k":
            n = w.write.key.shape[0]
            w.rope = dict(q=wl.normal_bits(wl.derive_seed(232_104, 12), n * 16 * 128, wl.BF16).reshape(n, 16, 128),
                          positions=wl.uniform_ints(wl.derive_seed(232_104, 11), n, 0, ROPE_MAX_POS - 1).astype(np.int64))
        return w
    if k == "rope256":
        w = wl.make_workload(4)
        w.rope = dict(q=w.decode.q, positions=w.decode.context_lens.astype(np.int64) - 1)
        return w
    return wl.make_workload(k)


def rope_write_bytes(w):
    """Positions and slots, query rows read and written, and per written row: key / value read,
    both cache rows written, one cos / sin table row read."""
    p, wr, q = w.pool, w.write, w.rope["q"]
    n = wr.slot_mapping.size
    valid = int((wr.slot_mapping >= 0).sum())
    row = p.n_kv_heads * p.head_dim * 2
    return 16 * n + 2 * q.nbytes + valid * (4 * row + p.head_dim * 4)


def workload_name(k, wl):
    if k == "write64k":
        return "bandwidth-scale KV write: 65,536 rows x 8 KV heads x 128 (bf16, 10% padded -1) to random slots"
    if k == "rope64k":
        return ("bandwidth-scale KV write with fused RoPE: 65,536 rows x 8 KV heads x 128 + 16 query heads rotated "
                "in place (bf16, 10% padded -1, positions U[0, 32768), base 1e6)")
    if k == "rope256":
        return "full decode step at batch 256 with the fused RoPE write (positions = context_len - 1, base 1e6)"
    return wl.WORKLOAD_NAMES[k]


def sample_units(w):
    """Units the oracle samples: sequences (their write rows + decode), or write rows."""
    return w.decode.num_seqs if w.decode is not None else int(w.write.slot_mapping.size)


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, or None
    when there is none or the kernels have been rebuilt from other sources since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel}@{workload}")
        from paged_kv_cache_232_gb300 import _build
        if rec and rec.get("build_digest") == _build._digest():
            return int(rec["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


# ----------------------------------------------------------------------------- our arm


def prefill_flops(pre, n_q_heads, head_dim):
    """4 * D flops (QK^T and PV) per visible (query row, key) pair and head: causal pairs only."""
    ql = np.diff(pre.query_start_loc).astype(np.int64)
    ctx = pre.seq_lens.astype(np.int64) - ql
    pairs = int(np.sum(ql * ctx + ql * (ql + 1) // 2))
    return 4 * head_dim * n_q_heads * pairs


def prefill_bytes(pre, pool):
    kv = int(pre.seq_lens.astype(np.int64).sum()) * 2 * pool.n_kv_heads * pool.head_dim * 2
    return kv + 2 * nbytes(pre.q) + int(np.ceil(pre.seq_lens / pool.block_size).sum()) * 4


def unique_decode_bytes(b, pool):
    """Decode bytes counting each physical block's tokens once (a shared prefix is read from
    HBM once, the rest of its reads hit L2); equals decode_bytes when no block is shared."""
    L = b.context_lens.astype(np.int64)
    bs = pool.block_size
    tokens = {}
    for s in range(b.num_seqs):
        n = -(-int(L[s]) // bs)
        for j, blk in enumerate(b.block_tables[s, :n].tolist()):
            tokens[blk] = max(tokens.get(blk, 0), min(bs, int(L[s]) - j * bs))
    kv = sum(tokens.values()) * 2 * pool.n_kv_heads * pool.head_dim * 2
    return kv + 2 * nbytes(b.q) + int(np.ceil(L / bs).sum()) * 4 + nbytes(b.context_lens)


def workload_config(w, k, wl, world):
    """The workload a line measures: the same dict in both arms (the GPU kernels and the fp64
    oracle), so that the two lines' configs compare equal."""
    p, b, wr, pre = w.pool, w.decode, w.write, w.prefill
    cfg = {"workload": workload_name(k, wl), "n_kv_heads": p.n_kv_heads, "head_dim": p.head_dim,
           "block_size": p.block_size}
    if b is not None:
        cfg.update({"num_seqs": int(b.num_seqs), "n_q_heads": int(b.q.shape[1]),
                    "total_context_tokens": int(b.context_lens.sum())})
        if w.meta.get("shared_prefix_tokens", 0):
            cfg["shared_prefix_tokens"] = int(w.meta["shared_prefix_tokens"])
    if wr is not None:
        cfg.update(write_rows=int(wr.slot_mapping.size), padded_rows=int((wr.slot_mapping < 0).sum()))
    if pre is not None:
        cfg.update(prefill_chunks=pre.num_chunks, prefill_rows=int(pre.q.shape[0]),
                   prefill_kv_lens=[int(x) for x in pre.seq_lens])
    cfg.update({"l2": "GPU arm: between timed steps, outside the events, a 512 MiB memset (L2 flush) then a 256 MiB "
                      "read (no dirty flush lines left to write back)",
                "parallelism": f"replicas x{world} (independent batches, no collective)"})
    return cfg


class _Ctx:
    pass


class _Arena:
    """One device buffer for a step's inputs, handed out as 256-byte aligned views, and a pinned
    host buffer with the same layout (the end-to-end leg's single upload)."""

    def __init__(self, torch, dev, capacity):
        self.dev_buf = torch.empty(capacity, dtype=torch.uint8, device=dev)
        self.host = torch.empty(capacity, dtype=torch.uint8).pin_memory()
        self.used = 0

    def put(self, a, torch_dtype):
        raw = np.ascontiguousarray(a).reshape(-1).view(np.uint8)
        off, nb = self.used, raw.size
        assert off + nb <= self.dev_buf.numel(), "input arena too small"
        self.used = (off + nb + 255) // 256 * 256
        self.host[off:off + nb].numpy()[:] = raw
        view = self.dev_buf[off:off + nb]
        view.copy_(self.host[off:off + nb])
        return view.view(torch_dtype).view(tuple(a.shape))


def prepare(args, name, dev, with_host=False):
    """Device inputs and the launches of one step of workload `name` (every rank builds its own
    copy of the same batch: weak scaling)."""
    import torch
    import paged_kv_cache_232_gb300 as pa
    import workloads as wl

    c = _Ctx()
    c.name, c.k = name, WORKLOADS[name]
    w = c.w = make_bench_workload(c.k, wl)
    p, b, wr, pre = w.pool, w.decode, w.write, w.prefill
    dt = torch.bfloat16 if p.dtype == wl.BF16 else torch.float16

    # the step's inputs live in one device buffer (256-byte aligned views) mirrored by one pinned
    # host buffer, so that the end-to-end leg uploads a step's inputs with one copy
    cand = []
    if b is not None:
        cand += [b.q, b.block_tables, b.context_lens]
    if pre is not None:
        cand += [pre.q, pre.block_tables, pre.query_start_loc, pre.seq_lens]
    if wr is not None:
        cand += [wr.key, wr.value, wr.slot_mapping]
    rope = getattr(w, "rope", None)
    if rope is not None:
        cand += [rope.get("positions"), rope.get("q")]
    cap = 2 * sum(int(np.asarray(a).nbytes) + 256 for a in cand if a is not None) + (1 << 20)
    arena = c.arena = _Arena(torch, dev, cap)

    def dev_bits(a):
        return arena.put(np.ascontiguousarray(a).view(np.int16), dt)

    def dev_int(a):
        a = np.ascontiguousarray(a)
        return arena.put(a, torch.int64 if a.dtype == np.int64 else torch.int32)

    def cache_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt).to(dev)

    kc, vc = cache_bits(p.k_cache), cache_bits(p.v_cache)
    stages = []   # name, launch, algorithmic amount, kind
    h_dev = []    # the step's inputs, for the end-to-end leg
    if rope is not None and b is not None:
        q_host = np.concatenate([b.q, pre.q]) if pre is not None else b.q
        q = dev_bits(q_host)                       # rotated in place by the fused write, then decoded
        q_rope = q[:b.num_seqs]
    elif rope is not None:
        q_rope = dev_bits(rope["q"])
    if wr is not None:
        key, val, sm = dev_bits(wr.key), dev_bits(wr.value), dev_int(wr.slot_mapping)
        h_dev += [key, val, sm]
        if rope is None:
            stages.append(("write", lambda: pa.pa_reshape_and_cache(key, val, kc, vc, sm), write_bytes(wr, p), "hbm"))
        else:
            pos_d = dev_int(rope["positions"])
            h_dev += [pos_d] + ([q_rope] if b is None else [])
            cos_sin = pa.rope_cos_sin(ROPE_MAX_POS, p.head_dim, ROPE_THETA, dev)
            stages.append(("rope_write", lambda: pa.pa_rope_reshape_and_cache(key, val, kc, vc, sm, pos_d, cos_sin,
                                                                              q=q_rope),
                           rope_write_bytes(w), "hbm"))
    S, which, dec_logical, dec_launches, part, prefix = 0, 0, 0, 0, 0, 0
    fused = False
    if b is not None:
        S, hq, D = b.q.shape
        if rope is None:
            q_host = np.concatenate([b.q, pre.q]) if pre is not None else b.q
            q = dev_bits(q_host)                   # decode rows first, then prefill rows
        out = torch.empty_like(q)
        bt, cl = dev_int(b.block_tables), dev_int(b.context_lens)
        h_dev += [q, bt, cl]
        maxL = int(b.context_lens.max())
        ws = torch.empty(max(pa.pa_decode_workspace_size(S, hq, D, maxL, 0), 16), dtype=torch.uint8, device=dev)
        code = pa.PA_BF16 if p.dtype == wl.BF16 else pa.PA_F16
        which, part = pa.pa_decode_plan(S, hq, p.n_kv_heads, D, p.block_size, maxL, code)
        if args.decode_path == "v1":
            which = 1
        elif args.decode_path == "splitk":
            which, part = 2, (args.partition or part)
        dec_logical = decode_bytes(b, p)
        dec_unique = unique_decode_bytes(b, p)
        prefix = int(w.meta.get("shared_prefix_tokens", 0))
        dec_launches = 1 if which == 1 else 2
        if args.decode_path == "auto" and prefix > 0:
            # the caller knows the blocks its sequences share (its prefix cache): the prefix part
            # once per KV head on the tensor cores, the rest per sequence
            which = 3
            ws = torch.empty(max(pa.pa_decode_shared_prefix_workspace_size(S, hq, D, maxL, prefix), 16),
                             dtype=torch.uint8, device=dev)
            sw, part = pa.pa_decode_plan(S, hq, p.n_kv_heads, D, p.block_size, maxL - prefix, code)
            dec_launches = 2 if sw == 1 else 3
            dec_fn = lambda: pa.pa_decode_shared_prefix(out[:S], q[:S], kc, vc, bt, cl, maxL, b.scale, prefix, ws,
                                                        prefix_piece_tokens=args.prefix_piece)
        elif args.decode_path in ("auto", "plain"):
            dec_fn = lambda: pa.pa_decode(out[:S], q[:S], kc, vc, bt, cl, maxL, b.scale, ws)
        elif which == 1:
            dec_fn = lambda: pa.pa_decode_v1(out[:S], q[:S], kc, vc, bt, cl, b.scale)
        else:
            ws = torch.empty(max(pa.pa_decode_workspace_size(S, hq, D, maxL, part), 16), dtype=torch.uint8,
                             device=dev)
            dec_fn = lambda: pa.pa_decode_splitk(out[:S], q[:S], kc, vc, bt, cl, maxL, b.scale, ws, part)
        stages.append(("decode", dec_fn, dec_unique, "hbm"))
        if (args.step_path == "fused" and wr is not None and rope is None and pre is None and which in (1, 2)
                and args.decode_path in ("auto", "plain") and wr.key.shape[0] == S):
            # the step as one call: pa_decode_write puts each sequence's new row into the cache and
            # decodes (on the persistent grid the decode CTAs write the rows themselves)
            stages = [("decode_write", lambda: pa.pa_decode_write(out[:S], q[:S], kc, vc, bt, cl, maxL, b.scale, key,
                                                                  val, sm, ws),
                       write_bytes(wr, p) + dec_unique, "hbm")]
            fused = True
    else:
        # write only: the step's result lives in the cache; the end-to-end leg reads back the
        # first written K row as its completion check
        slot0 = int(wr.slot_mapping[wr.slot_mapping >= 0][0])
        out = kc[slot0 // p.block_size, slot0 % p.block_size]
        if rope is not None:
            q = q_rope
    if pre is not None and args.unified:
        # one prefill launch over every row: decode sequences as one-row chunks, then the chunks
        u = wl.unified_batch(w)
        pbt, qsl, sl = dev_int(u.block_tables), dev_int(u.query_start_loc), dev_int(u.seq_lens)
        h_dev += [pbt, qsl, sl]
        stages = [s_ for s_ in stages if s_[0] != "decode"]
        stages.append(("unified", lambda: pa.pa_prefill_chunk(out, q, kc, vc, pbt, qsl, sl, u.max_q_len, u.scale,
                                                              small_m=args.small_m),
                       prefill_flops(u, hq, D), "tensor"))
        which, dec_logical, dec_launches = 0, 0, 0
    elif pre is not None:
        pbt, qsl, sl = dev_int(pre.block_tables), dev_int(pre.query_start_loc), dev_int(pre.seq_lens)
        h_dev += [pbt, qsl, sl]
        stages.append(("prefill", lambda: pa.pa_prefill_chunk(out[S:], q[S:], kc, vc, pbt, qsl, sl, pre.max_q_len,
                                                              pre.scale),
                       prefill_flops(pre, hq, D), "tensor"))
    c.stages, c.out, c.h_dev, c.fused = stages, out, h_dev, fused
    # (a fused step on the one-pass grid: batches this large run its persistent form, which writes
    # the rows itself; the other grids launch the KV-write kernel first)
    c.launches = ((1 if wr is not None and not (fused and which == 1) else 0) + dec_launches
                  + (1 if pre is not None else 0))
    wbytes = 0 if wr is None else (rope_write_bytes(w) if rope is not None else write_bytes(wr, p))
    c.step_bytes = wbytes + (decode_bytes(b, p) if (b is not None and args.unified) else dec_logical) + (
        prefill_bytes(pre, p) if pre is not None else 0)
    c.dec_logical = dec_logical
    c.has_pre_and_dec = pre is not None and b is not None
    c.decode_path = None
    if b is not None:
        c.decode_path = (("unified: decode rows as one-row chunks of the prefill launch"
                          + (" (small-M tiles)" if args.small_m else "")) if which == 0
                         else (f"shared prefix of {prefix} tokens on the tensor cores + suffix "
                               + ("one-pass" if dec_launches == 2 else f"split-K/{part}") if which == 3
                               else ("one-pass" if which == 1 else f"split-K/{part}"))
                         + ("" if args.decode_path in ("auto", "plain") else " (forced)")
                         + (" with the KV write in the same call (pa_decode_write)" if fused else ""))
    return c


def step_fn(c, stream):
    ns = len(c.stages)

    def step(ev=None):
        for i, st in enumerate(c.stages):
            if ev:
                ev[i].record(stream)
            st[1]()
        if ev:
            ev[ns].record(stream)
    return step


def time_steps(c, steps, warmup, world, local_rank, flush, stream, per_stage=True):
    """W untimed steps, then `steps` timed ones (L2 flushed before each, outside the events).
    per_stage: an event between every two launches, returning milliseconds [steps, stages];
    otherwise events only around each whole step (the launches of a step run back to back, as
    in use: the decode is a programmatic dependent of the write), returning [steps, 1].  Also
    returns the clock summary and the wall time."""
    import torch
    import paged_kv_cache_232_gb300 as pa
    step = step_fn(c, stream)
    ns = len(c.stages)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1 if per_stage else 2)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with ClockSampler(local_rank) as clocks:
        for i in range(steps):
            flush()                             # L2 flush between steps, outside the timed events
            if per_stage:
                step(evs[i])
            else:
                evs[i][0].record(stream)
                step()
                evs[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall0
    assert pa.pa_device_errors(clear=True) == 0
    st_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(len(e) - 1)] for e in evs])
    return st_ms, clocks.summary(), t_wall


def summarize(c, st_ms, world, peaks, traffic=None, whole_ms=None):
    """Step time (max over ranks; the whole-step timing when given, else the sum of the stages),
    whole-job value, per-stage rates and the dominant kernel's roofline."""
    step_ms = max_over_ranks(float(st_ms.sum(axis=1).mean()) if whole_ms is None else float(whole_ms.mean()), world)
    mean_ms = st_ms.mean(axis=0)
    breakdown = {}
    for (name, _, amount, kind), ms in zip(c.stages, mean_ms):
        if kind == "hbm":
            breakdown[name] = {"us": round(float(ms) * 1e3, 2), "gbs": round(amount / (ms * 1e-3) / 1e9, 1),
                               "frac_hbm": round(amount / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        else:
            breakdown[name] = {"us": round(float(ms) * 1e3, 2), "tflops": round(amount / (ms * 1e-3) / 1e12, 1),
                               "frac_bf16": round(amount / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                               "flop": amount}
    if c.has_pre_and_dec and "decode" in breakdown:
        breakdown["decode"]["logical_gbs"] = round(c.dec_logical / (mean_ms[0] * 1e-3) / 1e9, 1)
        breakdown["decode"]["note"] = "gbs / frac_hbm on unique bytes (a shared block counted once)"
    dom = int(np.argmax(mean_ms))
    dname, _, damount, dkind = c.stages[dom]
    dms = float(mean_ms[dom])
    if traffic is None:
        traffic = recorded_traffic(c.name, dname)
    if dkind == "hbm":
        ach = damount / (dms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": f"{dname}", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "peak_source": peaks["source"], "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes": damount}
    else:
        ach = damount / (dms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": f"{dname}", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                "peak_source": peaks["source"], "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
                "traffic": traffic, "algorithmic_flops": damount}
    return step_ms, world * c.step_bytes / (step_ms * 1e-3) / 1e9, breakdown, roof


# every configuration of the workload list, measured after the headline in the default run
ALL_CONFIGS = ("single", "decode64", "long4", "mixed", "write64k")


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_232_gb300 as pa
    import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    c = prepare(args, args.workload, dev)
    p = c.w.pool
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    peaks = measured_peaks()
    # the timed region: whole steps (one event pair per step); then, for a step of several
    # launches, a second pass with an event between every two launches for the per-kernel times
    whole, clocks, t_wall = time_steps(c, args.steps, args.warmup, world, local_rank, flush, stream, per_stage=False)
    st_ms = whole
    if len(c.stages) > 1:
        st_ms, _, _ = time_steps(c, args.steps, args.warmup, world, local_rank, flush, stream, per_stage=True)
    step_ms, value, breakdown, roof = summarize(c, st_ms, world, peaks, args.traffic, whole_ms=whole[:, 0])

    # end to end through the C ABI with host buffers, every step: the step's inputs go up in one
    # copy from the pinned mirror of the input buffer, then the launches, then the result comes down
    arena = c.arena
    h_out = torch.empty_like(c.out, device="cpu").pin_memory()
    h2d = arena.used
    d2h = c.out.numel() * c.out.element_size()
    up_dst, up_src = arena.dev_buf[:arena.used], arena.host[:arena.used]

    def e2e_step():
        up_dst.copy_(up_src, non_blocking=True)
        for st in c.stages:
            st[1]()
        h_out.copy_(c.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        e2e_ev[i][0].record(stream)
        e2e_step()
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b_) for a, b_ in e2e_ev])), world)

    # the same step captured once into a CUDA graph and replayed (launch overhead removed)
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for st in c.stages:
                st[1]()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        g_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            g_ev[i][0].record(stream)
            g.replay()
            g_ev[i][1].record(stream)
        torch.cuda.synchronize()
        graph_ms = max_over_ranks(float(np.mean([a.elapsed_time(b_) for a, b_ in g_ev])), world)
        assert pa.pa_device_errors(clear=True) == 0
    except RuntimeError as ex:   # capture refused: report it instead of a number
        graph_ms = f"capture failed: {str(ex).splitlines()[0][:120]}"

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
        "data": "synthetic (seeded SplitMix64/Box-Muller N(0,1), RNE to the 16-bit format)",
        "config": workload_config(c.w, c.k, wl, world),
        "decode_path": c.decode_path,
        "breakdown": breakdown,
        "breakdown_method": ("value: events around whole steps; breakdown and roofline: a second pass of the same "
                             "steps with an event between every two launches"),
        "step_bytes": c.step_bytes,
        "roofline": roof,
        "e2e": {
            "value": round(world * c.step_bytes / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
        },
        "graph": ({"us_per_step": round(graph_ms * 1e3, 2),
                   "value": round(world * c.step_bytes / (graph_ms * 1e-3) / 1e9, 2),
                   "unit": "GB/s", "note": "the step's launches captured once into a CUDA graph, replayed per step"}
                  if isinstance(graph_ms, float) else {"unavailable": graph_ms}),
        "gpu_launches": c.launches * args.steps,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if clocks:
        res["clocks"] = clocks
    if c.fused:
        # the same step as two calls (pa_reshape_and_cache, then pa_decode), for its per-kernel times
        sep = argparse.Namespace(**vars(args))
        sep.step_path = "separate"
        cs = prepare(sep, args.workload, dev)
        whs, _, _ = time_steps(cs, args.steps, args.warmup, world, local_rank, flush, stream, per_stage=False)
        sts, _, _ = time_steps(cs, args.steps, args.warmup, world, local_rank, flush, stream, per_stage=True)
        sms, _, sbd, _ = summarize(cs, sts, world, peaks, None, whole_ms=whs[:, 0])
        res["separate_step"] = {"us_per_step": round(sms * 1e3, 2), "breakdown": sbd,
                                "note": "pa_reshape_and_cache then pa_decode, two launches; the breakdown with an "
                                        "event between them"}
        del cs
    w_head, k_head = c.w, c.k
    del c, h_out, e2e_step, up_dst, up_src, arena
    if args.all_configs and args.workload == "step256":
        # the other configurations, each timed the same way in this run (its own clocks)
        extra = argparse.Namespace(**vars(args))
        extra.decode_path, extra.unified, extra.partition, extra.prefix_piece = "auto", False, 0, 0
        res["workloads"] = {}
        for name in ALL_CONFIGS:
            torch.cuda.empty_cache()
            c2 = prepare(extra, name, dev)
            wh2, clk2, _ = time_steps(c2, args.steps, args.warmup, world, local_rank, flush, stream, per_stage=False)
            st2 = wh2
            if len(c2.stages) > 1:
                st2, _, _ = time_steps(c2, args.steps, args.warmup, world, local_rank, flush, stream, per_stage=True)
            ms2, val2, br2, roof2 = summarize(c2, st2, world, peaks, whole_ms=wh2[:, 0])
            res["workloads"][name] = {
                "config": workload_config(c2.w, c2.k, wl, world), "decode_path": c2.decode_path,
                "us_per_step": round(ms2 * 1e3, 2), "value": round(val2, 2), "unit": "GB/s",
                "breakdown": br2, "roofline": roof2, "gpu_launches": c2.launches * args.steps,
                "clocks": clk2,
            }
            del c2
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w_head, k_head, budget_s=args.cpu_seconds,
                                           single_thread=args.all_configs and args.workload == "step256")
    return res


# ----------------------------------------------------------------------------- oracle arm


def oracle_sample_step(w, n_seqs):
    """One bounded step of the oracle: the write of the sample's rows, then decode of the
    first n_seqs sequences (a write-only workload: the write of its first n_seqs rows).
    Returns (bytes, seconds)."""
    import oracle
    p, b, wr = w.pool, w.decode, w.write
    t0 = time.perf_counter()
    nbytes_done = 0
    k_cache, v_cache = p.k_cache, p.v_cache
    rope = getattr(w, "rope", None)
    qs = None
    if wr is not None:
        sl = slice(0, n_seqs)
        if rope is None:
            k_cache, v_cache, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key[sl], wr.value[sl],
                                                  wr.slot_mapping[sl], p.block_size)
        else:
            qs, k_cache, v_cache, _ = oracle.rope_kv_write(rope["q"][sl], p.k_cache, p.v_cache, wr.key[sl],
                                                           wr.value[sl], wr.slot_mapping[sl], rope["positions"][sl],
                                                           ROPE_MAX_POS, ROPE_THETA, p.dtype)
            nbytes_done += 2 * rope["q"][sl].nbytes + 16 * n_seqs
        valid = int((wr.slot_mapping[sl] >= 0).sum())
        nbytes_done += 2 * valid * p.n_kv_heads * p.head_dim * 2 * 2 + 8 * n_seqs
    if b is None:
        return nbytes_done, time.perf_counter() - t0
    out = oracle.decode(b.q[:n_seqs] if qs is None else qs, k_cache, v_cache, b.block_tables[:n_seqs], b.context_lens[:n_seqs], b.scale,
                        p.dtype)
    dt = time.perf_counter() - t0
    sub = type(b)(b.q[:n_seqs], b.block_tables[:n_seqs], b.context_lens[:n_seqs], b.n_q_heads, b.scale)
    nbytes_done += decode_bytes(sub, p)
    assert np.isfinite(out).all()
    return nbytes_done, dt


def _sample_size(w, budget_s):
    n = 1
    nb, dt = oracle_sample_step(w, n)
    S = sample_units(w)
    while dt < budget_s / 4 and n < S:
        n = min(S, n * 2)
        nb, dt = oracle_sample_step(w, n)
    return n, nb, dt


def _timed_oracle(w, budget_s):
    n, nb, dt = _sample_size(w, budget_s)
    # time enough repetitions of the sample to fill roughly the budget
    reps = max(1, int(budget_s / max(dt, 1e-3)))
    t0 = time.perf_counter()
    tot = 0
    for _ in range(reps):
        b_, _ = oracle_sample_step(w, n)
        tot += b_
    el = time.perf_counter() - t0
    what = (f"{n} of {w.decode.num_seqs} sequences (their write rows + decode)" if w.decode is not None
            else f"{n} of {sample_units(w)} write rows") + f", {reps} reps, {el:.1f} s"
    return tot / el / 1e9, what


def cpu_baseline(w, k, budget_s=10.0, single_thread=False):
    """The fp64 oracle as it stands on the host's cores (all of them), on a bounded sample of
    the same workload; with single_thread, also on one core for the single-request, batch-64
    and long-context decode workloads."""
    import oracle
    import workloads as wl
    v, what = _timed_oracle(w, budget_s)
    res = {"value": round(v, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle", "sample": what}
    if single_thread:
        all_cores = oracle.num_threads()
        oracle.set_num_threads(1)
        try:
            res["single_thread"] = {}
            for name in ("single", "decode64", "long4"):
                v1, what1 = _timed_oracle(make_bench_workload(WORKLOADS[name], wl), 2.0)
                res["single_thread"][name] = {"value": round(v1, 4), "unit": "GB/s", "cores": 1, "sample": what1}
        finally:
            oracle.set_num_threads(all_cores)
    return res


def run_reference(args, rank, world):
    import oracle
    import workloads as wl
    if rank != 0:
        return None
    k = WORKLOADS[args.workload]
    w = make_bench_workload(k, wl)
    n, _, dt = _sample_size(w, budget_s=min(5.0, args.cpu_seconds))
    for _ in range(args.warmup):
        oracle_sample_step(w, n)
    tot, el = 0, 0.0
    for _ in range(args.steps):
        b_, t_ = oracle_sample_step(w, n)
        tot += b_
        el += t_
    value = tot / el / 1e9
    units = sample_units(w)
    what = "sequences" if w.decode is not None else "write rows"
    return {
        "impl": "reference",
        "metric": "paged decode attn us/step & achieved HBM GB/s (% of GB300 peak); KV-write GB/s",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": workload_config(w, k, wl, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{n} of {units} {what} per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- distributed glue


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
    ap.add_argument("--unified", action="store_true",
                    help="mixed batch: decode rows through the prefill kernel in the same launch (one-row chunks)")
    ap.add_argument("--small-m", action="store_true",
                    help="with --unified: pa_prefill_chunk_small_m (M = 64 tiles for the decode rows' units)")
    ap.add_argument("--decode-path", choices=["auto", "plain", "v1", "splitk"], default="auto",
                    help="force the one-pass or split-K decode kernel instead of the library's dispatcher "
                         "(plain: the dispatcher without the shared-prefix pass)")
    ap.add_argument("--step-path", choices=["fused", "separate"], default="fused",
                    help="a step with a KV write and a decode: one pa_decode_write call (fused) or "
                         "pa_reshape_and_cache then pa_decode (separate, timed launch by launch)")
    ap.add_argument("--prefix-piece", type=int, default=0,
                    help="shared-prefix pass: keys per CTA (multiple of 128; 0 = the library's choice)")
    ap.add_argument("--partition", type=int, default=0, help="split-K piece length in tokens (with --decode-path splitk)")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other configurations the default (batch-256 step) run also measures")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of this workload (reported as-is)")
    args = ap.parse_args(argv)
    args.all_configs = not args.headline_only
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
