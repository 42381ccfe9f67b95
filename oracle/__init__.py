"""fp64 CPU oracle for paged-KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline /
reference arm may import this package.  It shares no code with the CUDA
library (``paged_kv_cache_232_gb300``) and never imports it; the CUDA library
never imports this.  Inputs are numpy bit-pattern arrays (uint16 for fp16/bf16
tensors) produced by ``workloads``.

Each function is a thin ctypes marshal over ``pa_oracle.c``, whose header
comment states, for every routine, the passage of the pages it writes out:
paged address translation (MiniLLM Runtime, "Core class relationships"), the
slot mapping and padded-slot skip of the cache write (miniserve "Engine";
mini_engine "Custom CUDA kernels"), decode attention with GQA sharing and the
split-K max / exp-sum merge (mini_engine "Custom CUDA kernels"), the
bottom-right causal prefill chunk (miniserve "Engine"), and the
materialise-then-attend baseline (MiniLLM Runtime "Key benchmark results").

Parity status: every routine is pinned by ``tests/test_oracle_pins.py``
(library SDPA in fp64, closed forms, invariants, brute force on tiny inputs);
none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

F16, BF16 = 0, 1
OK, EARG, EBOUNDS = 0, -1, -2


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (fp64, OpenMP over independent rows)."""
    os.makedirs(_BUILD, exist_ok=True)
    so = os.path.join(_BUILD, f"libpaoracle_{_src_hash()}.so")
    if force or not os.path.exists(so):
        tmp = so + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, so)
        for old in os.listdir(_BUILD):          # older builds of other sources
            if old.endswith(".so") and os.path.join(_BUILD, old) != so:
                try:
                    os.remove(os.path.join(_BUILD, old))
                except OSError:
                    pass
    return so


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.pao_to_double.argtypes = [ctypes.c_uint16, i32]
        L.pao_to_double.restype = dbl
        L.pao_from_double.argtypes = [dbl, i32]
        L.pao_from_double.restype = ctypes.c_uint16
        L.pao_round_array.argtypes = [vp, i64, i32, vp]
        L.pao_widen_array.argtypes = [vp, i64, i32, vp]
        L.pao_kv_write.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64]
        L.pao_rope_exact.argtypes = [vp, vp, i32, dbl, dbl]
        L.pao_rope_exact.restype = None
        L.pao_rope_kv_write.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i64, i64, dbl, i32]
        L.pao_kv_write.restype = i32
        dec = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, dbl, i32]
        L.pao_decode.argtypes = dec
        L.pao_decode.restype = i32
        L.pao_decode_partitions.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64,
                                            dbl, i32, i32, i32]
        L.pao_decode_partitions.restype = i32
        L.pao_merge_partitions.argtypes = [vp, vp, vp, vp, i64, i32, i32]
        L.pao_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i64, dbl, i32]
        L.pao_prefill_chunk.restype = i32
        L.pao_naive_contiguous.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, dbl, i32]
        L.pao_naive_contiguous.restype = i32
        L.pao_num_threads.restype = i32
        L.pao_set_num_threads.argtypes = [i32]
        L.pao_set_num_threads.restype = None
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def num_threads() -> int:
    return int(lib().pao_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's OpenMP loops use from now on (results do not depend on it)."""
    lib().pao_set_num_threads(int(n))


def to_double(bits, dtype: int) -> np.ndarray:
    b, p = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().pao_widen_array(p, b.size, dtype, out.ctypes.data)
    return out


def round_to(x, dtype: int) -> np.ndarray:
    """Round doubles to fp16 (dtype 0) / bf16 (dtype 1) bits, nearest-even."""
    a, p = _c(x, np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().pao_round_array(p, a.size, dtype, out.ctypes.data)
    return out


def _check(st: int, what: str):
    if st != OK:
        raise RuntimeError(f"oracle {what} failed with status {st}")


def kv_write(k_cache, v_cache, key, value, slot_mapping, block_size: int, check: bool = True):
    """Return new (k_cache, v_cache) after scattering key/value rows to their slots."""
    k, kp = _c(np.array(k_cache, copy=True), np.uint16)
    v, vp_ = _c(np.array(v_cache, copy=True), np.uint16)
    key, keyp = _c(key, np.uint16)
    val, valp = _c(value, np.uint16)
    sm, smp = _c(slot_mapping, np.int64)
    nb, bs, hkv, d = k.shape
    assert bs == block_size
    st = lib().pao_kv_write(kp, vp_, keyp, valp, smp, sm.size, hkv, d, bs, nb)
    if check:
        _check(st, "kv_write")
    return k, v, st


def rope_exact(x, m: float, theta: float) -> np.ndarray:
    """Rotary embedding of one double row x (head_dim even) at position m, unrounded."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(x)
    lib().pao_rope_exact(x.ctypes.data, out.ctypes.data, x.size, float(m), float(theta))
    return out


def rope_kv_write(q, k_cache, v_cache, key, value, slot_mapping, positions, max_position: int, theta: float,
                  dtype: int, check: bool = True):
    """Fused rotary embedding + KV write.  Returns (q rotated or None, k_cache, v_cache, status),
    all new arrays; the inputs are not modified."""
    qq = None
    qptr = None
    if q is not None:
        qq, qptr = _c(np.array(q, copy=True), np.uint16)
    k, kp = _c(np.array(k_cache, copy=True), np.uint16)
    v, vp_ = _c(np.array(v_cache, copy=True), np.uint16)
    key, keyp = _c(key, np.uint16)
    val, valp = _c(value, np.uint16)
    sm, smp = _c(slot_mapping, np.int64)
    pos, posp = _c(positions, np.int64)
    nb, bs, hkv, d = k.shape
    hq = qq.shape[1] if qq is not None else 0
    st = lib().pao_rope_kv_write(qptr, kp, vp_, keyp, valp, smp, posp, sm.size, hq, hkv, d, bs, nb,
                                 int(max_position), float(theta), int(dtype))
    if check:
        _check(st, "rope_kv_write")
    return qq, k, v, st


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: int, want_weights=False):
    """fp64 decode attention. Returns out [S, Hq, D] (and weights [S, Hq, MB*bs])."""
    q, qp = _c(q, np.uint16)
    k, kp = _c(k_cache, np.uint16)
    v, vp_ = _c(v_cache, np.uint16)
    bt, btp = _c(block_tables, np.int32)
    cl, clp = _c(context_lens, np.int32)
    S, Hq, D = q.shape
    nb, bs, hkv, d2 = k.shape
    assert d2 == D and bt.shape[0] == S and cl.shape[0] == S
    out = np.empty((S, Hq, D), dtype=np.float64)
    w = np.empty((S, Hq, bt.shape[1] * bs), dtype=np.float64) if want_weights else None
    st = lib().pao_decode(out.ctypes.data, w.ctypes.data if w is not None else None, qp, kp, vp_, btp, bt.shape[1],
                          clp, S, Hq, hkv, D, bs, nb, float(scale), dtype)
    _check(st, "decode")
    return (out, w) if want_weights else out


def decode_partitions(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: int,
                      partition_tokens: int = 256, max_parts: int | None = None):
    """fp64 split-K pieces: (m, l, o) with m, l [S, Hq, P] and o [S, Hq, P, D]."""
    q, qp = _c(q, np.uint16)
    k, kp = _c(k_cache, np.uint16)
    v, vp_ = _c(v_cache, np.uint16)
    bt, btp = _c(block_tables, np.int32)
    cl, clp = _c(context_lens, np.int32)
    S, Hq, D = q.shape
    nb, bs, hkv, _ = k.shape
    if max_parts is None:
        max_parts = max(1, -(-int(cl.max()) // partition_tokens))
    m = np.empty((S, Hq, max_parts))
    l = np.empty((S, Hq, max_parts))
    o = np.empty((S, Hq, max_parts, D))
    st = lib().pao_decode_partitions(m.ctypes.data, l.ctypes.data, o.ctypes.data, qp, kp, vp_, btp, bt.shape[1],
                                     clp, S, Hq, hkv, D, bs, nb, float(scale), dtype, partition_tokens, max_parts)
    _check(st, "decode_partitions")
    return m, l, o


def merge_partitions(m, l, o):
    m, mp = _c(m, np.float64)
    l, lp = _c(l, np.float64)
    o, op = _c(o, np.float64)
    S, Hq, P, D = o.shape
    out = np.empty((S, Hq, D))
    lib().pao_merge_partitions(out.ctypes.data, mp, lp, op, S * Hq, P, D)
    return out


def prefill_chunk(q, k_cache, v_cache, block_tables, query_start_loc, seq_lens, scale: float, dtype: int):
    """fp64 prefill chunks with the bottom-right causal mask. Returns out [sum q_len, Hq, D]."""
    q, qp = _c(q, np.uint16)
    k, kp = _c(k_cache, np.uint16)
    v, vp_ = _c(v_cache, np.uint16)
    bt, btp = _c(block_tables, np.int32)
    qsl, qslp = _c(query_start_loc, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    T, Hq, D = q.shape
    nb, bs, hkv, _ = k.shape
    out = np.zeros((T, Hq, D), dtype=np.float64)
    st = lib().pao_prefill_chunk(out.ctypes.data, qp, kp, vp_, btp, bt.shape[1], qslp, slp, sl.size, Hq, hkv, D, bs,
                                 nb, float(scale), dtype)
    _check(st, "prefill_chunk")
    return out


def naive_contiguous(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: int):
    """Materialise each sequence's K/V contiguously, then textbook attention (fp64)."""
    q, qp = _c(q, np.uint16)
    k, kp = _c(k_cache, np.uint16)
    v, vp_ = _c(v_cache, np.uint16)
    bt, btp = _c(block_tables, np.int32)
    cl, clp = _c(context_lens, np.int32)
    S, Hq, D = q.shape
    nb, bs, hkv, _ = k.shape
    out = np.empty((S, Hq, D), dtype=np.float64)
    st = lib().pao_naive_contiguous(out.ctypes.data, qp, kp, vp_, btp, bt.shape[1], clp, S, Hq, hkv, D, bs, nb,
                                    float(scale), dtype)
    _check(st, "naive_contiguous")
    return out
