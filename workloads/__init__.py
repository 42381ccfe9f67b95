"""Seeded synthetic inputs for the paged-KV-cache kernels, their tests and the bench.

This module only produces inputs: bit patterns of fp16/bf16 tensors, lengths,
block tables and slot mappings.  It holds none of the attention arithmetic; the
CUDA library and the CPU oracle both consume what it makes, and neither imports
the other.

Random numbers come from ``wlgen.c`` (SplitMix64 -> Box-Muller normals ->
float32 -> round-to-nearest-even fp16/bf16; Lemire bounded integers; Fisher-Yates
permutations).  Every tensor has its own sub-stream derived from the workload
seed, and every normal element is addressable by its flat index, so a sampled
slice of a full-size workload can be regenerated on its own.

Workload shapes follow the three pages' descriptions (MiniLLM Runtime
"CUDA PagedAttention scope"; mini_engine "Custom CUDA kernels" and "Results";
miniserve "Engine"): block size 16, cache layout [num_blocks, block_size,
n_kv_heads, head_dim], block tables of physical block ids, slot =
block_id * block_size + offset, -1 marking a padded slot.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wlgen.c")
_BUILD = os.path.join(_HERE, "_build")

F16, BF16 = 0, 1
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}

# sub-stream tags (stable: changing one changes every workload)
TAG_LENS, TAG_PERM, TAG_Q, TAG_K, TAG_V, TAG_KEY, TAG_VALUE, TAG_PAD, TAG_CTX, TAG_PQ = range(1, 11)


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def build(force: bool = False) -> str:
    """Compile wlgen.c with gcc into workloads/_build; returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    so = os.path.join(_BUILD, f"libwlgen_{_src_hash()}.so")
    if force or not os.path.exists(so):
        tmp = so + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
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
        u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
        vp = ctypes.c_void_p
        L.wl_splitmix64_at.argtypes = [u64, u64]
        L.wl_splitmix64_at.restype = u64
        L.wl_splitmix64_fill.argtypes = [u64, u64, i64, vp]
        L.wl_derive_seed.argtypes = [u64, u64]
        L.wl_derive_seed.restype = u64
        L.wl_normal_f64_at.argtypes = [u64, u64]
        L.wl_normal_f64_at.restype = ctypes.c_double
        L.wl_normal_bits.argtypes = [u64, u64, i64, i32, vp]
        L.wl_normal_f32.argtypes = [u64, u64, i64, vp]
        L.wl_uniform_ints.argtypes = [u64, i64, i64, i64, vp]
        L.wl_permutation.argtypes = [u64, i64, vp]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def derive_seed(base: int, tag: int) -> int:
    return int(lib().wl_derive_seed(base & (2**64 - 1), tag))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    lib().wl_splitmix64_fill(seed, start, count, _ptr(out))
    return out


def normal_bits(seed: int, count: int, dtype: int, start: int = 0, out: Optional[np.ndarray] = None) -> np.ndarray:
    """Normals start..start+count of the stream, as fp16 (dtype 0) or bf16 (dtype 1) bit patterns."""
    if out is None:
        out = np.empty(count, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size == count
    lib().wl_normal_bits(seed, start, count, dtype, _ptr(out))
    return out


def normal_f32(seed: int, count: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    lib().wl_normal_f32(seed, start, count, _ptr(out))
    return out


def uniform_ints(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(count, dtype=np.int64)
    if count:
        lib().wl_uniform_ints(seed, count, lo, hi, _ptr(out))
    return out


def permutation(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if n:
        lib().wl_permutation(seed, n, _ptr(out))
    return out


def bits_to_float(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact widening of fp16/bf16 bit patterns to float32 (input plumbing for tests)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- pools


@dataclass
class PagedPool:
    """A block-paged K/V pool: k/v caches [NB, bs, Hkv, D] as fp16/bf16 bits."""
    dtype: int
    num_blocks: int
    block_size: int
    n_kv_heads: int
    head_dim: int
    k_cache: np.ndarray
    v_cache: np.ndarray
    poison_block: int
    valid: np.ndarray  # bool [NB, bs]: slot holds data some sequence owns


@dataclass
class DecodeBatch:
    q: np.ndarray               # uint16 [S, Hq, D]
    block_tables: np.ndarray    # int32 [S, MB]
    context_lens: np.ndarray    # int32 [S]
    n_q_heads: int
    scale: float

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


@dataclass
class WriteBatch:
    key: np.ndarray             # uint16 [N, Hkv, D]
    value: np.ndarray           # uint16 [N, Hkv, D]
    slot_mapping: np.ndarray    # int64 [N], -1 = padded


@dataclass
class PrefillBatch:
    q: np.ndarray               # uint16 [sum q_len, Hq, D]
    block_tables: np.ndarray    # int32 [C, MB]
    query_start_loc: np.ndarray  # int32 [C+1]
    seq_lens: np.ndarray        # int32 [C]  (kv length = cached context + q_len)
    n_q_heads: int
    scale: float

    @property
    def num_chunks(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_q_len(self) -> int:
        ql = np.diff(self.query_start_loc)
        return int(ql.max()) if ql.size else 0


@dataclass
class Workload:
    name: str
    seed: int
    pool: PagedPool
    decode: Optional[DecodeBatch] = None
    write: Optional[WriteBatch] = None
    prefill: Optional[PrefillBatch] = None
    meta: Dict = field(default_factory=dict)


class _BlockAllocator:
    """Hands out physical block ids in the order of a seeded permutation of the pool."""

    def __init__(self, seed: int, num_blocks: int):
        self.order = permutation(derive_seed(seed, TAG_PERM), num_blocks)
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        ids = self.order[self.next:self.next + n]
        assert ids.size == n, "pool too small"
        self.next += n
        return ids


def _fill_pool(seed: int, dtype: int, nb: int, bs: int, hkv: int, d: int, valid: np.ndarray,
               poison_block: int, nan_canaries: bool) -> PagedPool:
    n = nb * bs * hkv * d
    k = normal_bits(derive_seed(seed, TAG_K), n, dtype).reshape(nb, bs, hkv, d)
    v = normal_bits(derive_seed(seed, TAG_V), n, dtype).reshape(nb, bs, hkv, d)
    if nan_canaries:
        dead = ~valid
        k[dead] = NAN_BITS[dtype]
        v[dead] = NAN_BITS[dtype]
    return PagedPool(dtype, nb, bs, hkv, d, k, v, poison_block, valid)


def _ceil_div(a, b):
    return -(-a // b)


def build_workload(name: str, seed: int, *, dtype: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                   block_size: int = 16,
                   decode_lens: Sequence[int] = (),
                   shared_prefix_blocks: int = 0,
                   max_blocks_per_seq: Optional[int] = None,
                   write_rows: bool = False, n_padded: int = 0,
                   prefill_q_lens: Sequence[int] = (), prefill_ctx_lens: Sequence[int] = (),
                   prefill_max_blocks: Optional[int] = None,
                   extra_blocks: int = 0, pool_blocks: Optional[int] = None,
                   nan_canaries: bool = True, scale: Optional[float] = None) -> Workload:
    """General builder: decode sequences (optionally sharing a prefix), an optional
    KV-write batch (one new row per decode sequence, at its last position) and
    optional prefill chunks, all over one paged pool with NaN canaries in every
    slot no sequence owns and a NaN-filled poison block padding the tables."""
    bs = block_size
    decode_lens = [int(x) for x in decode_lens]
    ql = [int(x) for x in prefill_q_lens]
    cl = [int(x) for x in prefill_ctx_lens]
    assert len(ql) == len(cl)
    need = shared_prefix_blocks
    need += sum(max(0, _ceil_div(L, bs) - shared_prefix_blocks) for L in decode_lens)
    need += sum(_ceil_div(c + q, bs) for q, c in zip(ql, cl))
    need += 1 + extra_blocks  # poison block + unused blocks
    nb = pool_blocks if pool_blocks is not None else need
    assert nb >= need
    alloc = _BlockAllocator(seed, nb)
    poison = int(alloc.take(1)[0])
    valid = np.zeros((nb, bs), dtype=bool)
    scale = float(1.0 / np.sqrt(head_dim)) if scale is None else float(scale)

    decode = write = prefill = None
    if decode_lens:
        S = len(decode_lens)
        mb = max_blocks_per_seq or max([_ceil_div(L, bs) for L in decode_lens] + [shared_prefix_blocks])
        bt = np.full((S, mb), poison, dtype=np.int32)
        prefix = alloc.take(shared_prefix_blocks) if shared_prefix_blocks else np.empty(0, np.int64)
        for s, L in enumerate(decode_lens):
            nblk = _ceil_div(L, bs)
            assert max(nblk, shared_prefix_blocks) <= mb
            # every row lists the whole shared prefix, also when its own context ends inside it
            ids = np.concatenate([prefix, alloc.take(max(0, nblk - shared_prefix_blocks))])
            bt[s, :ids.size] = ids
            for t0 in range(0, L, bs):
                valid[ids[t0 // bs], : min(bs, L - t0)] = True
        q = normal_bits(derive_seed(seed, TAG_Q), S * n_q_heads * head_dim, dtype).reshape(S, n_q_heads, head_dim)
        decode = DecodeBatch(q, bt, np.asarray(decode_lens, dtype=np.int32), n_q_heads, scale)
        if write_rows:
            n = S * n_kv_heads * head_dim
            key = normal_bits(derive_seed(seed, TAG_KEY), n, dtype).reshape(S, n_kv_heads, head_dim)
            val = normal_bits(derive_seed(seed, TAG_VALUE), n, dtype).reshape(S, n_kv_heads, head_dim)
            last = np.asarray(decode_lens, dtype=np.int64) - 1
            slots = bt[np.arange(S), last // bs].astype(np.int64) * bs + last % bs
            if n_padded:
                pad_rows = permutation(derive_seed(seed, TAG_PAD), S)[:n_padded]
                slots[pad_rows] = -1
            write = WriteBatch(key, val, slots)
    if ql:
        C = len(ql)
        kv = [c + q for q, c in zip(ql, cl)]
        mbp = prefill_max_blocks or max(_ceil_div(x, bs) for x in kv)
        pbt = np.full((C, mbp), poison, dtype=np.int32)
        for c in range(C):
            nblk = _ceil_div(kv[c], bs)
            ids = alloc.take(nblk)
            pbt[c, :nblk] = ids
            for t0 in range(0, kv[c], bs):
                valid[ids[t0 // bs], : min(bs, kv[c] - t0)] = True
        qsl = np.zeros(C + 1, dtype=np.int32)
        qsl[1:] = np.cumsum(ql)
        tot = int(qsl[-1])
        pq = normal_bits(derive_seed(seed, TAG_PQ), tot * n_q_heads * head_dim, dtype).reshape(tot, n_q_heads, head_dim)
        prefill = PrefillBatch(pq, pbt, qsl, np.asarray(kv, dtype=np.int32), n_q_heads, scale)

    pool = _fill_pool(seed, dtype, nb, bs, n_kv_heads, head_dim, valid, poison, nan_canaries)
    return Workload(name, seed, pool, decode, write, prefill,
                    meta=dict(dtype=dtype, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                              block_size=bs, shared_prefix_tokens=shared_prefix_blocks * bs))


# ----------------------------------------------------------------- the five workloads

WORKLOAD_NAMES = {
    1: "single-request fp16 decode, 2/2 heads, hd 64, ctx 128, 64-block pool",
    2: "Qwen3-0.6B-shaped decode batch: 64 seqs bf16, 16/8 heads, hd 128, ctx U[100,2048]",
    3: "long-context split-K decode: 4 seqs bf16, 32/8 heads, hd 128, ctx 32768",
    4: "full decode step at batch 256: KV write of 256 rows (10% padded -1) + decode, 16/8 heads, ctx U[100,2048]",
    5: "mixed batch: 128 decodes sharing a 1024-token prefix + 8x512-token prefill chunks over 0-4096 cached tokens",
}


def workload_seed(k: int) -> int:
    return 232_000 + k


def make_workload(k: int, *, nan_canaries: bool = True) -> Workload:
    seed = workload_seed(k)
    if k == 1:
        return build_workload("single", seed, dtype=F16, n_q_heads=2, n_kv_heads=2, head_dim=64,
                              decode_lens=[128], pool_blocks=64, nan_canaries=nan_canaries, scale=1.0 / 8.0)
    if k == 2:
        lens = uniform_ints(derive_seed(seed, TAG_LENS), 64, 100, 2048)
        return build_workload("decode64", seed, dtype=BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                              decode_lens=lens, max_blocks_per_seq=128, nan_canaries=nan_canaries)
    if k == 3:
        return build_workload("long4", seed, dtype=BF16, n_q_heads=32, n_kv_heads=8, head_dim=128,
                              decode_lens=[32768] * 4, max_blocks_per_seq=2048, nan_canaries=nan_canaries)
    if k == 4:
        lens = uniform_ints(derive_seed(seed, TAG_LENS), 256, 100, 2048)
        return build_workload("step256", seed, dtype=BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                              decode_lens=lens, max_blocks_per_seq=128, write_rows=True,
                              n_padded=int(round(0.1 * 256)), nan_canaries=nan_canaries)
    if k == 5:
        suffix = uniform_ints(derive_seed(seed, TAG_LENS), 128, 1, 1024)
        ctx = [0] + [int(x) for x in uniform_ints(derive_seed(seed, TAG_CTX), 6, 0, 4096)] + [4096]
        return build_workload("mixed", seed, dtype=BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                              decode_lens=1024 + suffix, shared_prefix_blocks=64, max_blocks_per_seq=128,
                              prefill_q_lens=[512] * 8, prefill_ctx_lens=ctx, nan_canaries=nan_canaries)
    raise ValueError(f"no workload {k}")


def write_rows_case(seed: int, n_rows: int, *, n_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                    dtype: int = BF16, pad_frac: float = 0.1, extra_blocks: int = 8,
                    nan_canaries: bool = False) -> Workload:
    """A bandwidth-scale KV write: n_rows new rows scattered to distinct random slots
    of a pool sized for them, pad_frac of them marked -1."""
    bs = block_size
    nb = _ceil_div(n_rows, bs) + 1 + extra_blocks
    pool_valid = np.ones((nb, bs), dtype=bool)
    slots = permutation(derive_seed(seed, TAG_PERM), nb * bs)[:n_rows].astype(np.int64)
    pad = int(round(pad_frac * n_rows))
    if pad:
        slots[permutation(derive_seed(seed, TAG_PAD), n_rows)[:pad]] = -1
    n = n_rows * n_kv_heads * head_dim
    key = normal_bits(derive_seed(seed, TAG_KEY), n, dtype).reshape(n_rows, n_kv_heads, head_dim)
    val = normal_bits(derive_seed(seed, TAG_VALUE), n, dtype).reshape(n_rows, n_kv_heads, head_dim)
    pool = _fill_pool(seed, dtype, nb, bs, n_kv_heads, head_dim, pool_valid, -1, nan_canaries)
    return Workload(f"write{n_rows}", seed, pool, write=WriteBatch(key, val, slots),
                    meta=dict(dtype=dtype, n_kv_heads=n_kv_heads, head_dim=head_dim, block_size=bs))


def unified_batch(w: "Workload") -> PrefillBatch:
    """The mixed batch as one list of chunks for a single prefill launch: each decode sequence
    as a chunk of one query row whose kv length is its context length, then the prefill chunks.
    Rows keep their order (decode rows first), tables are padded to the wider of the two."""
    b, pre = w.decode, w.prefill
    mb = max(b.block_tables.shape[1], pre.block_tables.shape[1])
    pad = lambda t: np.pad(t, ((0, 0), (0, mb - t.shape[1])), constant_values=0).astype(np.int32)
    S = b.num_seqs
    qsl = np.concatenate([np.arange(S + 1, dtype=np.int64), S + pre.query_start_loc[1:].astype(np.int64)])
    return PrefillBatch(q=np.concatenate([b.q, pre.q]), block_tables=np.concatenate([pad(b.block_tables),
                                                                                     pad(pre.block_tables)]),
                        query_start_loc=qsl.astype(np.int32),
                        seq_lens=np.concatenate([b.context_lens, pre.seq_lens]).astype(np.int32),
                        n_q_heads=pre.n_q_heads, scale=pre.scale)
