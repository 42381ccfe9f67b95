"""Python binding of libpagedattn (include/pagedattn.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks that they are contiguous and of
the expected dtypes, and forwards their device pointers and sizes to the C ABI through
ctypes on the caller's current CUDA stream.  All computation happens in the library's
CUDA kernels; there is no fallback of any kind.  If the shared library has not been
built, the first call builds it with nvcc (see _build.py) or raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

PA_F16, PA_BF16 = 0, 1
PA_OK = 0
PA_DEVERR_SLOT, PA_DEVERR_BLOCK, PA_DEVERR_LENGTH, PA_DEVERR_TIMEOUT, PA_DEVERR_POSITION = 1, 2, 4, 8, 16
DEFAULT_PARTITION_TOKENS = 256

# names the header declares; the CPU test checks that the library exports each one
EXPORTED = (
    "pa_reshape_and_cache", "pa_decode_workspace_size", "pa_decode", "pa_decode_plan", "pa_decode_v1",
    "pa_decode_splitk", "pa_prefill_chunk", "pa_device_errors", "pa_status_string", "pa_version",
    "pa_decode_splitk_static", "pa_rope_table", "pa_rope_reshape_and_cache", "pa_decode_shared_prefix",
    "pa_decode_shared_prefix_workspace_size", "pa_prefill_chunk_small_m", "pa_decode_write",
)
STATIC_SCRATCH_BYTES = 16 << 20


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.library_path()


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpagedattn.so (building it first if needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libpagedattn is not built ({path}); run paged_kv_cache_232_gb300._build.build()")
        path = _build.build()
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, vp]
    L.pa_reshape_and_cache.restype = i32
    L.pa_rope_table.argtypes = [vp, i64, i32, ctypes.c_double]
    L.pa_rope_table.restype = i32
    L.pa_rope_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i64, i64, i32, vp]
    L.pa_rope_reshape_and_cache.restype = i32
    L.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.pa_decode_workspace_size.restype = sz
    L.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32, vp, sz, vp]
    L.pa_decode.restype = i32
    L.pa_decode_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32)]
    L.pa_decode_plan.restype = i32
    L.pa_decode_write.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32, vp, vp, vp,
                                  vp, sz, vp]
    L.pa_decode_write.restype = i32
    L.pa_decode_v1.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp]
    L.pa_decode_v1.restype = i32
    L.pa_decode_splitk.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32, i32, vp,
                                   sz, vp]
    L.pa_decode_splitk.restype = i32
    L.pa_decode_splitk_static.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32,
                                          i32, vp]
    L.pa_decode_splitk_static.restype = i32
    L.pa_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32,
                                          i32, i32, vp, sz, vp]
    L.pa_decode_shared_prefix.restype = i32
    L.pa_decode_shared_prefix_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.pa_decode_shared_prefix_workspace_size.restype = sz
    L.pa_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i64, f32, i32, vp]
    L.pa_prefill_chunk.restype = i32
    L.pa_prefill_chunk_small_m.argtypes = L.pa_prefill_chunk.argtypes
    L.pa_prefill_chunk_small_m.restype = i32
    L.pa_device_errors.argtypes = [i32]
    L.pa_device_errors.restype = i32
    L.pa_status_string.argtypes = [i32]
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_version.restype = i32
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().pa_status_string(status).decode()


# ------------------------------------------------------------------ marshalling helpers


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float16:
        return PA_F16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _dev(t, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = _torch().cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str):
    if status != PA_OK:
        raise PagedAttnError(status, what)


def _cache_dims(k_cache):
    nb, bs, hkv, d = k_cache.shape
    return int(nb), int(bs), int(hkv), int(d)


# ------------------------------------------------------------------ entry points


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Scatter key/value [N, Hkv, D] into the caches [NB, bs, Hkv, D] at slot_mapping [N] (int64, -1 skips)."""
    torch = _torch()
    dt = _dtype_code(key)
    nb, bs, hkv, d = _cache_dims(k_cache)
    n = int(key.shape[0])
    st = load().pa_reshape_and_cache(_dev(key, "key", key.dtype), _dev(value, "value", key.dtype),
                                     _dev(k_cache, "k_cache", key.dtype), _dev(v_cache, "v_cache", key.dtype),
                                     _dev(slot_mapping, "slot_mapping", torch.int64), n, hkv, d, bs, nb, dt,
                                     _stream(stream, key.device))
    _check(st, "pa_reshape_and_cache")


def pa_rope_table(max_position: int, head_dim: int, theta: float):
    """The float32 [max_position, head_dim] cos / sin table (host numpy array) the fused RoPE
    write reads; copy it to the device once."""
    import numpy as np
    out = np.empty((int(max_position), int(head_dim)), dtype=np.float32)
    _check(load().pa_rope_table(out.ctypes.data, int(max_position), int(head_dim), float(theta)), "pa_rope_table")
    return out


def rope_cos_sin(max_position: int, head_dim: int, theta: float, device="cuda"):
    """pa_rope_table's output as a device tensor."""
    return _torch().from_numpy(pa_rope_table(max_position, head_dim, theta)).to(device)


def pa_rope_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, positions, cos_sin, q=None,
                              stream=None) -> None:
    """Rotate key [N, Hkv, D] by positions [N] (int64) with the cos_sin table [max_position, D]
    (float32) and scatter it, and value unchanged, into the caches at slot_mapping [N] (int64,
    -1 skips); q [N, Hq, D], if given, is rotated in place."""
    torch = _torch()
    dt = _dtype_code(key)
    nb, bs, hkv, d = _cache_dims(k_cache)
    n = int(key.shape[0])
    qp, hq = (None, 0) if q is None else (_dev(q, "q", key.dtype), int(q.shape[1]))
    st = load().pa_rope_reshape_and_cache(
        qp, _dev(key, "key", key.dtype), _dev(value, "value", key.dtype), _dev(k_cache, "k_cache", key.dtype),
        _dev(v_cache, "v_cache", key.dtype), _dev(slot_mapping, "slot_mapping", torch.int64),
        _dev(positions, "positions", torch.int64), _dev(cos_sin, "cos_sin", torch.float32), n, hq, hkv, d, bs, nb,
        int(cos_sin.shape[0]), dt, _stream(stream, key.device))
    _check(st, "pa_rope_reshape_and_cache")


def pa_decode_workspace_size(num_seqs: int, n_q_heads: int, head_dim: int, max_context_len: int,
                             partition_tokens: int = 0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len, partition_tokens))


def pa_decode_plan(num_seqs: int, n_q_heads: int, n_kv_heads: int, head_dim: int, block_size: int,
                   max_context_len: int, dtype: int = PA_BF16):
    """(1 = one-pass kernel | 2 = split-K, partition_tokens) for these sizes on the current device."""
    pt = ctypes.c_int(0)
    r = load().pa_decode_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_context_len, dtype,
                              ctypes.byref(pt))
    if r < 0:
        raise PagedAttnError(r, "pa_decode_plan")
    return r, pt.value


def _decode_common(out, q, k_cache, v_cache, block_tables, context_lens):
    torch = _torch()
    dt = _dtype_code(q)
    nb, bs, hkv, d = _cache_dims(k_cache)
    S, hq, d2 = (int(x) for x in q.shape)
    if d2 != d or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out/cache head_dim mismatch")
    ptrs = (_dev(out, "out", q.dtype), _dev(q, "q", q.dtype), _dev(k_cache, "k_cache", q.dtype),
            _dev(v_cache, "v_cache", q.dtype), _dev(block_tables, "block_tables", torch.int32),
            _dev(context_lens, "context_lens", torch.int32))
    return dt, nb, bs, hkv, d, S, hq, int(block_tables.shape[1]), ptrs


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
              workspace=None, stream=None) -> None:
    """Decode attention with the library's dispatcher choosing one-pass or split-K."""
    dt, nb, bs, hkv, d, S, hq, mb, (po, pq, pk, pv, pbt, pcl) = _decode_common(out, q, k_cache, v_cache, block_tables,
                                                                             context_lens)
    wp, wb = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    st = load().pa_decode(po, pq, pk, pv, pbt, mb, pcl, int(max_context_len), S, hq, hkv, d, bs, nb, float(scale), dt,
                          wp, wb, _stream(stream, q.device))
    _check(st, "pa_decode")


def pa_decode_write(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                    key, value, slot_mapping, workspace=None, stream=None) -> None:
    """One decode step: key / value [S, Hkv, D] (sequence s's new token) into the caches at
    slot_mapping [S] (int64, -1 skips; otherwise the slot of token context_lens[s] - 1), then the
    decode as pa_decode, over contexts that include those rows."""
    torch = _torch()
    dt, nb, bs, hkv, d, S, hq, mb, (po, pq, pk, pv, pbt, pcl) = _decode_common(out, q, k_cache, v_cache, block_tables,
                                                                             context_lens)
    if tuple(key.shape) != (S, hkv, d) or tuple(value.shape) != (S, hkv, d):
        raise ValueError("key / value must be [num_seqs, n_kv_heads, head_dim]")
    if tuple(slot_mapping.shape) != (S,):
        raise ValueError("slot_mapping must hold one slot per sequence")
    wp, wb = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    st = load().pa_decode_write(po, pq, pk, pv, pbt, mb, pcl, int(max_context_len), S, hq, hkv, d, bs, nb, float(scale),
                                dt, _dev(key, "key", q.dtype), _dev(value, "value", q.dtype),
                                _dev(slot_mapping, "slot_mapping", torch.int64), wp, wb, _stream(stream, q.device))
    _check(st, "pa_decode_write")


def pa_decode_v1(out, q, k_cache, v_cache, block_tables, context_lens, scale: float, stream=None) -> None:
    """One-pass decode: one CTA per (sequence, KV head) over the whole context."""
    dt, nb, bs, hkv, d, S, hq, mb, (po, pq, pk, pv, pbt, pcl) = _decode_common(out, q, k_cache, v_cache, block_tables,
                                                                             context_lens)
    st = load().pa_decode_v1(po, pq, pk, pv, pbt, mb, pcl, S, hq, hkv, d, bs, nb, float(scale), dt,
                             _stream(stream, q.device))
    _check(st, "pa_decode_v1")


def pa_decode_splitk(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                     workspace, partition_tokens: int = 0, stream=None) -> None:
    """Split-K decode over partition_tokens-token pieces plus the merge kernel."""
    dt, nb, bs, hkv, d, S, hq, mb, (po, pq, pk, pv, pbt, pcl) = _decode_common(out, q, k_cache, v_cache, block_tables,
                                                                             context_lens)
    wp, wb = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    st = load().pa_decode_splitk(po, pq, pk, pv, pbt, mb, pcl, int(max_context_len), S, hq, hkv, d, bs, nb,
                                 float(scale), dt, int(partition_tokens), wp, wb, _stream(stream, q.device))
    _check(st, "pa_decode_splitk")


def pa_decode_splitk_static(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                            scale: float, partition_tokens: int = 0, stream=None) -> None:
    """Split-K decode for callers that cannot allocate device memory: the partials live in a
    fixed STATIC_SCRATCH_BYTES array inside the library (shared by all calls, so calls that
    overlap on the GPU race).  Raises PagedAttnError(PA_ERR_WORKSPACE) when the sizes need
    more than that."""
    dt, nb, bs, hkv, d, S, hq, mb, (po, pq, pk, pv, pbt, pcl) = _decode_common(out, q, k_cache, v_cache, block_tables,
                                                                             context_lens)
    st = load().pa_decode_splitk_static(po, pq, pk, pv, pbt, mb, pcl, int(max_context_len), S, hq, hkv, d, bs, nb,
                                        float(scale), dt, int(partition_tokens), _stream(stream, q.device))
    _check(st, "pa_decode_splitk_static")


def pa_decode_shared_prefix_workspace_size(num_seqs: int, n_q_heads: int, head_dim: int, max_context_len: int,
                                           prefix_tokens: int) -> int:
    return int(load().pa_decode_shared_prefix_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len,
                                                             prefix_tokens))


def pa_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len: int, scale: float,
                            prefix_tokens: int, workspace, prefix_piece_tokens: int = 0, stream=None) -> None:
    """Decode for sequences whose first prefix_tokens tokens are the same cache blocks: the prefix
    part once per KV head on the tensor cores, the rest per sequence, merged."""
    dt, nb, bs, hkv, d, S, hq, mb, (po, pq, pk, pv, pbt, pcl) = _decode_common(out, q, k_cache, v_cache, block_tables,
                                                                             context_lens)
    wp, wb = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None else (None, 0)
    st = load().pa_decode_shared_prefix(po, pq, pk, pv, pbt, mb, pcl, int(max_context_len), S, hq, hkv, d, bs, nb,
                                        float(scale), dt, int(prefix_tokens), int(prefix_piece_tokens), wp, wb,
                                        _stream(stream, q.device))
    _check(st, "pa_decode_shared_prefix")


def pa_prefill_chunk(out, q, k_cache, v_cache, block_tables, query_start_loc, seq_lens, max_q_len: int, scale: float,
                     stream=None, small_m: bool = False) -> None:
    """Prefill chunks (bottom-right causal over their cached context) on the tcgen05 tensor cores;
    small_m=True calls pa_prefill_chunk_small_m (M = 64 tiles for units of at most 64 rows)."""
    torch = _torch()
    dt = _dtype_code(q)
    nb, bs, hkv, d = _cache_dims(k_cache)
    T, hq, d2 = (int(x) for x in q.shape)
    if d2 != d or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out/cache head_dim mismatch")
    C = int(seq_lens.shape[0])
    fn = load().pa_prefill_chunk_small_m if small_m else load().pa_prefill_chunk
    st = fn(_dev(out, "out", q.dtype), _dev(q, "q", q.dtype), _dev(k_cache, "k_cache", q.dtype),
            _dev(v_cache, "v_cache", q.dtype), _dev(block_tables, "block_tables", torch.int32),
            int(block_tables.shape[1]), _dev(query_start_loc, "query_start_loc", torch.int32),
            _dev(seq_lens, "seq_lens", torch.int32), C, int(max_q_len), hq, hkv, d, bs, nb,
            float(scale), dt, _stream(stream, q.device))
    _check(st, "pa_prefill_chunk_small_m" if small_m else "pa_prefill_chunk")


def pa_device_errors(clear: bool = True) -> int:
    """PA_DEVERR_* bits recorded by the kernels on the current device (synchronises)."""
    r = load().pa_device_errors(1 if clear else 0)
    if r < 0:
        raise PagedAttnError(r, "pa_device_errors")
    return r


def version() -> int:
    return int(load().pa_version())
