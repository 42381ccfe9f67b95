"""The C-ABI library builds, loads without a GPU and exports every entry point that
include/pagedattn.h declares; host-only calls (sizes, status strings, argument
validation that rejects before touching the device) behave as documented."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_232_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(pa_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    return pa.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"pa_reshape_and_cache", "pa_decode", "pa_prefill_chunk"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert names == set(pa.EXPORTED)


def test_host_only_calls(lib):
    assert pa.version() >= 100
    assert pa.status_string(0) == "ok"
    assert pa.status_string(-7).startswith("split-K workspace")
    # one piece needs no workspace; several pieces need m, l (256-byte aligned), o and a 256-byte
    # control region (the dynamic grid's piece counter), with room for three pieces more than the
    # uniform split (the dynamic grid's tail pieces)
    assert pa.pa_decode_workspace_size(4, 32, 128, 256) == 0
    rows = 4 * 32 * (128 + 3)
    expect = 2 * ((rows * 4 + 255) // 256 * 256) + (rows * 128 * 4 + 255) // 256 * 256 + 256
    assert pa.pa_decode_workspace_size(4, 32, 128, 32768) == expect


def test_validation_rejects_before_any_device_work(lib):
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # n_q_heads not a multiple of n_kv_heads
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 6, 4, 128, 16, 10, 0.1, 1, None) == -2
    # unsupported head_dim / block_size / dtype / group size
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 8, 8, 80, 16, 10, 0.1, 1, None) == -3
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 8, 8, 128, 24, 10, 0.1, 1, None) == -3
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 8, 8, 128, 16, 10, 0.1, 7, None) == -3
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 48, 3, 128, 16, 10, 0.1, 1, None) == -3
    # head_dim 256: group size up to 4
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 64, 8, 256, 16, 10, 0.1, 1, None) == -3
    assert lib.pa_prefill_chunk(vp, vp, vp, vp, vp, 8, vp, vp, 1, 1, 64, 8, 256, 16, 10, 0.1, 1, None) == -3
    # null pointers, misalignment
    assert lib.pa_decode_v1(None, vp, vp, vp, vp, 8, vp, 1, 8, 8, 128, 16, 10, 0.1, 1, None) == -1
    assert lib.pa_decode_v1(ctypes.c_void_p(8), vp, vp, vp, vp, 8, vp, 1, 8, 8, 128, 16, 10, 0.1, 1, None) == -6
    # max_context_len beyond the table's capacity
    assert lib.pa_decode(vp, vp, vp, vp, vp, 8, vp, 129, 1, 8, 8, 128, 16, 10, 0.1, 1, None, 0, None) == -5
    # empty batches launch nothing
    assert lib.pa_decode_v1(None, None, None, None, None, 8, None, 0, 8, 8, 128, 16, 10, 0.1, 1, None) == 0
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 128, 16, 10, 1, None) == 0
    assert lib.pa_prefill_chunk(None, None, None, None, None, 8, None, None, 0, 0, 8, 8, 128, 16, 10, 0.1, 1,
                                None) == 0
    # write: a row of 1 head x 3 columns (6 bytes) is not a whole number of 16-byte chunks
    assert lib.pa_reshape_and_cache(vp, vp, vp, vp, vp, 4, 1, 3, 16, 10, 1, None) == -3


def test_decode_write_validation_rejects_before_any_device_work(lib):
    """pa_decode_write: the write's own arguments are checked before the decode's plan (no device
    call): a missing key / value / slot_mapping, a misaligned key, a context bound past the table."""
    vp = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    call = lambda key=vp, val=vp, sm=vp, maxL=100: lib.pa_decode_write(
        vp, vp, vp, vp, vp, 8, vp, maxL, 1, 8, 8, 128, 16, 10, 0.1, 1, key, val, sm, vp, 1 << 30, None)
    assert call(key=None) == -1
    assert call(val=None) == -1
    assert call(sm=None) == -1
    assert call(key=ctypes.c_void_p(8)) == -6
    assert call(maxL=129) == -5
    # nothing to decode: nothing written either
    assert lib.pa_decode_write(None, None, None, None, None, 8, None, 0, 0, 8, 8, 128, 16, 10, 0.1, 1, None, None,
                               None, None, 0, None) == 0


def test_rope_table_matches_the_formula_and_validates(lib):
    """pa_rope_table is host code: row m = [cos(m f_i) ..., sin(m f_i) ...], f_i = theta^(-2i/D),
    computed in double and stored as float; compared with numpy's float64 cos / sin."""
    import numpy as np
    t = pa.pa_rope_table(257, 64, 1.0e6)
    i = np.arange(32)
    f = 1.0e6 ** (-2.0 * i / 64)
    m = np.arange(257)[:, None]
    want = np.concatenate([np.cos(m * f), np.sin(m * f)], axis=1).astype(np.float32)
    assert np.array_equal(t, want)
    buf = (ctypes.c_float * 16)()
    assert lib.pa_rope_table(None, 2, 8, 1e4) == -1
    assert lib.pa_rope_table(buf, 2, 7, 1e4) == -2
    assert lib.pa_rope_table(buf, 0, 8, 1e4) == -2
    assert lib.pa_rope_table(buf, 2, 8, -1.0) == -2


def test_rope_write_validation_rejects_before_any_device_work(lib):
    vp = ctypes.c_void_p(16)
    args = lambda q=vp, d=128, n=4, dt=1, mp=100: (q, vp, vp, vp, vp, vp, vp, vp, n, 16, 8, d, 16, 10, mp, dt, None)
    assert lib.pa_rope_reshape_and_cache(*args(d=80)) == -3          # head_dim
    assert lib.pa_rope_reshape_and_cache(*args(dt=7)) == -3          # dtype
    assert lib.pa_rope_reshape_and_cache(*args(mp=0)) == -2          # empty table
    assert lib.pa_rope_reshape_and_cache(*args(n=0)) == 0            # nothing to do
    assert lib.pa_rope_reshape_and_cache(ctypes.c_void_p(8), vp, vp, vp, vp, vp, vp, vp, 4, 16, 8, 128, 16, 10,
                                         100, 1, None) == -6         # q misaligned
    assert lib.pa_rope_reshape_and_cache(vp, None, vp, vp, vp, vp, vp, vp, 4, 16, 8, 128, 16, 10, 100, 1,
                                         None) == -1                 # key NULL


def test_shared_prefix_sizes_and_validation(lib):
    """pa_decode_shared_prefix: with nothing shared its workspace is pa_decode's; with a shared
    prefix it is the prefix pass's partials (pieces of 128 tokens at most: m, l, o regions, each
    256-byte aligned) plus the split-K workspace of the tokens past the prefix.  Bad sizes are
    rejected on the host."""
    ws = pa.pa_decode_shared_prefix_workspace_size
    assert ws(4, 32, 128, 32768, 0) == pa.pa_decode_workspace_size(4, 32, 128, 32768)
    assert ws(4, 32, 128, 32768, 15) == pa.pa_decode_workspace_size(4, 32, 128, 32768)
    rows = 128 * 16 * (1024 // 128)
    pf = 2 * ((rows * 4 + 255) // 256 * 256) + (rows * 128 * 4 + 255) // 256 * 256 + 256
    assert ws(128, 16, 128, 2048, 1024) == pf + pa.pa_decode_workspace_size(128, 16, 128, 2048 - 1024)
    # only whole 16-token chunks within the longest context are shared
    rows = 2 * 8 * 2
    pf = 2 * ((rows * 4 + 255) // 256 * 256) + (rows * 64 * 4 + 255) // 256 * 256 + 256
    assert ws(2, 8, 64, 200, 1000) == pf + pa.pa_decode_workspace_size(2, 8, 64, 200 - 192)
    vp = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    call = lambda prefix, piece=0, maxL=100: lib.pa_decode_shared_prefix(
        vp, vp, vp, vp, vp, 8, vp, maxL, 1, 8, 8, 128, 16, 10, 0.1, 1, prefix, piece, vp, 1 << 30, None)
    assert call(129) == -5              # prefix beyond the table's 8 x 16 tokens
    assert call(-1) == -5
    assert call(64, maxL=129) == -5     # max_context_len beyond the table
    assert call(64, piece=100) == -3    # pieces are multiples of 128
    assert lib.pa_decode_shared_prefix(vp, vp, vp, vp, vp, 8, vp, 100, 1, 8, 8, 80, 16, 10, 0.1, 1, 64, 0, vp,
                                       1 << 30, None) == -3   # head_dim
