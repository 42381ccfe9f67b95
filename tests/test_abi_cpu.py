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
    # one piece needs no workspace; several pieces need m, l (256-byte aligned) and o
    assert pa.pa_decode_workspace_size(4, 32, 128, 256) == 0
    rows = 4 * 32 * 128
    expect = 2 * ((rows * 4 + 255) // 256 * 256) + (rows * 128 * 4 + 255) // 256 * 256
    assert pa.pa_decode_workspace_size(4, 32, 128, 32768) == expect


def test_validation_rejects_before_any_device_work(lib):
    vp = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # n_q_heads not a multiple of n_kv_heads
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 6, 4, 128, 16, 10, 0.1, 1, None) == -2
    # unsupported head_dim / block_size / dtype / group size
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 8, 8, 96, 16, 10, 0.1, 1, None) == -3
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 8, 8, 128, 32, 10, 0.1, 1, None) == -3
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 8, 8, 128, 16, 10, 0.1, 7, None) == -3
    assert lib.pa_decode_v1(vp, vp, vp, vp, vp, 8, vp, 1, 48, 3, 128, 16, 10, 0.1, 1, None) == -3
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
