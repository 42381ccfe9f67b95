"""pa_decode_splitk_static: split-K decode whose scratch is a fixed array inside the library,
for callers that cannot allocate device memory (a framework that owns every allocation, a
latency-critical path, a capture mode that forbids cudaMalloc).

The test calls the entry point through the C ABI and compares its output with the existing
pa_decode_splitk (caller-allocated workspace) on the same inputs, twice in a row -- the second
call runs over whatever the first left in the shared array.  This file is collected last so
that a run stopping at its first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import ATOL, bits_of, to_dev, to_dev_i

pytestmark = pytest.mark.gpu


def _inputs(seed, lens, hq, hkv):
    w = wl.build_workload("nalloc", seed, dtype=wl.BF16, n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                          decode_lens=lens)
    p, b = w.pool, w.decode
    return dict(kc=to_dev(p.k_cache, p.dtype), vc=to_dev(p.v_cache, p.dtype), q=to_dev(b.q, p.dtype),
                bt=to_dev_i(b.block_tables, torch.int32), cl=to_dev_i(b.context_lens, torch.int32),
                maxL=int(b.context_lens.max()), scale=b.scale)


def _static_call(lib, t, out, part=0):
    S, hq, d = t["q"].shape
    nb, bs, hkv, _ = t["kc"].shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_decode_splitk_static(out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
                                       t["bt"].data_ptr(), t["bt"].shape[1], t["cl"].data_ptr(), t["maxL"], S, hq,
                                       hkv, d, bs, nb, ctypes.c_float(t["scale"]), pa.PA_BF16, part, stream)


@pytest.mark.parametrize("lens,hq,hkv", [([5000, 300, 2048, 16, 4097], 32, 8), ([32768] * 4, 32, 8)])
def test_static_scratch_matches_caller_workspace_twice(lens, hq, hkv):
    lib = pa.load()
    t = _inputs(4321 + len(lens), lens, hq, hkv)
    S, _, d = t["q"].shape
    ref = torch.empty_like(t["q"])
    ws = torch.empty(pa.pa_decode_workspace_size(S, hq, d, t["maxL"], 0), dtype=torch.uint8, device="cuda")
    pa.pa_decode_splitk(ref, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], t["maxL"], t["scale"], ws)
    torch.cuda.synchronize()
    want = bits_of(ref).view(np.int16).view(np.uint16)
    want_f = wl.bits_to_float(want, wl.BF16)
    for call in range(2):
        out = torch.full_like(t["q"], float("nan"))
        assert _static_call(lib, t, out) == pa.PA_OK
        torch.cuda.synchronize()
        got_f = wl.bits_to_float(bits_of(out), wl.BF16)
        assert np.isfinite(got_f).all()
        assert np.abs(got_f - want_f).max() <= ATOL, f"call {call}"
    assert pa.pa_device_errors(clear=True) == 0


def test_static_scratch_rejects_sizes_beyond_its_limit():
    lib = pa.load()
    t = _inputs(99, [64, 64], 16, 8)
    # 4096 sequences x 32 heads x a 64K-token bound need far more partials than the array holds
    S, hq, d, maxL = 4096, 32, 128, 65536
    assert pa.pa_decode_workspace_size(S, hq, d, maxL, 0) > pa.STATIC_SCRATCH_BYTES
    out = torch.empty(S, hq, d, dtype=torch.bfloat16, device="cuda")
    st = lib.pa_decode_splitk_static(out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
                                     t["bt"].data_ptr(), 4096, t["cl"].data_ptr(), maxL, S, hq, 8, d, 16,
                                     t["kc"].shape[0], ctypes.c_float(0.1), pa.PA_BF16, 0, None)
    assert st == -7   # PA_ERR_WORKSPACE: nothing launched
