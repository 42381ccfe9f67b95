"""pa_decode_splitk_static: split-K decode whose scratch is a fixed array inside the library,
for callers that cannot allocate device memory (a framework that owns every allocation, a
latency-critical path, a capture mode that forbids cudaMalloc).

The test calls the entry point through the C ABI and compares its output with the existing
pa_decode_splitk (caller-allocated workspace) on the same inputs and the same pieces, twice in
a row -- the second call runs over whatever the first left in the shared array.  Both run the
same kernels over the same pieces, so the outputs must be bitwise equal; both are also checked
against the fp64 oracle.  This file is collected last so that a run stopping at its first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, to_dev, to_dev_i

pytestmark = pytest.mark.gpu


def _inputs(seed, lens, hq, hkv, mb=None):
    w = wl.build_workload("nalloc", seed, dtype=wl.BF16, n_q_heads=hq, n_kv_heads=hkv, head_dim=128,
                          decode_lens=lens, max_blocks_per_seq=mb)
    p, b = w.pool, w.decode
    return w, dict(kc=to_dev(p.k_cache, p.dtype), vc=to_dev(p.v_cache, p.dtype), q=to_dev(b.q, p.dtype),
                   bt=to_dev_i(b.block_tables, torch.int32), cl=to_dev_i(b.context_lens, torch.int32),
                   maxL=int(b.context_lens.max()), scale=b.scale)


def _static_call(lib, t, out, part=0, maxL=None):
    S, hq, d = t["q"].shape
    nb, bs, hkv, _ = t["kc"].shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.pa_decode_splitk_static(out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(),
                                       t["bt"].data_ptr(), t["bt"].shape[1], t["cl"].data_ptr(),
                                       t["maxL"] if maxL is None else maxL, S, hq, hkv, d, bs, nb,
                                       ctypes.c_float(t["scale"]), pa.PA_BF16, part, stream)


@pytest.mark.parametrize("lens,hq,hkv", [([5000, 300, 2048, 16, 4097], 32, 8), ([32768] * 4, 32, 8),
                                         ([200, 17, 256, 1], 16, 8)])
def test_static_scratch_matches_caller_workspace_twice(lens, hq, hkv):
    """The last case has every context within one 256-token piece: the one-piece path, where the
    pieces write the output directly and no scratch address is taken."""
    lib = pa.load()
    w, t = _inputs(4321 + len(lens), lens, hq, hkv)
    S, _, d = t["q"].shape
    ref = torch.empty_like(t["q"])
    ws = torch.empty(max(16, pa.pa_decode_workspace_size(S, hq, d, t["maxL"], 0)), dtype=torch.uint8, device="cuda")
    pa.pa_decode_splitk(ref, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], t["maxL"], t["scale"], ws)
    torch.cuda.synchronize()
    want = bits_of(ref)
    p, b = w.pool, w.decode
    ex = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, p.k_cache, abs_bits(p.v_cache), b.block_tables, b.context_lens, b.scale, p.dtype)
    check_attention(want, ex, p.dtype, "caller workspace", cond=cd)
    for call in range(2):
        out = torch.full_like(t["q"], float("nan"))
        assert _static_call(lib, t, out) == pa.PA_OK
        torch.cuda.synchronize()
        got = bits_of(out)
        assert np.array_equal(got, want), f"call {call}: not bitwise equal to the caller-workspace result"
        check_attention(got, ex, p.dtype, f"static scratch, call {call}", cond=cd)
    assert pa.pa_device_errors(clear=True) == 0


def test_static_scratch_rejects_sizes_beyond_its_limit():
    """A 128K-token bound for 2 sequences x 32 heads needs 512 pieces of partials per row,
    16.25 MiB > the array; the call must refuse before launching.  Every tensor matches the
    arguments (a real 2 x 8192-entry table, real lengths), so even a call that did launch would
    stay inside its buffers."""
    lib = pa.load()
    w, t = _inputs(99, [100, 200], 32, 8, mb=8192)
    maxL = 8192 * 16
    assert pa.pa_decode_workspace_size(2, 32, 128, maxL, 0) > pa.STATIC_SCRATCH_BYTES
    out = torch.empty_like(t["q"])
    assert _static_call(lib, t, out, maxL=maxL) == -7   # PA_ERR_WORKSPACE: nothing launched
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0
