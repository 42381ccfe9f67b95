"""GPU parity of pa_decode_shared_prefix against the fp64 oracle.

The call computes exactly what pa_decode computes (the oracle is the same decode definition);
only the order of the arithmetic differs: the prefix all sequences share goes through the
tensor-core prefill kernel once per KV head (its softmax weights enter the PV product as two
16-bit terms, as in prefill), and the per-sequence suffix through the decode kernels, merged
at the end.  So the tests use the prefill allowance on top of the decode rule: rel = 1e-4 +
2^-16 (bf16) / 2^-22 (fp16) of the row's condition scale.  Source: mini_engine, "Features"
(hash-based prefix caching shares KV blocks) and "Custom CUDA kernels" (paged decode)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, to_dev, to_dev_i

pytestmark = pytest.mark.gpu

P_ROUND = {wl.BF16: 2.0 ** -16, wl.F16: 2.0 ** -22}


def dev_inputs(w):
    p, b = w.pool, w.decode
    return (to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype), to_dev(b.q, p.dtype),
            to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32))


def run_shared(w, prefix_tokens, max_context_len=None, piece=0, inputs=None):
    p, b = w.pool, w.decode
    kc, vc, q, bt, cl = dev_inputs(w) if inputs is None else inputs
    maxL = int(b.context_lens.max()) if max_context_len is None else max_context_len
    S, hq, d = b.q.shape
    ws = torch.empty(max(16, pa.pa_decode_shared_prefix_workspace_size(S, hq, d, maxL, prefix_tokens)),
                     dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_shared_prefix(out, q, kc, vc, bt, cl, maxL, b.scale, prefix_tokens, ws, prefix_piece_tokens=piece)
    torch.cuda.synchronize()
    return bits_of(out)


def reference(w, k_cache=None, v_cache=None):
    p, b = w.pool, w.decode
    kc = p.k_cache if k_cache is None else k_cache
    vc = p.v_cache if v_cache is None else v_cache
    ex = oracle.decode(b.q, kc, vc, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, kc, abs_bits(vc), b.block_tables, b.context_lens, b.scale, p.dtype)
    return ex, cd


def check(got, ref, dt, what):
    ex, cd = ref
    return check_attention(got, ex, dt, what, cond=cd, rel=1e-4 + P_ROUND[dt])


def shared_case(seed, lens, prefix_blocks, *, dt=wl.BF16, hq=16, hkv=8, d=128, bs=16, mb=None):
    return wl.build_workload("shp", seed, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, block_size=bs,
                             decode_lens=lens, shared_prefix_blocks=prefix_blocks, max_blocks_per_seq=mb)


def test_shared_prefix_mixed_workload_every_row():
    """The mixed batch's 128 decode sequences (a 1024-token prefix of 64 shared blocks, private
    suffixes of 1..1024 tokens), full size: every output row against the oracle, with the
    library's default prefix pieces and with explicit ones."""
    w = wl.make_workload(5)
    ref = reference(w)
    inputs = dev_inputs(w)
    for piece in (0, 128, 512, 1024):
        got = run_shared(w, 1024, piece=piece, inputs=inputs)
        check(got, ref, wl.BF16, f"mixed decode rows, prefix pieces {piece}")
    assert pa.pa_device_errors(clear=True) == 0


def test_prefix_zero_is_plain_decode_bitwise():
    """No shared tokens: the call is pa_decode, bit for bit."""
    w = shared_case(11, [300, 17, 1000, 64], 0)
    kc, vc, q, bt, cl = dev_inputs(w)
    b = w.decode
    ws = torch.empty(max(16, pa.pa_decode_workspace_size(4, 16, 128, 1000, 0)), dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(q)
    pa.pa_decode(ref, q, kc, vc, bt, cl, 1000, b.scale, ws)
    torch.cuda.synchronize()
    for pt in (0, 15):   # fewer than 16 shared tokens: no prefix pass either
        got = run_shared(w, pt, inputs=(kc, vc, q, bt, cl))
        assert np.array_equal(got, bits_of(ref))
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("case", ["whole_context", "mid_block", "mid_chunk", "shorter_than_prefix",
                                  "loose_bound", "many_tiles", "split_k_suffix", "dynamic_split_suffix",
                                  "dynamic_units"])
def test_shared_prefix_edges(case):
    """whole_context: every context is exactly the prefix (no suffix).  mid_block / mid_chunk: the
    prefix the caller names ends inside a block (and inside a 16-token chunk: the remainder is
    streamed per sequence).  shorter_than_prefix: some contexts end inside the prefix.
    loose_bound: every context ends inside the prefix and max_context_len is far above them, so
    the prefix pass meets tokens no sequence owns (NaN canaries) and must cut at the longest
    context.  many_tiles: 300 sequences (five 128-row query tiles per KV head).  split_k_suffix:
    four sequences with long suffixes, where the dispatcher splits the suffix and the split-K
    merge folds in the prefix partials.  dynamic_split_suffix: 16 sequences at group size 2 with
    long suffixes, whose split goes to the dynamic grid (tail pieces; the CTA that finishes a
    unit merges it with the prefix partials).  dynamic_units: 200 sequences x 4 KV heads at group
    size 1 and head_dim 64 with one-pass suffixes (some empty): more units than the dynamic grid's
    slots, so the suffix runs on that grid over whole units, longest first."""
    maxL = None
    if case == "whole_context":
        w, P = shared_case(21, [512] * 9, 32), 512
    elif case == "mid_block":
        w, P = shared_case(22, [1100, 1008, 1500, 2000], 63), 1000
    elif case == "mid_chunk":
        w, P = shared_case(23, [700, 650, 1200], 40, bs=32), 637
    elif case == "shorter_than_prefix":
        w, P = shared_case(24, [5, 100, 2048, 700, 1, 1024, 1025], 64), 1024
    elif case == "loose_bound":
        w, P, maxL = shared_case(25, [5, 100, 300], 40, mb=128), 640, 2048
    elif case == "many_tiles":
        lens = 512 + wl.uniform_ints(wl.derive_seed(26, 1), 300, 1, 700)
        w, P = shared_case(26, lens, 32), 512
    elif case == "split_k_suffix":
        w, P = shared_case(27, [12000, 9000, 16000, 2049], 128, hq=32, hkv=8), 2048
    elif case == "dynamic_units":
        lens = 512 + wl.uniform_ints(wl.derive_seed(29, 1), 200, 0, 700)
        lens[[3, 77]] = 512
        w, P = shared_case(29, lens, 32, hq=4, hkv=4, d=64), 512
    else:
        lens = 1024 + wl.uniform_ints(wl.derive_seed(28, 1), 16, 3000, 8000)
        lens[5] = 1024
        w, P = shared_case(28, lens, 64), 1024
    if case == "split_k_suffix":
        which, _ = pa.pa_decode_plan(4, 32, 8, 128, 16, 16000 - 2048)
        assert which == 2
    if case == "dynamic_split_suffix":
        which, part = pa.pa_decode_plan(16, 16, 8, 128, 16, int(w.decode.context_lens.max()) - 1024)
        assert which == 2 and 16 * 8 * -(-(int(w.decode.context_lens.max()) - 1024) // part) > 456
    got = run_shared(w, P, max_context_len=maxL)
    check(got, reference(w), w.pool.dtype, case)
    assert pa.pa_device_errors(clear=True) == 0


def test_workspace_shared_with_split_decode():
    """One workspace for split-K decode calls and shared-prefix calls in turn.  The split-K calls
    run the dynamic grid (200 sequences x 4 KV heads, 256-token pieces), whose merge leaves the
    counter at the workspace's start at zero with its tag set; the shared-prefix call runs its
    suffix on the dynamic grid over whole units with a counter at the same place, zeroed with the
    tag before its prefix pass and left where its claims stopped, so the next split-K call finds
    no tag and takes the fixed order.  Every split-K call gives the same bits (and the oracle's
    values), the shared-prefix call the oracle's values."""
    lens = 512 + wl.uniform_ints(wl.derive_seed(29, 1), 200, 0, 700)
    lens[[3, 77]] = 512
    w = shared_case(29, lens, 32, hq=4, hkv=4, d=64)
    kc, vc, q, bt, cl = dev_inputs(w)
    b = w.decode
    maxL = int(b.context_lens.max())
    nbytes = max(pa.pa_decode_shared_prefix_workspace_size(200, 4, 64, maxL, 512),
                 pa.pa_decode_workspace_size(200, 4, 64, maxL, 256))
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")

    def split():
        out = torch.full_like(q, float("nan"))
        pa.pa_decode_splitk(out, q, kc, vc, bt, cl, maxL, b.scale, ws, 256)
        torch.cuda.synchronize()
        return bits_of(out)

    def tag():
        return int(ws[8:16].cpu().numpy().view(np.uint64)[0])

    ref = reference(w)
    first = split()                     # no tag yet: the fixed order
    check(first, ref, wl.BF16, "split-K, fresh workspace")
    assert tag() == 0x7FC0A5177FC02C32
    assert np.array_equal(split(), first)   # from the counter
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_shared_prefix(out, q, kc, vc, bt, cl, maxL, b.scale, 512, ws)
    torch.cuda.synchronize()
    check(bits_of(out), ref, wl.BF16, "shared prefix on the split-K workspace")
    assert tag() == 0
    assert np.array_equal(split(), first)   # the fixed order again
    assert np.array_equal(split(), first)   # from the counter
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("dt,hq,hkv,d,bs", [(wl.BF16, 8, 8, 128, 16), (wl.F16, 32, 8, 128, 16), (wl.BF16, 64, 8, 64, 16),
                                            (wl.F16, 16, 8, 96, 8), (wl.BF16, 8, 4, 256, 32), (wl.BF16, 16, 4, 256, 16),
                                            (wl.F16, 4, 4, 64, 128)])
def test_shared_prefix_shapes(dt, hq, hkv, d, bs):
    """Group sizes 1-8, head_dim 64/96/128/256, fp16 and bf16, blocks of 8-128 tokens."""
    nP = max(1, 768 // bs)
    lens = nP * bs + wl.uniform_ints(wl.derive_seed(31, hq + d + bs), 40, 1, 600)
    w = shared_case(31 + hq + d + bs, lens, nP, dt=dt, hq=hq, hkv=hkv, d=d, bs=bs)
    got = run_shared(w, nP * bs)
    check(got, reference(w), dt, f"shapes {dt} {hq}/{hkv} hd {d} bs {bs}")
    assert pa.pa_device_errors(clear=True) == 0


def test_shared_prefix_relabelling_is_bitwise_invariant():
    """Moving the blocks to other physical ids (the data with them) changes nothing, bit for bit:
    the same values are read in the same order."""
    w = shared_case(41, 1024 + wl.uniform_ints(wl.derive_seed(41, 1), 50, 1, 500), 64)
    got = run_shared(w, 1024)
    p, b = w.pool, w.decode
    perm = wl.permutation(wl.derive_seed(41, 2), p.num_blocks)
    k2, v2 = np.empty_like(p.k_cache), np.empty_like(p.v_cache)
    k2[perm], v2[perm] = p.k_cache, p.v_cache
    w.pool.k_cache, w.pool.v_cache = k2, v2
    w.decode.block_tables = perm[b.block_tables].astype(np.int32)
    assert np.array_equal(run_shared(w, 1024), got)


def test_shared_prefix_repeated_calls_bitwise_identical():
    w = wl.make_workload(5)
    inputs = dev_inputs(w)
    first = run_shared(w, 1024, inputs=inputs)
    for _ in range(10):
        assert np.array_equal(run_shared(w, 1024, inputs=inputs), first)
    assert pa.pa_device_errors(clear=True) == 0


def test_shared_prefix_argument_errors():
    w = shared_case(51, [600, 700], 32)
    kc, vc, q, bt, cl = dev_inputs(w)
    b = w.decode
    out = torch.empty_like(q)
    ws = torch.empty(pa.pa_decode_shared_prefix_workspace_size(2, 16, 128, 700, 512), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_shared_prefix(out, q, kc, vc, bt, cl, 700, b.scale, 512, ws[:-256])
    assert e.value.status == -7
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_shared_prefix(out, q, kc, vc, bt, cl, 700, b.scale, 512, ws, prefix_piece_tokens=100)
    assert e.value.status == -3
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_shared_prefix(out, q, kc, vc, bt, cl, 700, b.scale, 10 ** 6, ws)
    assert e.value.status == -5
