"""CUDA-graph capture of the hot path (the decode step of a serving loop): the KV write and the
decode are captured once on torch's capture stream and replayed.  A replay must reproduce the
eager result bit for bit; a replay after new inputs are written in place (new query rows and
K/V rows, more padded -1 slots, shorter contexts) must match the oracle.  Every launch of the
library goes to the stream it is given, with no allocation or synchronisation inside, and the
one-time set-up (function attributes, device state) happens on the first, eager call."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, to_dev, to_dev_i

pytestmark = pytest.mark.gpu


def _new_inputs(w, seed):
    """Fresh query and K/V rows of the same shapes, 40 more padded slots and contexts shortened
    by up to 50 tokens (each context stays >= 1 and the write's slots stay inside it or are -1)."""
    p, b, wr = w.pool, w.decode, w.write
    q = wl.normal_bits(wl.derive_seed(seed, 1), b.q.size, p.dtype).reshape(b.q.shape)
    key = wl.normal_bits(wl.derive_seed(seed, 2), wr.key.size, p.dtype).reshape(wr.key.shape)
    val = wl.normal_bits(wl.derive_seed(seed, 3), wr.value.size, p.dtype).reshape(wr.value.shape)
    sm = wr.slot_mapping.copy()
    sm[wl.permutation(wl.derive_seed(seed, 4), sm.size)[:40]] = -1
    cut = wl.uniform_ints(wl.derive_seed(seed, 5), b.num_seqs, 0, 50).astype(np.int32)
    lens = np.maximum(b.context_lens - cut, 1).astype(np.int32)
    return q, key, val, sm, lens


def _oracle_step(cache_k, cache_v, key, val, sm, q, b, lens, p):
    k2, v2, _ = oracle.kv_write(cache_k, cache_v, key, val, sm, p.block_size)
    ex = oracle.decode(q, k2, v2, b.block_tables, lens, b.scale, p.dtype)
    cd = oracle.decode(q, k2, abs_bits(v2), b.block_tables, lens, b.scale, p.dtype)
    return k2, v2, ex, cd


@pytest.mark.parametrize("path", ["auto", "splitk", "fused"])
def test_decode_step_graph_replay(path):
    """auto: pa_reshape_and_cache then pa_decode (the persistent one-pass grid); splitk: the same
    with 256-token pieces (the dynamic split-K grid); fused: one pa_decode_write call, whose decode
    CTAs write the rows."""
    w = wl.make_workload(4)
    p, b, wr = w.pool, w.decode, w.write
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    key, val = to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype)
    sm = to_dev_i(wr.slot_mapping, torch.int64)
    q = to_dev(b.q, p.dtype)
    out = torch.empty_like(q)
    bt, cl = to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32)
    maxL = int(b.context_lens.max())   # fixed at capture: it sizes the grid and the split
    S, hq, D = b.q.shape
    ws = torch.zeros(max(16, pa.pa_decode_workspace_size(S, hq, D, maxL, 256)), dtype=torch.uint8, device="cuda")

    def step():
        if path == "fused":
            pa.pa_decode_write(out, q, kc, vc, bt, cl, maxL, b.scale, key, val, sm, ws)
            return
        pa.pa_reshape_and_cache(key, val, kc, vc, sm)
        if path == "auto":
            pa.pa_decode(out, q, kc, vc, bt, cl, maxL, b.scale, ws)
        else:
            pa.pa_decode_splitk(out, q, kc, vc, bt, cl, maxL, b.scale, ws, 256)

    pa.pa_device_errors(clear=True)
    step()                                   # eager: one-time set-up happens here
    torch.cuda.synchronize()
    eager = bits_of(out)
    eager_k, eager_v = bits_of(kc), bits_of(vc)

    kc.copy_(to_dev(p.k_cache, p.dtype))
    vc.copy_(to_dev(p.v_cache, p.dtype))
    out.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(out), eager)
    assert np.array_equal(bits_of(kc), eager_k) and np.array_equal(bits_of(vc), eager_v)

    # next step: new inputs written into the captured buffers, same graph
    q2, key2, val2, sm2, lens2 = _new_inputs(w, 232_777)
    if path == "fused":
        # pa_decode_write's rows sit at each context's last token: move the live slots there
        last = lens2.astype(np.int64) - 1
        at_last = b.block_tables[np.arange(b.num_seqs), last // p.block_size].astype(np.int64) * p.block_size + \
            last % p.block_size
        sm2 = np.where(sm2 >= 0, at_last, -1).astype(np.int64)
    before_k, before_v = bits_of(kc), bits_of(vc)
    q.copy_(to_dev(q2, p.dtype))
    key.copy_(to_dev(key2, p.dtype))
    val.copy_(to_dev(val2, p.dtype))
    sm.copy_(to_dev_i(sm2, torch.int64))
    cl.copy_(to_dev_i(lens2, torch.int32))
    g.replay()
    torch.cuda.synchronize()
    k2, v2, ex, cd = _oracle_step(before_k, before_v, key2, val2, sm2, q2, b, lens2, p)
    assert np.array_equal(bits_of(kc), k2) and np.array_equal(bits_of(vc), v2)
    check_attention(bits_of(out), ex, p.dtype, f"graph replay ({path})", cond=cd)
    assert pa.pa_device_errors(clear=True) == 0


def test_prefill_graph_replay_matches_eager():
    w = wl.build_workload("pfg", 41, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                          prefill_q_lens=[1, 64, 200, 17], prefill_ctx_lens=[0, 300, 1000, 16], extra_blocks=3)
    p, pre = w.pool, w.prefill
    kc, vc, q = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype), to_dev(pre.q, p.dtype)
    out = torch.empty_like(q)
    bt = to_dev_i(pre.block_tables, torch.int32)
    qsl, sl = to_dev_i(pre.query_start_loc, torch.int32), to_dev_i(pre.seq_lens, torch.int32)

    def step():
        pa.pa_prefill_chunk(out, q, kc, vc, bt, qsl, sl, pre.max_q_len, pre.scale)

    step()
    torch.cuda.synchronize()
    eager = bits_of(out)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(out), eager)
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("case", ["mixed", "split_suffix"])
def test_shared_prefix_graph_replay(case):
    """pa_decode_shared_prefix captured once -- the prefix pass, the suffix decode as its
    programmatic dependent and, for long suffixes, the split-K merge as theirs -- replays bit for
    bit, and after new query rows and shorter contexts are written in place it matches the oracle
    (mini_engine, "Features": shared prefix blocks; "Roadmap": decode CUDA graphs)."""
    if case == "mixed":
        w = wl.make_workload(5)
        P = 1024
    else:
        w = wl.build_workload("gsp", 61, dtype=wl.BF16, n_q_heads=32, n_kv_heads=8, head_dim=128,
                              decode_lens=[12000, 9000, 16000, 2049], shared_prefix_blocks=128)
        P = 2048
    p, b = w.pool, w.decode
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    q = to_dev(b.q, p.dtype)
    out = torch.empty_like(q)
    bt, cl = to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32)
    maxL = int(b.context_lens.max())
    S, hq, D = b.q.shape
    ws = torch.zeros(pa.pa_decode_shared_prefix_workspace_size(S, hq, D, maxL, P), dtype=torch.uint8, device="cuda")

    def step():
        pa.pa_decode_shared_prefix(out, q, kc, vc, bt, cl, maxL, b.scale, P, ws)

    step()                                   # eager first call: one-time set-up
    torch.cuda.synchronize()
    eager = bits_of(out)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(out), eager)
    # new inputs in place: fresh query rows, contexts shortened by up to 50 tokens (never below 1)
    q_new = wl.normal_bits(wl.derive_seed(61, 9), b.q.size, p.dtype).reshape(b.q.shape)
    cut = wl.uniform_ints(wl.derive_seed(61, 10), S, 0, 50).astype(np.int32)
    lens = np.maximum(b.context_lens - cut, 1).astype(np.int32)
    q.copy_(to_dev(q_new, p.dtype))
    cl.copy_(to_dev_i(lens, torch.int32))
    g.replay()
    torch.cuda.synchronize()
    ex = oracle.decode(q_new, p.k_cache, p.v_cache, b.block_tables, lens, b.scale, p.dtype)
    cd = oracle.decode(q_new, p.k_cache, abs_bits(p.v_cache), b.block_tables, lens, b.scale, p.dtype)
    check_attention(bits_of(out), ex, p.dtype, f"shared prefix replay {case}", cond=cd, rel=1e-4 + 2.0 ** -16)
    assert pa.pa_device_errors(clear=True) == 0
