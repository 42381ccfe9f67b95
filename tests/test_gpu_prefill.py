"""GPU parity of pa_prefill_chunk (tcgen05 tensor cores) against the fp64 oracle, and of
the mixed batch (decode rows through pa_decode, prefill rows through pa_prefill_chunk,
one output tensor).

The kernel carries the softmax weights into the PV product as two 16-bit terms
(P_hi + P_lo), whose sum is within 2^-17 (bf16) / 2^-23 (fp16) of each fp32 weight, so the
fp32-level rule gets an extra allowance of 2^-16 * cond (bf16) or 2^-22 * cond (fp16) on
top of its 1e-4 * cond; the 2e-3 absolute bound applies unchanged."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, to_dev, to_dev_i

pytestmark = pytest.mark.gpu

P_ROUND = {wl.BF16: 2.0 ** -16, wl.F16: 2.0 ** -22}


def run_prefill(w, out=None, q=None, kc=None, vc=None, small_m=False):
    p, pre = w.pool, w.prefill
    kc = to_dev(p.k_cache, p.dtype) if kc is None else kc
    vc = to_dev(p.v_cache, p.dtype) if vc is None else vc
    q = to_dev(pre.q, p.dtype) if q is None else q
    out = torch.empty_like(q) if out is None else out
    pa.pa_prefill_chunk(out, q, kc, vc, to_dev_i(pre.block_tables, torch.int32),
                        to_dev_i(pre.query_start_loc, torch.int32), to_dev_i(pre.seq_lens, torch.int32),
                        pre.max_q_len, pre.scale, small_m=small_m)
    torch.cuda.synchronize()
    return out


def oracle_rows(w, rows=None):
    """fp64 oracle for the given global query rows (all rows if None), with cond scales.
    Sampled rows are run as one-row chunks whose kv length is ctx + j + 1, which is what
    the bottom-right mask gives row j."""
    p, pre = w.pool, w.prefill
    if rows is None:
        ex = oracle.prefill_chunk(pre.q, p.k_cache, p.v_cache, pre.block_tables, pre.query_start_loc, pre.seq_lens,
                                  pre.scale, p.dtype)
        cd = oracle.prefill_chunk(pre.q, p.k_cache, abs_bits(p.v_cache), pre.block_tables, pre.query_start_loc,
                                  pre.seq_lens, pre.scale, p.dtype)
        return ex, cd
    rows = np.asarray(rows)
    qsl = pre.query_start_loc
    chunk = np.searchsorted(qsl, rows, side="right") - 1
    j = rows - qsl[chunk]
    ctx = pre.seq_lens[chunk] - np.diff(qsl)[chunk]
    q = np.ascontiguousarray(pre.q[rows])
    bt = np.ascontiguousarray(pre.block_tables[chunk])
    one = np.arange(len(rows) + 1, dtype=np.int32)
    kv = (ctx + j + 1).astype(np.int32)
    ex = oracle.prefill_chunk(q, p.k_cache, p.v_cache, bt, one, kv, pre.scale, p.dtype)
    cd = oracle.prefill_chunk(q, p.k_cache, abs_bits(p.v_cache), bt, one, kv, pre.scale, p.dtype)
    return ex, cd


def check(got_bits, ref, dt, what):
    ex, cd = ref
    return check_attention(got_bits, ex, dt, what, cond=cd, rel=1e-4 + P_ROUND[dt])


SHAPES = [(wl.BF16, 16, 8, 128), (wl.F16, 16, 8, 128), (wl.BF16, 8, 8, 128), (wl.BF16, 32, 8, 128),
          (wl.F16, 16, 2, 128), (wl.BF16, 16, 8, 64), (wl.F16, 8, 8, 64), (wl.BF16, 32, 4, 64), (wl.F16, 2, 2, 64),
          (wl.BF16, 16, 8, 96), (wl.F16, 8, 2, 96), (wl.BF16, 16, 8, 256), (wl.F16, 8, 2, 256), (wl.BF16, 4, 4, 256)]


@pytest.mark.parametrize("dt,hq,hkv,d", SHAPES)
def test_prefill_ragged_chunks_full_parity(dt, hq, hkv, d):
    w = wl.build_workload("pf", 300 + hq + hkv + d, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                          prefill_q_lens=[1, 7, 64, 65, 128, 200, 17],
                          prefill_ctx_lens=[0, 20, 5, 127, 300, 1000, 16], extra_blocks=3)
    got = bits_of(run_prefill(w))
    check(got, oracle_rows(w), dt, f"prefill {dt} {hq}/{hkv} hd {d}")
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("dt,hq,hkv,d", [(wl.BF16, 16, 8, 128), (wl.F16, 32, 8, 128), (wl.BF16, 16, 2, 64),
                                         (wl.BF16, 8, 8, 128), (wl.F16, 16, 8, 256), (wl.F16, 8, 2, 96)])
def test_prefill_small_m_tiles(dt, hq, hkv, d):
    """pa_prefill_chunk_small_m: chunks whose rows (query tokens x group heads) fit in 64 run as
    M = 64 MMAs (rows in TMEM lanes 0-15 of each quarter; the other lanes hold S = 0 and weight
    0): chunks right at 64 rows and one token past it (a 128-row tile), single tokens over long
    contexts (the unified launch's decode rows), every row against the oracle."""
    G = hq // hkv
    at = 64 // G
    w = wl.build_workload("pfsm", 400 + hq + hkv + d, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                          prefill_q_lens=[at, at + 1, 1, 1, max(1, at // 2), at],
                          prefill_ctx_lens=[0, 37, 2047, 0, 1000, 3001], extra_blocks=3)
    got = bits_of(run_prefill(w, small_m=True))
    check(got, oracle_rows(w), dt, f"small-M {dt} {hq}/{hkv} hd {d}")
    assert pa.pa_device_errors(clear=True) == 0


def test_prefill_head_dim_64_long_context_sampled_rows():
    """hd 64 at a mixed-workload-like size: 4 chunks of 300 rows over 0..3000 cached tokens."""
    w = wl.build_workload("pf64", 64_064, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=64,
                          prefill_q_lens=[300, 300, 300, 300], prefill_ctx_lens=[0, 1000, 2047, 3000], extra_blocks=3)
    got = bits_of(run_prefill(w)).reshape(w.prefill.q.shape)
    rows = np.unique(np.concatenate([np.arange(0, 1200, 37), [0, 299, 300, 599, 600, 899, 900, 1199]]))
    check(got[rows], oracle_rows(w, rows), wl.BF16, "hd 64 long context")
    assert pa.pa_device_errors(clear=True) == 0


def test_prefill_single_row_no_context_returns_v0():
    w = wl.build_workload("pf1", 7, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                          prefill_q_lens=[1, 1], prefill_ctx_lens=[0, 0])
    got = bits_of(run_prefill(w)).reshape(2, 16, 128)
    for c in range(2):
        v0 = w.pool.v_cache[w.prefill.block_tables[c, 0], 0]
        assert np.array_equal(got[c], np.repeat(v0, 2, axis=0))


_MIXED = {}


def mixed_prefill_oracle(w):
    """The fp64 oracle over every prefill row of the mixed batch (about 71 GFLOP of visible
    pairs, twice with the condition scales), computed once for the tests that need it."""
    if "ref" not in _MIXED:
        _MIXED["ref"] = oracle_rows(w)
    return _MIXED["ref"]


def test_prefill_mixed_batch_workload_every_row():
    """The mixed batch's eight 512-token chunks over 0..4096 cached tokens, full size: every
    row of every chunk against the oracle."""
    w = wl.make_workload(5)
    got = bits_of(run_prefill(w)).reshape(w.prefill.q.shape)
    check(got, mixed_prefill_oracle(w), wl.BF16, "mixed batch prefill, every row")
    assert pa.pa_device_errors(clear=True) == 0


def test_mixed_batch_one_output_tensor():
    """Decode rows and prefill rows of one batch write disjoint rows of one output; every row
    of both is checked."""
    w = wl.make_workload(5)
    p, b, pre = w.pool, w.decode, w.prefill
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    q_all = to_dev(np.concatenate([b.q, pre.q]), p.dtype)
    out = torch.full_like(q_all, float("nan"))
    S = b.num_seqs
    maxL = int(b.context_lens.max())
    ws = torch.empty(max(16, pa.pa_decode_workspace_size(S, 16, 128, maxL, 0)), dtype=torch.uint8, device="cuda")
    pa.pa_decode(out[:S], q_all[:S], kc, vc, to_dev_i(b.block_tables, torch.int32),
                 to_dev_i(b.context_lens, torch.int32), maxL, b.scale, ws)
    run_prefill(w, out=out[S:], q=q_all[S:], kc=kc, vc=vc)
    got = bits_of(out)
    ex = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, p.k_cache, abs_bits(p.v_cache), b.block_tables, b.context_lens, b.scale, p.dtype)
    check_attention(got[:S], ex, p.dtype, "mixed: decode rows", cond=cd)
    check(got[S:], mixed_prefill_oracle(w), p.dtype, "mixed: prefill rows")
    assert pa.pa_device_errors(clear=True) == 0


def test_prefill_out_of_pool_block_is_flagged_not_faulted():
    w = wl.build_workload("pfb", 8, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                          prefill_q_lens=[40, 30], prefill_ctx_lens=[100, 10])
    bt = w.prefill.block_tables.copy()
    bt[0, 2] = w.pool.num_blocks + 11
    w.prefill.block_tables = bt
    pa.pa_device_errors(clear=True)
    out = run_prefill(w)
    assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_BLOCK
    got = bits_of(out).reshape(w.prefill.q.shape)
    rows = np.arange(40, 70)                      # the second chunk does not touch the bad entry
    check(got[rows], oracle_rows(w, rows), wl.BF16, "good chunk")


def test_prefill_chunk_longer_than_max_q_len_is_flagged():
    """max_q_len sizes the grid; a chunk longer than it is skipped and flagged
    (PA_DEVERR_LENGTH) instead of leaving its later rows silently unwritten, and the other
    chunks are still computed."""
    w = wl.build_workload("pfq", 9, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                          prefill_q_lens=[40, 300], prefill_ctx_lens=[100, 10])
    p, pre = w.pool, w.prefill
    q = to_dev(pre.q, p.dtype)
    out = torch.full_like(q, float("nan"))
    pa.pa_device_errors(clear=True)
    pa.pa_prefill_chunk(out, q, to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype),
                        to_dev_i(pre.block_tables, torch.int32), to_dev_i(pre.query_start_loc, torch.int32),
                        to_dev_i(pre.seq_lens, torch.int32), 100, pre.scale)
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_LENGTH
    got = bits_of(out).reshape(pre.q.shape)
    rows = np.arange(0, 40)
    check(got[rows], oracle_rows(w, rows), wl.BF16, "chunk within max_q_len")
    assert np.isnan(wl.bits_to_float(got[40:], wl.BF16)).all()   # the long chunk was not written


@pytest.mark.parametrize("cfg", ["mixed", "short"])
def test_prefill_repeated_runs_bitwise_identical_and_no_device_errors(cfg):
    """The kernel's pipeline has no data-dependent order of accumulation, so repeated runs
    must agree bit for bit, and no barrier wait may ever reach its time limit (a wait that
    mistook an earlier phase for the one it wanted would either time out -- raising
    PA_DEVERR_TIMEOUT and leaving rows unwritten -- or read O early)."""
    if cfg == "mixed":
        w = wl.make_workload(5)
    else:  # many short chunks: most CTAs finish within a few sub-tiles, where phases race most
        w = wl.build_workload("pfr", 31, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                              prefill_q_lens=[1, 3, 64, 65, 127, 128, 129, 200, 256, 17, 90, 40],
                              prefill_ctx_lens=[0, 1, 0, 63, 64, 1, 130, 5, 0, 300, 47, 2000], extra_blocks=3)
    p, pre = w.pool, w.prefill
    kc, vc, q = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype), to_dev(pre.q, p.dtype)
    pa.pa_device_errors(clear=True)
    first = bits_of(run_prefill(w, kc=kc, vc=vc, q=q))
    for _ in range(24):
        out = torch.full_like(q, float("nan"))
        again = bits_of(run_prefill(w, out=out, kc=kc, vc=vc, q=q))
        assert np.array_equal(again, first)
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("small_m", [False, True])
def test_unified_mixed_batch_single_launch(small_m):
    """The mixed batch through one prefill launch: each decode sequence a chunk of one query
    row over its whole context, then the prefill chunks (the unified variant the split
    dispatch is compared with), with 128-row tiles and with small-M tiles for the decode rows.
    Decode rows against the oracle's decode, prefill rows sampled."""
    w = wl.make_workload(5)
    p, b = w.pool, w.decode
    u = wl.unified_batch(w)
    kc, vc, q = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype), to_dev(u.q, p.dtype)
    out = torch.full_like(q, float("nan"))
    pa.pa_device_errors(clear=True)
    pa.pa_prefill_chunk(out, q, kc, vc, to_dev_i(u.block_tables, torch.int32), to_dev_i(u.query_start_loc, torch.int32),
                        to_dev_i(u.seq_lens, torch.int32), u.max_q_len, u.scale, small_m=small_m)
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0
    got = bits_of(out)
    S = b.num_seqs
    ex = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, p.k_cache, abs_bits(p.v_cache), b.block_tables, b.context_lens, b.scale, p.dtype)
    check(got[:S], (ex, cd), p.dtype, "unified: decode rows")
    rows = np.arange(0, w.prefill.q.shape[0], 97)
    check(got[S:][rows], oracle_rows(w, rows), p.dtype, "unified: prefill rows")


@pytest.mark.parametrize("bs", [8, 32, 64, 128])
@pytest.mark.parametrize("d", [128, 64, 256])
def test_prefill_block_sizes(bs, d):
    w = wl.build_workload("pfbs", 950 + bs + d, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=d, block_size=bs,
                          prefill_q_lens=[1, 7, 64, 65, 128, 200, 17],
                          prefill_ctx_lens=[0, 20, 5, 127, 300, 1000, bs - 1], extra_blocks=3)
    got = bits_of(run_prefill(w))
    check(got, oracle_rows(w), wl.BF16, f"prefill bs {bs} hd {d}")
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("bs", [8, 32])
def test_write_then_decode_block_sizes(bs):
    w = wl.build_workload("wbs", 977 + bs, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128, block_size=bs,
                          decode_lens=[33, 64, 65, 500], write_rows=True, extra_blocks=2)
    p, b, wr = w.pool, w.decode, w.write
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    pa.pa_reshape_and_cache(to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype), kc, vc,
                            to_dev_i(wr.slot_mapping, torch.int64))
    q, out = to_dev(b.q, p.dtype), torch.empty(b.q.shape, dtype=torch.bfloat16, device="cuda")
    pa.pa_decode_v1(out, q, kc, vc, to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32),
                    b.scale)
    torch.cuda.synchronize()
    k2, v2, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, wr.slot_mapping, bs)
    assert np.array_equal(bits_of(kc), k2) and np.array_equal(bits_of(vc), v2)
    ex = oracle.decode(b.q, k2, v2, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, k2, abs_bits(v2), b.block_tables, b.context_lens, b.scale, p.dtype)
    check_attention(bits_of(out), ex, p.dtype, f"bs {bs} write + decode", cond=cd)


def test_prefill_head_dim_256_long_context_sampled_rows():
    """head_dim 256 (one query tile per CTA, 64-key stages) over long cached contexts: every
    row of a sample against the oracle."""
    w = wl.build_workload("pf256", 25_625, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=256,
                          prefill_q_lens=[300, 129, 64], prefill_ctx_lens=[2500, 700, 4000], extra_blocks=3)
    got = bits_of(run_prefill(w))
    rows = np.arange(0, w.prefill.q.shape[0], 7)
    check(got[rows], oracle_rows(w, rows), wl.BF16, "prefill hd 256 long")
    assert pa.pa_device_errors(clear=True) == 0


def test_prefill_empty_chunks_between_others():
    """Chunks with no query rows (a sequence with nothing new this step) between real ones:
    nothing is written for them and the others are unaffected."""
    w = wl.build_workload("pfz", 4141, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                          prefill_q_lens=[0, 70, 0, 5, 0], prefill_ctx_lens=[40, 300, 16, 1000, 0], extra_blocks=3)
    pa.pa_device_errors(clear=True)
    got = bits_of(run_prefill(w))
    check(got, oracle_rows(w), wl.BF16, "prefill with empty chunks")
    assert pa.pa_device_errors(clear=True) == 0
