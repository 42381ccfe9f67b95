"""GPU parity of pa_decode (dispatcher), pa_decode_v1 and pa_decode_splitk against the
fp64 oracle: the four decode workloads at full size, edge sweeps over lengths, group
sizes, head dims and dtypes, NaN canaries in every slot no sequence owns, exact special
cases, relabelling invariance, split-K intermediates and device error flags."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, to_dev, to_dev_i, ulp_distance

pytestmark = pytest.mark.gpu


class Dev:
    """A workload's pool and decode batch on the GPU."""

    def __init__(self, w, k_cache=None, v_cache=None):
        p, b = w.pool, w.decode
        self.w, self.dt = w, p.dtype
        self.kc = to_dev(p.k_cache if k_cache is None else k_cache, p.dtype)
        self.vc = to_dev(p.v_cache if v_cache is None else v_cache, p.dtype)
        self.q = to_dev(b.q, p.dtype)
        self.bt = to_dev_i(b.block_tables, torch.int32)
        self.cl = to_dev_i(b.context_lens, torch.int32)
        self.maxL = int(b.context_lens.max())
        self.scale = b.scale

    def run(self, mode="auto", part=0, cl=None):
        out = torch.empty_like(self.q)
        cl = self.cl if cl is None else cl
        S, hq, d = self.q.shape
        if mode == "v1":
            pa.pa_decode_v1(out, self.q, self.kc, self.vc, self.bt, cl, self.scale)
        else:
            ws_bytes = pa.pa_decode_workspace_size(S, hq, d, self.maxL, part)
            ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=out.device)
            self.ws = ws
            if mode == "splitk":
                pa.pa_decode_splitk(out, self.q, self.kc, self.vc, self.bt, cl, self.maxL, self.scale, ws, part)
            else:
                pa.pa_decode(out, self.q, self.kc, self.vc, self.bt, cl, self.maxL, self.scale, ws)
        torch.cuda.synchronize()
        return bits_of(out)


def oracle_decode(w, k_cache=None, v_cache=None):
    """(exact, cond): the fp64 outputs and each output's condition scale sum_t w_t |V_t|."""
    p, b = w.pool, w.decode
    k = p.k_cache if k_cache is None else k_cache
    v = p.v_cache if v_cache is None else v_cache
    exact = oracle.decode(b.q, k, v, b.block_tables, b.context_lens, b.scale, p.dtype)
    cond = oracle.decode(b.q, k, abs_bits(v), b.block_tables, b.context_lens, b.scale, p.dtype)
    return exact, cond


def check(got, ref, dt, what):
    return check_attention(got, ref[0], dt, what, cond=ref[1])


# ------------------------------------------------------------------ the decode workloads


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("mode", ["auto", "v1", "splitk"])
def test_decode_workloads_full_size(k, mode):
    w = wl.make_workload(k)
    pa.pa_device_errors(clear=True)
    got = Dev(w).run(mode)
    err = check(got, oracle_decode(w), w.pool.dtype, f"workload {k}/{mode}")
    assert err <= 2e-3
    assert pa.pa_device_errors(clear=True) == 0


def test_full_decode_step_batch_256_write_then_decode():
    """The batch-256 step: the write lands, then every sequence decodes over its context including
    the row just written (padded rows keep the slot's previous content)."""
    w = wl.make_workload(4)
    p, b, wr = w.pool, w.decode, w.write
    d = Dev(w)
    pa.pa_reshape_and_cache(to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype), d.kc, d.vc,
                            to_dev_i(wr.slot_mapping, torch.int64))
    got = d.run("auto")
    k2, v2, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, wr.slot_mapping, 16)
    assert np.array_equal(bits_of(d.kc), k2) and np.array_equal(bits_of(d.vc), v2)
    ref = oracle_decode(w, k2, v2)
    check(got, ref, p.dtype, "step256")
    for mode in ("v1", "splitk"):
        check(d.run(mode), ref, p.dtype, f"step256/{mode}")


def test_mixed_batch_decode_rows_with_shared_prefix():
    w = wl.make_workload(5)
    got = Dev(w).run("auto")
    check(got, oracle_decode(w), w.pool.dtype, "mixed batch decode rows")


# ------------------------------------------------------------------ edge sweeps


EDGE_LENS = [1, 15, 16, 17, 255, 256, 257, 513, 4097]


@pytest.mark.parametrize("dt,hq,hkv,d", [(wl.BF16, 16, 8, 128), (wl.F16, 2, 2, 64), (wl.BF16, 32, 8, 128),
                                         (wl.F16, 8, 1, 128), (wl.BF16, 8, 2, 64), (wl.F16, 16, 4, 128),
                                         (wl.BF16, 8, 1, 64), (wl.BF16, 16, 8, 96), (wl.F16, 32, 4, 96),
                                         (wl.BF16, 8, 8, 256), (wl.F16, 16, 8, 256), (wl.BF16, 16, 4, 256)])
@pytest.mark.parametrize("mode,part", [("v1", 0), ("splitk", 0), ("splitk", 64), ("splitk", 512), ("splitk", 48),
                                       ("splitk", 400)])
def test_decode_edge_lengths(dt, hq, hkv, d, mode, part):
    w = wl.build_workload("edge", 77 + hq + d, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                          decode_lens=EDGE_LENS, max_blocks_per_seq=300, extra_blocks=5)
    got = Dev(w).run(mode, part)
    check(got, oracle_decode(w), dt, f"edge {mode}/{part}")


@pytest.mark.parametrize("mode,part", [("v1", 0), ("splitk", 0), ("splitk", 64), ("splitk", 512), ("auto", 0)])
def test_decode_empty_contexts_among_others(mode, part):
    """Sequences with an empty context give an all-zero row, whichever grid runs them (in the
    split-K grid's longest-first order such a sequence has one empty piece, ranked last)."""
    lens = [0, 300, 0, 1000, 17, 0, 2049, 1]
    w = wl.build_workload("empty", 91, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                          decode_lens=[max(L, 1) for L in lens], max_blocks_per_seq=200, extra_blocks=3)
    w.decode.context_lens = np.asarray(lens, dtype=np.int32)
    got = Dev(w).run(mode, part)
    check(got, oracle_decode(w), wl.BF16, f"empty contexts {mode}/{part}")
    rows = got.reshape(len(lens), 16, 128)
    for s_, L in enumerate(lens):
        if L == 0:
            assert not rows[s_].any(), f"row {s_} not zero"
    assert pa.pa_device_errors(clear=True) == 0


def test_single_token_context_returns_v_bitwise():
    w = wl.build_workload("one", 5, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128, decode_lens=[1] * 9)
    p, b = w.pool, w.decode
    for mode in ("v1", "splitk"):
        got = Dev(w).run(mode).reshape(9, 16, 128)
        for s in range(9):
            v0 = p.v_cache[b.block_tables[s, 0], 0]          # [Hkv, D]
            assert np.array_equal(got[s], np.repeat(v0, 2, axis=0))


def test_uniform_v_within_one_ulp():
    w = wl.build_workload("u", 6, dtype=wl.F16, n_q_heads=4, n_kv_heads=2, head_dim=64, decode_lens=[700, 33, 2])
    p = w.pool
    vrow = wl.normal_bits(8, 2 * 64, wl.F16).reshape(2, 64)
    v = p.v_cache.copy()
    v[p.valid] = vrow
    for mode in ("v1", "splitk"):
        got = Dev(w, v_cache=v).run(mode).reshape(3, 4, 64)
        want = np.broadcast_to(np.repeat(vrow, 2, axis=0), (3, 4, 64))
        assert ulp_distance(got, want).max() <= 1


def test_block_relabelling_is_bitwise_invariant():
    w = wl.make_workload(2)
    p, b = w.pool, w.decode
    pi = wl.permutation(4242, p.num_blocks)
    k2, v2 = np.empty_like(p.k_cache), np.empty_like(p.v_cache)
    k2[pi], v2[pi] = p.k_cache, p.v_cache
    d1 = Dev(w)
    d2 = Dev(w, k2, v2)
    d2.bt = to_dev_i(pi[b.block_tables], torch.int32)
    for mode in ("v1", "splitk"):
        assert np.array_equal(d1.run(mode), d2.run(mode))


def test_splitk_intermediates_match_oracle_pieces():
    """fp32 per-piece max, exp-sum and normalised output, read back from the workspace
    (layout of pa_decode_workspace_size: the control region, then m, l, o), against the oracle's
    fp64 pieces at 1e-5.  Eight units of at most six pieces: the static split-K grid."""
    w = wl.build_workload("ws", 9, dtype=wl.BF16, n_q_heads=8, n_kv_heads=2, head_dim=128,
                          decode_lens=[1000, 256, 1300, 3], max_blocks_per_seq=96)
    p, b = w.pool, w.decode
    d = Dev(w)
    d.run("splitk", 256)
    S, hq, D, P = 4, 8, 128, -(-1300 // 256)
    rows = S * hq * P
    al = lambda x: (x + 255) // 256 * 256
    raw = d.ws.cpu().numpy()[256:]    # past the 256-byte control region
    gm = raw[: rows * 4].view(np.float32).reshape(S, hq, P)
    gl = raw[al(rows * 4): al(rows * 4) + rows * 4].view(np.float32).reshape(S, hq, P)
    go = raw[2 * al(rows * 4): 2 * al(rows * 4) + rows * D * 4].view(np.float32).reshape(S, hq, P, D)
    m, l, o = oracle.decode_partitions(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale,
                                       p.dtype, 256, P)
    # the same pieces over |V| give each output's condition scale sum_t w_t |V_t|
    absv = p.v_cache & np.uint16(0x7FFF)
    _, _, oabs = oracle.decode_partitions(b.q, p.k_cache, absv, b.block_tables, b.context_lens, b.scale,
                                          p.dtype, 256, P)
    for s in range(S):
        n = -(-int(b.context_lens[s]) // 256)
        if n <= 1:
            continue    # single-piece sequences are written directly, not through the workspace
        sl = np.s_[s, :, :n]
        np.testing.assert_allclose(gm[sl], m[sl], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(gl[sl], l[sl], rtol=1e-5, atol=0)
        assert np.all(np.abs(go[sl] - o[sl]) <= 1e-5 * oabs[sl] + 1e-7)


# ------------------------------------------------------------------ canaries and error flags


def test_out_of_pool_block_id_is_flagged_not_faulted():
    w = wl.build_workload("bad", 10, dtype=wl.BF16, n_q_heads=4, n_kv_heads=2, head_dim=128, decode_lens=[64, 40])
    d = Dev(w)
    bt = w.decode.block_tables.copy()
    bt[0, 1] = w.pool.num_blocks + 3        # outside the pool: the kernel reads zeros, records the error
    d.bt = to_dev_i(bt, torch.int32)
    pa.pa_device_errors(clear=True)
    for mode in ("v1", "splitk"):
        got = d.run(mode)
        assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_BLOCK
        # the other sequence is untouched by the bad entry
        ex, cd = oracle_decode(w)
        check_attention(got.reshape(2, 4, 128)[1:], ex[1:], wl.BF16, "good row", cond=cd[1:])


def test_context_longer_than_table_is_clamped_and_flagged():
    w = wl.build_workload("len", 11, dtype=wl.BF16, n_q_heads=4, n_kv_heads=2, head_dim=128, decode_lens=[32, 20])
    d = Dev(w)
    cl = to_dev_i(np.array([32 + 1000, 20], np.int32), torch.int32)
    pa.pa_device_errors(clear=True)
    got = d.run("v1", cl=cl)
    assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_LENGTH
    check(got.reshape(2, 4, 128), oracle_decode(w), wl.BF16, "clamped")


def test_zero_length_context_gives_zeros():
    w = wl.build_workload("z", 12, dtype=wl.BF16, n_q_heads=4, n_kv_heads=2, head_dim=128, decode_lens=[5, 300])
    d = Dev(w)
    cl = to_dev_i(np.array([0, 300], np.int32), torch.int32)
    for mode in ("v1", "splitk"):
        got = d.run(mode, cl=cl).reshape(2, 4, 128)
        assert np.all(got[0] == 0)


@pytest.mark.parametrize("bs", [8, 32, 64, 128])
@pytest.mark.parametrize("mode,part", [("v1", 0), ("splitk", 0), ("splitk", 512), ("splitk", 48)])
def test_decode_block_sizes(bs, mode, part):
    """Cache blocks of 8 / 32 / 64 / 128 tokens: 16-token chunks are read from their rows inside
    the block, or from two 8-token blocks (lengths straddling block and chunk boundaries, NaN in
    every unowned slot and in the poison block padding the tables)."""
    if part % max(bs, 16):
        pytest.skip("split-K pieces hold whole blocks")
    lens = [1, 15, 16, 17, bs - 1, bs, bs + 1, 3 * bs + 5, 2000]
    for dt, hq, hkv, d in [(wl.BF16, 16, 8, 128), (wl.F16, 8, 2, 64), (wl.BF16, 8, 4, 256)]:
        w = wl.build_workload("bs", 900 + bs + d, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, block_size=bs,
                              decode_lens=lens, extra_blocks=3)
        pa.pa_device_errors(clear=True)
        got = Dev(w).run(mode, part)
        check(got, oracle_decode(w), dt, f"bs {bs} {mode}/{part} hd {d}")
        assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("S,hq,hkv,d,bs,L", [(4, 32, 8, 128, 16, 32768), (2, 16, 8, 128, 16, 5000),
                                            (8, 8, 1, 64, 64, 20000), (300, 16, 8, 128, 16, 16384),
                                            (1, 2, 2, 64, 128, 300)])
def test_dispatcher_plan_pieces(S, hq, hkv, d, bs, L):
    """Split-K plans: pieces are a multiple of the block size and at least the default 256
    tokens, so a workspace sized for the default piece fits every plan."""
    which, part = pa.pa_decode_plan(S, hq, hkv, d, bs, L, pa.PA_BF16)
    assert which == 2
    assert part % bs == 0 and part >= 256
    assert pa.pa_decode_workspace_size(S, hq, d, L, part) <= pa.pa_decode_workspace_size(S, hq, d, L, 0)
    assert pa.pa_decode_plan(256, 16, 8, 128, 16, 2048)[0] == 1       # one-pass: enough units, short contexts


def _uniform_split_ws_bytes(S, hq, d, maxL, part):
    """The split-K workspace without room for tail pieces: m, l, o for ceil(maxL / part) pieces
    (each region 256-byte aligned) and the 256-byte control region."""
    kd = 128 if d == 96 else d
    rows = S * hq * (-(-maxL // part))
    a = lambda n: (n + 255) // 256 * 256
    return 2 * a(rows * 4) + a(rows * kd * 4) + 256


DYN_TAG = 0x7FC0A5177FC02C32   # the control region's "counter at zero" mark (two quiet-NaN floats)


def assert_counter_armed(ws):
    """After a call on the dynamic grid: the counter (bytes 0-3) at zero, the tag (8-15) set."""
    ctl = ws[:16].cpu().numpy()
    assert int(ctl[0:4].view(np.int32)[0]) == 0
    assert int(ctl[8:16].view(np.uint64)[0]) == DYN_TAG


def test_dynamic_grid_workspace_reused_across_sizes():
    """One workspace for successive batches of other sizes (a decode loop whose contexts grow and
    whose batch changes): the control region sits at the workspace's start for every size, so the
    counter each call leaves at zero is the one the next call takes pieces from; every call
    against the oracle, and the counter left at zero after each."""
    ws = torch.full((64 << 20,), 0x5A, dtype=torch.uint8, device="cuda")
    pa.pa_device_errors(clear=True)
    for i, (S, maxlen, part) in enumerate(((96, 3000, 256), (64, 2048, 512), (130, 1500, 256), (96, 3100, 256))):
        lens = wl.uniform_ints(wl.derive_seed(91, i), S, 1, maxlen)
        lens[7] = maxlen
        w = wl.build_workload("dynre", 91 + i, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                              block_size=16, decode_lens=lens.tolist())
        dev = Dev(w)
        assert pa.pa_decode_workspace_size(S, 16, 128, dev.maxL, part) <= ws.numel()
        out = torch.full_like(dev.q, float("nan"))
        pa.pa_decode_splitk(out, dev.q, dev.kc, dev.vc, dev.bt, dev.cl, dev.maxL, dev.scale, ws, part)
        torch.cuda.synchronize()
        check(bits_of(out), oracle_decode(w), wl.BF16, f"reused workspace, batch {i}")
        assert_counter_armed(ws)
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("dt,hq,hkv,d,bs,S,maxlen", [(wl.BF16, 16, 8, 128, 16, 96, 3000), (wl.F16, 8, 8, 64, 8, 96, 3000),
                                                   (wl.BF16, 4, 2, 256, 32, 96, 3000), (wl.F16, 16, 8, 96, 16, 96, 3000),
                                                   (wl.BF16, 16, 8, 128, 16, 300, 1200),
                                                   (wl.BF16, 8, 8, 128, 64, 40, 5000),
                                                   (wl.F16, 16, 8, 128, 128, 64, 4000)])
def test_dynamic_split_grid(dt, hq, hkv, d, bs, S, maxlen):
    """Group size 1 or 2 with more split-K pieces than resident CTAs: one CTA per resident slot
    takes pieces from a counter in the workspace, in whatever order the CTAs free up; batches of
    up to 256 sequences cut the last piece-length of every context into quarter pieces (tail
    pieces), larger ones (300) keep uniform pieces, as does a workspace sized without room for the
    tail pieces.  The workspace starts filled with 0x7f bytes, so the first call finds no tag
    beside the counter and hands the pieces out in the fixed order (CTA b: pieces b, b + grid, ...);
    its merge leaves the counter at 0 and the tag set, so the later calls take pieces from the
    counter.  A piece's arithmetic does not depend on which CTA takes it, so all calls agree bit for
    bit; against the oracle, with empty and one-token contexts among long ones."""
    lens = wl.uniform_ints(wl.derive_seed(77, hq + d + S), S, 1, maxlen)
    lens[[3, 20, 21]] = 0
    lens[[10, 30]] = 1
    lens[35] = maxlen
    w = wl.build_workload("dyn", 77 + hq + d + bs + S, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                          block_size=bs, decode_lens=lens.tolist(), extra_blocks=3)
    dev = Dev(w)
    ref = oracle_decode(w)
    pa.pa_device_errors(clear=True)
    for part, ws_bytes in ((256, None), (512, None), (256, _uniform_split_ws_bytes(S, hq, d, dev.maxL, 256))):
        part = max(part, bs)
        if ws_bytes is None:
            ws_bytes = pa.pa_decode_workspace_size(S, hq, d, dev.maxL, part)
        ws = torch.full((max(16, ws_bytes),), 0x7F, dtype=torch.uint8, device="cuda")
        first = None
        for _ in range(4):
            out = torch.full_like(dev.q, float("nan"))
            pa.pa_decode_splitk(out, dev.q, dev.kc, dev.vc, dev.bt, dev.cl, dev.maxL, dev.scale, ws, part)
            torch.cuda.synchronize()
            got = bits_of(out)
            if first is None:
                first = got
                check(got, ref, dt, f"dynamic split grid {part}")
            assert np.array_equal(got, first)
            assert_counter_armed(ws)
    check(dev.run("auto"), ref, dt, "dispatcher")
    assert pa.pa_device_errors(clear=True) == 0


def test_long_context_planned_pieces_match_oracle():
    """The dispatcher's piece length for four 32K-token contexts (not a power of two) through
    pa_decode, against the oracle."""
    w = wl.make_workload(3)
    b = w.decode
    which, part = pa.pa_decode_plan(b.num_seqs, b.q.shape[1], w.pool.n_kv_heads, b.q.shape[2], 16,
                                    int(b.context_lens.max()), pa.PA_BF16)
    assert which == 2 and part % 16 == 0
    pa.pa_device_errors(clear=True)
    got = Dev(w).run("splitk", part)
    check(got, oracle_decode(w), w.pool.dtype, f"long4/splitk {part}")
    assert pa.pa_device_errors(clear=True) == 0


def test_head_dim_256_batch_longer_than_a_wave():
    """head_dim 256 (G = 2: two CTAs per SM) with more (sequence, KV head) units than resident
    CTAs, so the one-pass grid runs longest first; and the split-K path on the same batch."""
    lens = wl.uniform_ints(wl.derive_seed(256, 1), 200, 100, 1500).tolist()
    w = wl.build_workload("hd256", 2561, dtype=wl.BF16, n_q_heads=8, n_kv_heads=4, head_dim=256, decode_lens=lens,
                          extra_blocks=3)
    ref = oracle_decode(w)
    pa.pa_device_errors(clear=True)
    for mode in ("auto", "splitk"):
        check(Dev(w).run(mode), ref, w.pool.dtype, f"hd 256 {mode}")
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("dt,hq,hkv,d,bs", [(wl.BF16, 16, 8, 128, 8), (wl.F16, 8, 8, 96, 32), (wl.BF16, 16, 8, 64, 16),
                                            (wl.F16, 4, 2, 256, 16)])
def test_many_short_sequences_persistent_grid(dt, hq, hkv, d, bs):
    """More than two waves of (sequence, KV head) units at group size <= 2: the dispatcher's
    one-pass grid runs one CTA per resident slot over longest-first unit lists.  Lengths from 0
    to 300 (empty contexts included), NaN in every unowned slot."""
    S = 400 if d != 256 else 700
    lens = wl.uniform_ints(wl.derive_seed(4242 + d + bs, 1), S, 0, 300).tolist()
    w = wl.build_workload("many", 4242 + d + bs, dtype=dt, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, block_size=bs,
                          decode_lens=lens, extra_blocks=2)
    pa.pa_device_errors(clear=True)
    got = Dev(w).run("auto")
    check(got, oracle_decode(w), dt, f"many short {hq}/{hkv} hd {d} bs {bs}")
    assert pa.pa_device_errors(clear=True) == 0


def test_persistent_grid_flags_bad_entries_and_finishes_the_rest():
    """The persistent one-pass grid with an out-of-pool block id in one sequence and a context
    longer than the table in another: both are flagged, no fault, every other row is right."""
    lens = wl.uniform_ints(wl.derive_seed(5151, 1), 300, 10, 300).tolist()
    w = wl.build_workload("pbad", 5151, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128, decode_lens=lens,
                          extra_blocks=2)
    d = Dev(w)
    bt = w.decode.block_tables.copy()
    bt[5, 0] = w.pool.num_blocks + 3
    d.bt = to_dev_i(bt, torch.int32)
    cl = w.decode.context_lens.copy()
    cl[7] = 1_000_000
    pa.pa_device_errors(clear=True)
    got = d.run("auto", cl=to_dev_i(cl, torch.int32)).reshape(300, 16, 128)
    errs = pa.pa_device_errors(clear=True)
    assert errs & pa.PA_DEVERR_BLOCK and errs & pa.PA_DEVERR_LENGTH
    ex, cd = oracle_decode(w)
    keep = np.array([i for i in range(300) if i not in (5, 7)])
    check_attention(got[keep], ex.reshape(300, 16, 128)[keep], wl.BF16, "persistent grid, good rows",
                    cond=cd.reshape(300, 16, 128)[keep])
