"""Pins for the fp64 oracle, against things other than the oracle itself.

The pages print no worked numeric example for these kernels, so the oracle is
pinned by: library routines (numpy / torch number-format conversions, torch
scaled_dot_product_attention in fp64 on materialised tensors), closed forms
(two-token sigmoid form, one-hot limits, means), invariants the pages fix
(paged == materialised contiguous, MiniLLM Runtime "Key benchmark results";
physical block relabelling), and brute force on tiny integer inputs.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as wl
from workloads import BF16, F16


def f64(bits, dtype):
    return oracle.to_double(bits, dtype)


def materialise(pool_cache, bt_row, L):
    """Contiguous [L, Hkv, D] gather via numpy fancy indexing (independent of the oracle)."""
    nb, bs, hkv, d = pool_cache.shape
    t = np.arange(L)
    return pool_cache[bt_row[t // bs], t % bs]


def sdpa_decode(q_bits, k_bits, v_bits, bt, cl, scale, dtype, n_kv_heads):
    """torch SDPA (fp64) over materialised K/V, GQA by repeat_interleave (head h -> kv head h // G)."""
    S, Hq, D = q_bits.shape
    G = Hq // n_kv_heads
    out = np.zeros((S, Hq, D))
    for s in range(S):
        L = int(cl[s])
        K = torch.from_numpy(f64(materialise(k_bits, bt[s], L), dtype))  # [L, Hkv, D]
        V = torch.from_numpy(f64(materialise(v_bits, bt[s], L), dtype))
        q = torch.from_numpy(f64(q_bits[s], dtype))                       # [Hq, D]
        Kx = K.permute(1, 0, 2).repeat_interleave(G, dim=0)               # [Hq, L, D]
        Vx = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = F.scaled_dot_product_attention(q[:, None, :], Kx, Vx, scale=scale)
        out[s] = o[:, 0, :].numpy()
    return out


def small_decode(seed, lens, hq=4, hkv=2, d=16, dtype=BF16, **kw):
    return wl.build_workload("t", seed, dtype=dtype, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, decode_lens=lens, **kw)


# --------------------------------------------------------------- number formats


def test_f16_widening_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = f64(bits, F16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_widening_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = f64(bits, BF16)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 5, 20000),
        # exact ties between neighbouring fp16 values, normal and subnormal
        (np.arange(0, 4096, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0 ** -10,
        np.array([65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -25, 2.0 ** -26]),
    ])
    ref = x.astype(np.float16).view(np.uint16)
    got = oracle.round_to(x, F16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    # float32-representable inputs, so torch's float->bf16 rounding is the exact reference
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    ties = ((np.arange(0x3F80, 0x4000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1e-40], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_to(x.astype(np.float64), BF16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------- KV-cache write


@pytest.mark.parametrize("bs", [8, 16, 32, 128])
def test_kv_write_lands_at_block_and_offset(bs):
    w = wl.write_rows_case(7, 300, n_kv_heads=2, head_dim=16, block_size=bs, pad_frac=0.1)
    p, wr = w.pool, w.write
    k, v, st = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, wr.slot_mapping, bs)
    assert st == oracle.OK
    touched = np.zeros((p.num_blocks, bs), dtype=bool)
    for i, slot in enumerate(wr.slot_mapping):
        if slot < 0:
            continue
        b, o = divmod(int(slot), bs)          # slot = block_id * block_size + offset
        assert np.array_equal(k[b, o], wr.key[i]) and np.array_equal(v[b, o], wr.value[i])
        touched[b, o] = True
    assert (wr.slot_mapping == -1).sum() == 30
    assert np.array_equal(k[~touched], p.k_cache[~touched])
    assert np.array_equal(v[~touched], p.v_cache[~touched])


def test_kv_write_out_of_pool_slot_is_reported_and_skipped():
    w = wl.write_rows_case(8, 4, n_kv_heads=1, head_dim=8, pad_frac=0.0, extra_blocks=0)
    p, wr = w.pool, w.write
    sm = wr.slot_mapping.copy()
    sm[1] = p.num_blocks * 16          # one past the pool
    k, v, st = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, sm, 16, check=False)
    assert st == oracle.EBOUNDS
    for i in (0, 2, 3):
        b, o = divmod(int(sm[i]), 16)
        assert np.array_equal(k[b, o], wr.key[i])


# --------------------------------------------------------------- decode


@pytest.mark.parametrize("dtype,hq,hkv,d", [(BF16, 4, 2, 16), (F16, 2, 2, 64), (BF16, 8, 2, 32), (F16, 3, 1, 8)])
def test_decode_matches_torch_sdpa_fp64(dtype, hq, hkv, d):
    w = small_decode(11 + d, [1, 15, 16, 17, 40, 100], hq=hq, hkv=hkv, d=d, dtype=dtype)
    p, b = w.pool, w.decode
    got = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, dtype)
    ref = sdpa_decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, dtype, hkv)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bs,d", [(8, 96), (32, 24), (128, 8)])
def test_decode_matches_torch_sdpa_other_block_sizes_and_widths(bs, d):
    """The oracle's block addressing at 8-, 32- and 128-token blocks (lengths straddling block
    boundaries) and head widths that are not powers of two, against SDPA over gathered K/V."""
    w = small_decode(31 + bs, [1, bs - 1, bs, bs + 1, 3 * bs + 2], hq=6, hkv=3, d=d, block_size=bs)
    p, b = w.pool, w.decode
    got = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    ref = sdpa_decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16, 3)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert np.isfinite(got).all()


def test_paged_equals_materialised_contiguous():
    w = small_decode(21, [3, 16, 33, 64, 129], hq=6, hkv=3, d=32)
    p, b = w.pool, w.decode
    a = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    c = oracle.naive_contiguous(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12)
    assert np.isfinite(a).all()        # NaN canaries in unowned slots and the poison block were never read


def test_block_relabelling_invariance():
    w = small_decode(22, [5, 31, 48, 77], hq=4, hkv=2, d=16, extra_blocks=6)
    p, b = w.pool, w.decode
    pi = wl.permutation(99, p.num_blocks)
    k2 = np.empty_like(p.k_cache)
    v2 = np.empty_like(p.v_cache)
    k2[pi] = p.k_cache
    v2[pi] = p.v_cache
    bt2 = pi[b.block_tables].astype(np.int32)
    a = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    c = oracle.decode(b.q, k2, v2, bt2, b.context_lens, b.scale, BF16)
    assert np.array_equal(a, c)


def test_single_token_returns_v_exactly():
    w = small_decode(23, [1, 1, 1], hq=4, hkv=2, d=16)
    p, b = w.pool, w.decode
    out = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    for s in range(3):
        v0 = f64(p.v_cache[b.block_tables[s, 0], 0], BF16)  # [Hkv, D]
        for h in range(4):
            assert np.array_equal(out[s, h], v0[h // 2])


def test_uniform_v_returns_that_v():
    w = small_decode(24, [50], hq=2, hkv=1, d=8)
    p, b = w.pool, w.decode
    vrow = wl.normal_bits(5, 8, BF16)
    v = p.v_cache.copy()
    v[:, :, 0, :] = vrow
    out = oracle.decode(b.q, p.k_cache, v, b.block_tables, b.context_lens, b.scale, BF16)
    np.testing.assert_allclose(out[0], np.broadcast_to(f64(vrow, BF16), (2, 8)), rtol=1e-12, atol=1e-15)


def test_equal_scores_give_mean_of_v():
    w = small_decode(25, [37], hq=2, hkv=1, d=8)
    p, b = w.pool, w.decode
    k = p.k_cache.copy()
    k[:, :, 0, :] = wl.normal_bits(6, 8, BF16)        # every key row identical
    out = oracle.decode(b.q, k, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    V = f64(materialise(p.v_cache, b.block_tables[0], 37), BF16)[:, 0, :]
    np.testing.assert_allclose(out[0, 0], V.mean(axis=0), rtol=0, atol=1e-13)


def _manual_case(kvals, vvals, qvals, scale, dtype=F16, bs=4):
    """One sequence, one head, exact small-integer inputs written straight into a pool."""
    L, D = len(kvals), len(qvals)
    nb = -(-L // bs) + 1
    k = np.zeros((nb, bs, 1, D), np.uint16)
    v = np.zeros((nb, bs, 1, D), np.uint16)
    bt = np.array([[nb - 1 - i for i in range(nb - 1)]], np.int32)  # reversed physical order
    for t in range(L):
        k[bt[0, t // bs], t % bs, 0] = np.asarray(kvals[t], np.float16).view(np.uint16)
        v[bt[0, t // bs], t % bs, 0] = np.asarray(vvals[t], np.float16).view(np.uint16)
    q = np.asarray([[qvals]], np.float16).view(np.uint16)
    return oracle.decode(q, k, v, bt, np.array([L], np.int32), scale, dtype, want_weights=True)


def test_two_token_sigmoid_closed_form():
    # s0 = scale*(q.k0) = 0.5*1 ; s1 = 0.5*3  ->  o = V0 + (V1 - V0) * sigmoid(s1 - s0)
    out, w = _manual_case([[1, 0], [1, 1]], [[2, -1], [-4, 3]], [1, 2], 0.5)
    sig = 1.0 / (1.0 + math.exp(-(1.5 - 0.5)))
    expect = np.array([2 + (-6) * sig, -1 + 4 * sig])
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-14)
    np.testing.assert_allclose(w[0, 0, :2], [1 - sig, sig], rtol=0, atol=1e-15)


def test_weights_sum_to_one_and_follow_score_differences():
    # integer q, k: s_t = scale * (q . k_t) exactly; ratio w_i / w_j = exp(s_i - s_j)
    ks = [[1, 0, 0], [0, 1, 0], [0, 0, 1], [1, 1, 1], [-2, 0, 1]]
    q = [1, -1, 2]
    scores = [0.25 * sum(a * b for a, b in zip(q, kk)) for kk in ks]
    out, w = _manual_case(ks, [[1, 0, 0]] * 5, q, 0.25)
    w = w[0, 0, :5]
    assert abs(w.sum() - 1.0) < 1e-15
    for i in range(5):
        for j in range(5):
            assert abs(w[i] / w[j] - math.exp(scores[i] - scores[j])) < 1e-13


def test_large_scores_are_stable_and_pick_the_max():
    # scores of +-1000: a naive exp would overflow; the max-subtracted form gives a one-hot result
    ks = [[10, 0], [0, 10], [-10, 0]]
    vs = [[1, 2], [3, 4], [5, 6]]
    out, w = _manual_case(ks, vs, [100, 1], 1.0)   # scores 1000, 10, -1000
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out[0, 0], [1, 2], rtol=0, atol=1e-12)


def test_brute_force_tiny_integer_inputs():
    # every (L, D) with tiny integer inputs: exact scores; compare with a Fraction-free
    # sum of exp over explicit scores (math.fsum), independently of the oracle's loops.
    rng = np.random.default_rng(5)
    for D in (1, 2, 4):
        for L in range(1, 6):
            ks = rng.integers(-3, 4, (L, D)).tolist()
            vs = rng.integers(-3, 4, (L, D)).tolist()
            q = rng.integers(-3, 4, D).tolist()
            out, _ = _manual_case(ks, vs, q, 0.5)
            s = [0.5 * sum(a * b for a, b in zip(q, kk)) for kk in ks]
            e = [math.exp(x) for x in s]
            den = math.fsum(e)
            expect = [math.fsum(e[t] * vs[t][d] for t in range(L)) / den for d in range(D)]
            np.testing.assert_allclose(out[0, 0], expect, rtol=1e-13, atol=1e-13)


def test_gqa_groups_are_consecutive_heads():
    # kv head 0 holds V = +1 everywhere, kv head 1 holds V = -1: query heads 0,1 must read +1, 2,3 must read -1
    w = small_decode(26, [20, 9], hq=4, hkv=2, d=8)
    p, b = w.pool, w.decode
    v = p.v_cache.copy()
    v[:, :, 0, :] = np.float32(1.0).view(np.uint32) >> 16
    v[:, :, 1, :] = np.float32(-1.0).view(np.uint32) >> 16
    out = oracle.decode(b.q, p.k_cache, v, b.block_tables, b.context_lens, b.scale, BF16)
    assert np.array_equal(out[:, :2], np.ones((2, 2, 8)))
    assert np.array_equal(out[:, 2:], -np.ones((2, 2, 8)))


def test_zero_length_context_gives_zeros():
    w = small_decode(27, [0 + 1, 5], hq=2, hkv=1, d=8)
    p, b = w.pool, w.decode
    cl = b.context_lens.copy()
    cl[0] = 0
    out = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, cl, b.scale, BF16)
    assert np.array_equal(out[0], np.zeros((2, 8)))


# --------------------------------------------------------------- split-K pieces


def test_partitions_merge_to_the_full_result():
    w = small_decode(31, [1, 255, 256, 257, 700, 1030], hq=4, hkv=2, d=16)
    p, b = w.pool, w.decode
    m, l, o = oracle.decode_partitions(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16, 256)
    full = oracle.decode(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16)
    np.testing.assert_allclose(oracle.merge_partitions(m, l, o), full, rtol=0, atol=1e-12)


def test_each_partition_is_attention_over_its_token_range():
    w = small_decode(32, [600], hq=2, hkv=1, d=16)
    p, b = w.pool, w.decode
    m, l, o = oracle.decode_partitions(b.q, p.k_cache, p.v_cache, b.block_tables, b.context_lens, b.scale, BF16, 256)
    assert m.shape[2] == 3
    for part in range(3):
        n = min(256, 600 - 256 * part)
        bt = np.ascontiguousarray(b.block_tables[:, 16 * part:])        # 256 tokens = 16 blocks of 16
        ref = oracle.decode(b.q, p.k_cache, p.v_cache, bt, np.array([n], np.int32), b.scale, BF16)
        np.testing.assert_allclose(o[0, :, part], ref[0], rtol=0, atol=1e-13)
        # l_p = sum exp(s_t - m_p) >= 1 (the max term contributes exactly 1)
        assert np.all(l[0, :, part] >= 1.0) and np.all(l[0, :, part] <= n)


# --------------------------------------------------------------- prefill chunk


def sdpa_prefill(pre, pool, n_kv_heads, dtype):
    T, Hq, D = pre.q.shape
    G = Hq // n_kv_heads
    out = np.zeros((T, Hq, D))
    for c in range(pre.num_chunks):
        r0, r1 = int(pre.query_start_loc[c]), int(pre.query_start_loc[c + 1])
        kv = int(pre.seq_lens[c])
        ctx = kv - (r1 - r0)
        K = torch.from_numpy(f64(materialise(pool.k_cache, pre.block_tables[c], kv), dtype)).permute(1, 0, 2)
        V = torch.from_numpy(f64(materialise(pool.v_cache, pre.block_tables[c], kv), dtype)).permute(1, 0, 2)
        q = torch.from_numpy(f64(pre.q[r0:r1], dtype)).permute(1, 0, 2)       # [Hq, q_len, D]
        j = torch.arange(r1 - r0)[:, None]
        t = torch.arange(kv)[None, :]
        mask = t <= ctx + j                                                     # bottom-right causal
        o = F.scaled_dot_product_attention(q, K.repeat_interleave(G, 0), V.repeat_interleave(G, 0),
                                           attn_mask=mask, scale=pre.scale)
        out[r0:r1] = o.permute(1, 0, 2).numpy()
    return out


def test_prefill_matches_torch_sdpa_bottom_right_mask():
    w = wl.build_workload("p", 41, dtype=BF16, n_q_heads=4, n_kv_heads=2, head_dim=16,
                          prefill_q_lens=[1, 7, 16, 33], prefill_ctx_lens=[0, 20, 5, 64])
    got = oracle.prefill_chunk(w.prefill.q, w.pool.k_cache, w.pool.v_cache, w.prefill.block_tables,
                               w.prefill.query_start_loc, w.prefill.seq_lens, w.prefill.scale, BF16)
    ref = sdpa_prefill(w.prefill, w.pool, 2, BF16)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bs,d,dt", [(8, 96, BF16), (32, 24, F16), (128, 8, BF16)])
def test_prefill_matches_torch_sdpa_other_block_sizes_and_widths(bs, d, dt):
    """The prefill oracle's block addressing at 8-, 32- and 128-token blocks (chunks and cached
    contexts straddling block boundaries) and widths that are not powers of two, against SDPA
    with the bottom-right mask over gathered K/V."""
    w = wl.build_workload("pb", 43 + bs, dtype=dt, n_q_heads=6, n_kv_heads=3, head_dim=d, block_size=bs,
                          prefill_q_lens=[1, bs + 1, 2 * bs - 1, 5],
                          prefill_ctx_lens=[bs - 1, 0, bs + 3, 3 * bs])
    pre, p = w.prefill, w.pool
    got = oracle.prefill_chunk(pre.q, p.k_cache, p.v_cache, pre.block_tables, pre.query_start_loc, pre.seq_lens,
                               pre.scale, dt)
    ref = sdpa_prefill(pre, p, 3, dt)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert np.isfinite(got).all()


def test_prefill_row_is_a_decode_row_with_shorter_context():
    w = wl.build_workload("p", 42, dtype=BF16, n_q_heads=4, n_kv_heads=2, head_dim=16,
                          prefill_q_lens=[9, 1], prefill_ctx_lens=[23, 0])
    pre, p = w.prefill, w.pool
    got = oracle.prefill_chunk(pre.q, p.k_cache, p.v_cache, pre.block_tables, pre.query_start_loc, pre.seq_lens,
                               pre.scale, BF16)
    for j in range(9):
        ref = oracle.decode(pre.q[j:j + 1], p.k_cache, p.v_cache, pre.block_tables[:1],
                            np.array([23 + j + 1], np.int32), pre.scale, BF16)
        assert np.array_equal(got[j], ref[0])
    # chunk with no cached context and one query row: attends to its own key only -> V0
    v0 = f64(p.v_cache[pre.block_tables[1, 0], 0], BF16)
    for h in range(4):
        assert np.array_equal(got[9, h], v0[h // 2])


# ------------------------------------------------------------------ rotary embedding (fused RoPE + KV write)
# Pins for the textbook rotation the oracle's fused write uses: each (i, i + D/2) pair turned
# by m * theta^(-2i/D).  Every pin is independent of the oracle's own formula.


def test_rope_one_pair_is_complex_multiplication():
    """D = 2, one pair, f_0 = 1: x0 + i x1 times e^{i m} (Python's complex arithmetic)."""
    import cmath
    for m in [0.0, 1.0, 2.5, 100.0, 12345.0]:
        for x0, x1 in [(1.0, 0.0), (0.3, -1.7), (-2.0, 0.5)]:
            z = complex(x0, x1) * cmath.exp(1j * m)
            got = oracle.rope_exact([x0, x1], m, 10000.0)
            assert abs(got[0] - z.real) < 1e-12 and abs(got[1] - z.imag) < 1e-12


def test_rope_pairing_frequencies_and_norm():
    """e_i moves only within the pair (i, i + D/2), by the angle m * theta^(-2i/D) (recovered with
    atan2), and every pair keeps its length."""
    D, theta, m = 128, 1.0e6, 37.0
    for i in [0, 1, 5, 31, 63]:
        x = np.zeros(D)
        x[i] = 1.0
        y = oracle.rope_exact(x, m, theta)
        nz = set(np.nonzero(np.abs(y) > 1e-15)[0].tolist())
        assert nz <= {i, i + D // 2}
        ang = math.atan2(y[i + D // 2], y[i])
        want = math.remainder(m * theta ** (-2.0 * i / D), 2 * math.pi)
        assert abs(math.remainder(ang - want, 2 * math.pi)) < 1e-9
    rng = np.random.default_rng(3)
    x = rng.standard_normal(D)
    y = oracle.rope_exact(x, 1234.0, theta)
    h = D // 2
    assert np.allclose(x[:h] ** 2 + x[h:] ** 2, y[:h] ** 2 + y[h:] ** 2, rtol=1e-12, atol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    """<R_m q, R_n k> == <R_{m+s} q, R_{n+s} k>: the property RoPE exists for."""
    D, theta = 64, 10000.0
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for m, n, s in [(5, 2, 100), (0, 7, 3), (1000, 999, 12345)]:
        a = float(np.dot(oracle.rope_exact(q, m, theta), oracle.rope_exact(k, n, theta)))
        b = float(np.dot(oracle.rope_exact(q, m + s, theta), oracle.rope_exact(k, n + s, theta)))
        assert abs(a - b) < 1e-9 * max(1.0, abs(a))


@pytest.mark.parametrize("dt", [BF16, F16])
def test_rope_kv_write_position_zero_and_row_handling(dt):
    """Position 0 is the identity (bit for bit); V rows are copied as by the plain write; a
    padded row rotates q but writes nothing; an out-of-range position leaves its row alone."""
    w = wl.write_rows_case(91, 12, n_kv_heads=2, head_dim=64, dtype=dt, pad_frac=0.0)
    p, wr = w.pool, w.write
    n = wr.key.shape[0]
    q = wl.normal_bits(wl.derive_seed(91, 7), n * 4 * 64, dt).reshape(n, 4, 64)
    sm = wr.slot_mapping.copy()
    sm[3] = -1
    pos = np.zeros(n, np.int64)
    pos[5:] = np.arange(5, n) * 17
    pos[7] = 1 << 40                      # out of range
    q2, k2, v2, st = oracle.rope_kv_write(q, p.k_cache, p.v_cache, wr.key, wr.value, sm, pos, 4096, 1.0e6, dt,
                                          check=False)
    assert st == oracle.EBOUNDS
    # V exactly as the plain write of the rows that are written
    keep = sm.copy()
    keep[7] = -1
    _, v_ref, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, keep, p.block_size)
    assert np.array_equal(v2, v_ref)
    flat_k = k2.reshape(-1, 2, 64)
    for i in range(n):
        if sm[i] < 0 or i == 7:
            continue
        if pos[i] == 0:
            assert np.array_equal(flat_k[sm[i]], wr.key[i])
        else:  # the written row is the rotation of the key row
            want = np.stack([oracle.round_to(oracle.rope_exact(f64(wr.key[i, h], dt), pos[i], 1.0e6), dt)
                             for h in range(2)])
            assert np.array_equal(flat_k[sm[i]], want)
    assert np.array_equal(q2[:5], q[:5])           # position 0: identity, padded row 3 included
    assert np.array_equal(q2[7], q[7])             # out of range: untouched
    assert not np.array_equal(q2[6], q[6])


def _rope_complex(x, m, theta):
    """The rotation written as complex multiplication with numpy: pair i is the complex number
    x[i] + i x[i + D/2], turned by e^{i m theta^(-2i/D)} -- independent of the oracle's code."""
    h = x.size // 2
    f = theta ** (-2.0 * np.arange(h) / x.size)
    z = (x[:h] + 1j * x[h:]) * np.exp(1j * m * f)
    return np.concatenate([z.real, z.imag])


@pytest.mark.parametrize("dt", [BF16, F16])
@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (8, 2, 128), (2, 2, 96)])
def test_rope_kv_write_query_rows_every_head(dt, hq, hkv, d):
    """Every head of every query row at a non-zero position equals the rounded rotation of that
    head alone, as numpy's complex multiplication gives it (and as the oracle's exact rotation
    gives it); a padded (-1) row still rotates its query at its own position.  Query heads and KV
    heads differ in number, so a query branch that used the key-head count as its stride, or
    rotated a padded row at another row's position, fails here (mini_engine, "Roadmap": RoPE
    folded into the KV-cache write; "Features": GQA)."""
    theta, maxpos = 1.0e6, 1 << 20
    w = wl.write_rows_case(93 + hq + d, 10, n_kv_heads=hkv, head_dim=d, dtype=dt, pad_frac=0.0)
    p, wr = w.pool, w.write
    n = wr.key.shape[0]
    q = wl.normal_bits(wl.derive_seed(93, hq + d), n * hq * d, dt).reshape(n, hq, d)
    sm = wr.slot_mapping.copy()
    sm[[2, 7]] = -1                                   # padded rows, non-zero positions below
    pos = (np.arange(n, dtype=np.int64) * 7919 + 13) % maxpos
    pos[4] = maxpos - 1
    q2, k2, _, st = oracle.rope_kv_write(q, p.k_cache, p.v_cache, wr.key, wr.value, sm, pos, maxpos, theta, dt)
    assert st == oracle.OK and (pos > 0).all()
    for i in range(n):
        for h in range(hq):
            x = f64(q[i, h], dt)
            want = oracle.round_to(_rope_complex(x, float(pos[i]), theta), dt)
            assert np.array_equal(q2[i, h], oracle.round_to(oracle.rope_exact(x, pos[i], theta), dt)), (i, h)
            # the numpy rotation rounds the same except where an exact value sits within a few
            # ulps of 1e-16 of a rounding boundary
            diff = np.abs(f64(q2[i, h], dt) - f64(want, dt))
            assert (diff <= 2.0 ** -6 * np.maximum(np.abs(f64(want, dt)), 1e-30) + 1e-300).all(), (i, h)
            assert (q2[i, h] == want).mean() > 0.98, (i, h)
    # keys of the padded rows were not written anywhere new: the cache equals the write of the
    # other rows
    keep = sm >= 0
    _, k_ref, _, _ = oracle.rope_kv_write(None, p.k_cache, p.v_cache, wr.key[keep], wr.value[keep], sm[keep],
                                          pos[keep], maxpos, theta, dt)
    assert np.array_equal(k2, k_ref)
