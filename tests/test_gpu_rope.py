"""GPU parity of pa_rope_reshape_and_cache (rotary embedding fused into the KV write) against
the fp64 oracle.

The kernel rotates in fp32 with float32 cos / sin from pa_rope_table; the oracle rotates in
double with cos / sin computed in double.  Both round each result once to the 16-bit format,
so a result differs where the exact value sits within ~1e-7 of a rounding boundary (one unit
in the last place, in fewer than 1 in 1000 elements), or where the pair nearly cancels
(x[i] cos ~ x[i + D/2] sin): there the fp32 error, ~2^-22 of the operands, spans several
ulps of the small result.  Rule: every element within one ulp of the rounded oracle, or else
|gpu - exact| <= half_ulp(exact) + 2^-21 (|x[i]| + |x[i + D/2]|) against the oracle's
unrounded rotation.  Values, untouched slots and untouched rows are compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, half_ulp, to_dev, to_dev_i, ulp_distance

pytestmark = pytest.mark.gpu

THETA = 1.0e6       # Qwen3's rotary base (the workloads are Qwen3-shaped)
MAX_POS = 32768


def assert_close_bits(got, want, what, source, dt):
    """got / want: 16-bit results; source(flat index) -> (input row as doubles, position, dim)
    for the oracle's unrounded rotation of the elements more than one ulp apart."""
    d = ulp_distance(got, want)
    frac = float((d == 1).mean())
    assert frac < 1e-3, f"{what}: {frac:.2e} of the elements are 1 ulp apart"
    far = np.flatnonzero(d > 1)
    assert far.size < 1e-3 * d.size, f"{what}: {far.size} elements more than 1 ulp apart"
    g = oracle.to_double(got.reshape(-1)[far], dt)
    for k, f in enumerate(far.tolist()):
        x, m, e = source(f)
        exact = oracle.rope_exact(x, m, THETA)[e]
        h = x.size // 2
        allow = half_ulp(np.array([exact]), dt)[0] + 2.0 ** -21 * (abs(x[e % h]) + abs(x[e % h + h]))
        assert abs(g[k] - exact) <= allow, f"{what}: element {f}: gpu {g[k]!r} exact {exact!r} allow {allow:.3e}"


def run_rope(w, q_bits, positions, slot_mapping=None, with_q=True, max_pos=MAX_POS):
    p, wr = w.pool, w.write
    sm = wr.slot_mapping if slot_mapping is None else slot_mapping
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    q = to_dev(q_bits, p.dtype) if with_q else None
    cs = pa.rope_cos_sin(max_pos, p.head_dim, THETA)
    pa.pa_rope_reshape_and_cache(to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype), kc, vc,
                                 to_dev_i(sm, torch.int64), to_dev_i(positions, torch.int64), cs, q=q)
    torch.cuda.synchronize()
    return (bits_of(q) if with_q else None), bits_of(kc), bits_of(vc)


def check_against_oracle(w, q_bits, positions, slot_mapping=None, with_q=True, max_pos=MAX_POS, expect=oracle.OK):
    p, wr = w.pool, w.write
    sm = wr.slot_mapping if slot_mapping is None else slot_mapping
    pa.pa_device_errors(clear=True)
    gq, gk, gv = run_rope(w, q_bits, positions, sm, with_q, max_pos)
    oq, ok_, ov, st = oracle.rope_kv_write(q_bits if with_q else None, p.k_cache, p.v_cache, wr.key, wr.value, sm,
                                           positions, max_pos, THETA, p.dtype, check=False)
    assert st == expect
    assert np.array_equal(gv, ov), "v_cache differs"
    nb, bs, hkv, d = p.k_cache.shape
    row_of_slot = {int(sl): i for i, sl in enumerate(sm.tolist()) if sl >= 0}

    def k_source(f):
        slot, h, e = f // (hkv * d), (f // d) % hkv, f % d
        i = row_of_slot[slot]
        return oracle.to_double(wr.key[i, h], p.dtype), int(positions[i]), e

    assert_close_bits(gk, ok_, "k_cache", k_source, p.dtype)
    # untouched slots of k_cache are bit-identical
    untouched = ok_ == p.k_cache
    assert np.array_equal(gk[untouched], ok_[untouched])
    if with_q:
        hq = q_bits.shape[1]

        def q_source(f):
            i, h, e = f // (hq * d), (f // d) % hq, f % d
            return oracle.to_double(q_bits[i, h], p.dtype), int(positions[i]), e

        assert_close_bits(gq, oq, "q", q_source, p.dtype)
    return pa.pa_device_errors(clear=True)


def test_rope_write_decode_step_batch_256():
    """The batch-256 decode step's write (256 rows, 26 padded) with the query rows and new keys at
    position context_len - 1."""
    w = wl.make_workload(4)
    b = w.decode
    pos = (b.context_lens.astype(np.int64) - 1)
    assert check_against_oracle(w, b.q, pos) == 0


def test_rope_write_bandwidth_scale_64k_rows():
    w = wl.write_rows_case(232_104, 65536)
    n = w.write.key.shape[0]
    pos = wl.uniform_ints(wl.derive_seed(232_104, 11), n, 0, MAX_POS - 1).astype(np.int64)
    q = wl.normal_bits(wl.derive_seed(232_104, 12), n * 16 * 128, wl.BF16).reshape(n, 16, 128)
    assert check_against_oracle(w, q, pos) == 0


@pytest.mark.parametrize("dt,hq,hkv,d,with_q", [(wl.F16, 8, 8, 64, True), (wl.BF16, 32, 8, 128, True),
                                               (wl.F16, 16, 4, 128, False), (wl.BF16, 2, 2, 64, True),
                                               (wl.BF16, 16, 8, 96, True), (wl.F16, 8, 4, 256, True)])
def test_rope_write_shapes(dt, hq, hkv, d, with_q):
    w = wl.write_rows_case(700 + hq + d, 333, n_kv_heads=hkv, head_dim=d, dtype=dt, pad_frac=0.2, nan_canaries=True)
    n = w.write.key.shape[0]
    pos = wl.uniform_ints(wl.derive_seed(700 + hq, 3), n, 0, 4999).astype(np.int64)   # inclusive bounds
    pos[:3] = [0, 1, 4999]
    q = wl.normal_bits(wl.derive_seed(700 + hq, 4), n * hq * d, dt).reshape(n, hq, d)
    assert check_against_oracle(w, q, pos, with_q=with_q, max_pos=5000) == 0


def test_rope_write_bad_positions_and_slots_are_flagged():
    w = wl.write_rows_case(95, 40, pad_frac=0.0)
    n = w.write.key.shape[0]
    pos = np.arange(n, dtype=np.int64) * 3
    pos[4] = -2
    pos[9] = MAX_POS              # one past the table
    sm = w.write.slot_mapping.copy()
    sm[12] = w.pool.num_blocks * 16 + 5
    q = wl.normal_bits(wl.derive_seed(95, 1), n * 16 * 128, wl.BF16).reshape(n, 16, 128)
    errs = check_against_oracle(w, q, pos, slot_mapping=sm, expect=oracle.EBOUNDS)
    assert errs & pa.PA_DEVERR_POSITION and errs & pa.PA_DEVERR_SLOT


def test_rope_write_then_decode_matches_oracle():
    """The fused write feeds decode: rotated q and rotated cached keys, against the oracle's
    own rotation followed by its decode."""
    w = wl.make_workload(2)
    p, b = w.pool, w.decode
    S = b.num_seqs
    # one new token per sequence at position L - 1, written to that position's slot
    L = b.context_lens.astype(np.int64)
    slots = np.array([b.block_tables[s, (L[s] - 1) // 16] * 16 + (L[s] - 1) % 16 for s in range(S)], np.int64)
    key = wl.normal_bits(wl.derive_seed(51, 1), S * 8 * 128, p.dtype).reshape(S, 8, 128)
    val = wl.normal_bits(wl.derive_seed(51, 2), S * 8 * 128, p.dtype).reshape(S, 8, 128)
    q, kc, vc = to_dev(b.q, p.dtype), to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    cs = pa.rope_cos_sin(MAX_POS, 128, THETA)
    pa.pa_device_errors(clear=True)
    pa.pa_rope_reshape_and_cache(to_dev(key, p.dtype), to_dev(val, p.dtype), kc, vc, to_dev_i(slots, torch.int64),
                                 to_dev_i(L - 1, torch.int64), cs, q=q)
    out = torch.empty_like(q)
    pa.pa_decode_v1(out, q, kc, vc, to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32),
                    b.scale)
    torch.cuda.synchronize()
    assert pa.pa_device_errors(clear=True) == 0
    # the oracle's own pipeline: its rotation, then its decode on its rotated q and cache
    oq, ok_, ov, _ = oracle.rope_kv_write(b.q, p.k_cache, p.v_cache, key, val, slots, L - 1, MAX_POS, THETA, p.dtype)
    ex = oracle.decode(oq, ok_, ov, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(oq, ok_, abs_bits(ov), b.block_tables, b.context_lens, b.scale, p.dtype)
    # the q / key rounding may differ by one ulp in rare elements: allow that score shift
    check_attention(bits_of(out), ex, p.dtype, "rope write + decode", cond=cd, rel=1e-4 + 2.0 ** -8)
