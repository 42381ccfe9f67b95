"""GPU parity of pa_reshape_and_cache against the oracle: the whole cache must be
bit-identical after the write (written slots hold the rows, -1 rows and every other
slot unchanged)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import bits_of, to_dev, to_dev_i

pytestmark = pytest.mark.gpu


def run_write(w, slot_mapping=None):
    p, wr = w.pool, w.write
    dt = p.dtype
    sm = wr.slot_mapping if slot_mapping is None else slot_mapping
    kc, vc = to_dev(p.k_cache, dt), to_dev(p.v_cache, dt)
    pa.pa_reshape_and_cache(to_dev(wr.key, dt), to_dev(wr.value, dt), kc, vc, to_dev_i(sm, torch.int64))
    torch.cuda.synchronize()
    return bits_of(kc), bits_of(vc)


def assert_write_matches_oracle(w, slot_mapping=None, expect_status=oracle.OK):
    p, wr = w.pool, w.write
    sm = wr.slot_mapping if slot_mapping is None else slot_mapping
    pa.pa_device_errors(clear=True)
    gk, gv = run_write(w, sm)
    ok, ov, st = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, sm, p.block_size, check=False)
    assert st == expect_status
    assert np.array_equal(gk, ok), "k_cache differs from the oracle"
    assert np.array_equal(gv, ov), "v_cache differs from the oracle"
    return pa.pa_device_errors(clear=True)


def test_write_full_step_batch_256():
    w = wl.make_workload(4)
    assert assert_write_matches_oracle(w) == 0


def test_write_bandwidth_scale_64k_rows():
    w = wl.write_rows_case(232_104, 65536)
    assert assert_write_matches_oracle(w) == 0


@pytest.mark.parametrize("n,hkv,d,dt", [(1, 8, 128, wl.BF16), (3, 2, 64, wl.F16), (37, 1, 64, wl.BF16),
                                        (1023, 4, 128, wl.F16), (4099, 8, 64, wl.BF16), (513, 8, 96, wl.BF16),
                                        (300, 4, 256, wl.F16)])
def test_write_shapes_and_ragged_counts(n, hkv, d, dt):
    w = wl.write_rows_case(1000 + n, n, n_kv_heads=hkv, head_dim=d, dtype=dt, pad_frac=0.25, nan_canaries=True)
    assert assert_write_matches_oracle(w) == 0


@pytest.mark.parametrize("n,hkv,d,dt", [(300, 64, 128, wl.BF16), (257, 32, 256, wl.F16), (99, 24, 256, wl.BF16),
                                        (64, 40, 96, wl.F16)])
def test_write_wide_rows(n, hkv, d, dt):
    """Rows wider than 512 16-byte chunks per (K, V) pair (64 KV heads x 128, 32 x 256 ...): each
    thread copies several chunks; the cache is still bit-identical to the oracle's."""
    w = wl.write_rows_case(3000 + hkv + d, n, n_kv_heads=hkv, head_dim=d, dtype=dt, pad_frac=0.2, nan_canaries=True)
    assert assert_write_matches_oracle(w) == 0


def test_write_then_decode_wide_rows():
    """A cache of 64 KV heads x 128 is written and then decoded (group size 1): every shape the
    decode accepts can be written."""
    from pa_testutil import abs_bits, check_attention
    w = wl.build_workload("wide", 3100, dtype=wl.BF16, n_q_heads=64, n_kv_heads=64, head_dim=128,
                          decode_lens=[1, 130, 600], write_rows=True, n_padded=1)
    p, b, wr = w.pool, w.decode, w.write
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    pa.pa_reshape_and_cache(to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype), kc, vc,
                            to_dev_i(wr.slot_mapping, torch.int64))
    k2, v2, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, wr.slot_mapping, p.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(kc), k2) and np.array_equal(bits_of(vc), v2)
    q = to_dev(b.q, p.dtype)
    out = torch.empty_like(q)
    pa.pa_decode_v1(out, q, kc, vc, to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32),
                    b.scale)
    torch.cuda.synchronize()
    ex = oracle.decode(b.q, k2, v2, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, k2, abs_bits(v2), b.block_tables, b.context_lens, b.scale, p.dtype)
    check_attention(bits_of(out), ex, p.dtype, "decode after a wide write", cond=cd)
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("bs", [8, 32, 128])
def test_write_block_sizes(bs):
    w = wl.write_rows_case(2000 + bs, 777, n_kv_heads=4, head_dim=128, block_size=bs, pad_frac=0.2, nan_canaries=True)
    assert assert_write_matches_oracle(w) == 0


def test_write_all_padded_changes_nothing():
    w = wl.write_rows_case(5, 64)
    sm = np.full(64, -1, dtype=np.int64)
    assert assert_write_matches_oracle(w, sm) == 0
    gk, gv = run_write(w, sm)
    assert np.array_equal(gk, w.pool.k_cache) and np.array_equal(gv, w.pool.v_cache)


def test_write_out_of_pool_slot_is_flagged_and_dropped():
    w = wl.write_rows_case(6, 40, pad_frac=0.0)
    sm = w.write.slot_mapping.copy()
    sm[3] = w.pool.num_blocks * 16 + 7      # past the pool
    sm[9] = -5                               # negative, not the padding marker
    errs = assert_write_matches_oracle(w, sm, expect_status=oracle.EBOUNDS)
    assert errs & pa.PA_DEVERR_SLOT
