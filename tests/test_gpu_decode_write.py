"""GPU parity of pa_decode_write, one decode step in one call: sequence s's new K/V row goes
into slot_mapping[s] (the slot of its last context token, -1 for none), then every sequence is
decoded over a context that includes that row.  It must leave the caches and the output bit for
bit as pa_reshape_and_cache followed by pa_decode does, whichever grid the dispatcher picks (the
persistent one-pass grid and the dynamic split-K grid write the rows from inside the decode CTAs;
the other grids launch the KV-write kernel first), and match the oracle's write-then-decode.
Source: mini_engine, "Custom CUDA kernels" (the KV-cache write and the paged decode of a step);
miniserve, "Engine" (slot mapping)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_232_gb300 as pa
import workloads as wl
from pa_testutil import abs_bits, bits_of, check_attention, to_dev, to_dev_i

pytestmark = pytest.mark.gpu


def _case(name):
    """(workload, description): every one carries a write batch of one row per sequence at its
    last position, some rows padded with -1."""
    if name == "step256":
        return wl.make_workload(4)      # batch 256, group 2: the persistent grid
    lens = lambda seed, n, lo, hi: [int(x) for x in wl.uniform_ints(wl.derive_seed(seed, 1), n, lo, hi)]
    if name == "decode64":              # 64 sequences: the dynamic split-K grid
        return wl.build_workload(name, 61, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=128,
                                 decode_lens=lens(61, 64, 100, 2048), write_rows=True, n_padded=6)
    if name == "g1_hd64_bs8":           # 1000 x 2 units at group 1, 8-token blocks: persistent grid
        return wl.build_workload(name, 62, dtype=wl.F16, n_q_heads=2, n_kv_heads=2, head_dim=64, block_size=8,
                                 decode_lens=lens(62, 1000, 1, 300), write_rows=True, n_padded=100)
    if name == "hd96_bs32":             # 600 x 8 units at group 2, head_dim 96, 32-token blocks
        return wl.build_workload(name, 63, dtype=wl.BF16, n_q_heads=16, n_kv_heads=8, head_dim=96, block_size=32,
                                 decode_lens=lens(63, 600, 1, 500), write_rows=True, n_padded=60)
    if name == "few_long":              # 4 long contexts: split-K on the static grid
        return wl.build_workload(name, 64, dtype=wl.BF16, n_q_heads=32, n_kv_heads=8, head_dim=128,
                                 decode_lens=[9000, 17, 4096, 12000], write_rows=True, n_padded=1)
    raise KeyError(name)


def _run(w, fused, slots=None):
    p, b, wr = w.pool, w.decode, w.write
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    q = to_dev(b.q, p.dtype)
    out = torch.full_like(q, float("nan"))
    bt, cl = to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32)
    key, val = to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype)
    sm = to_dev_i(wr.slot_mapping if slots is None else slots, torch.int64)
    maxL = int(b.context_lens.max())
    S, hq, d = b.q.shape
    ws = torch.full((max(16, pa.pa_decode_workspace_size(S, hq, d, maxL, 0)),), 0x7F, dtype=torch.uint8,
                    device="cuda")
    if fused:
        pa.pa_decode_write(out, q, kc, vc, bt, cl, maxL, b.scale, key, val, sm, ws)
    else:
        pa.pa_reshape_and_cache(key, val, kc, vc, sm)
        pa.pa_decode(out, q, kc, vc, bt, cl, maxL, b.scale, ws)
    torch.cuda.synchronize()
    return bits_of(out), bits_of(kc), bits_of(vc)


@pytest.mark.parametrize("name", ["step256", "decode64", "g1_hd64_bs8", "hd96_bs32", "few_long"])
def test_decode_write_equals_write_then_decode(name):
    w = _case(name)
    p, b, wr = w.pool, w.decode, w.write
    pa.pa_device_errors(clear=True)
    fo, fk, fv = _run(w, fused=True)
    assert pa.pa_device_errors(clear=True) == 0
    so, sk, sv = _run(w, fused=False)
    assert pa.pa_device_errors(clear=True) == 0
    assert np.array_equal(fk, sk) and np.array_equal(fv, sv), "caches differ from the separate write"
    assert np.array_equal(fo, so), "output differs from write-then-decode"
    k2, v2, _ = oracle.kv_write(p.k_cache, p.v_cache, wr.key, wr.value, wr.slot_mapping, p.block_size)
    assert np.array_equal(fk, k2) and np.array_equal(fv, v2)
    ex = oracle.decode(b.q, k2, v2, b.block_tables, b.context_lens, b.scale, p.dtype)
    cd = oracle.decode(b.q, k2, abs_bits(v2), b.block_tables, b.context_lens, b.scale, p.dtype)
    check_attention(fo, ex, p.dtype, f"decode_write {name}", cond=cd)


def test_decode_write_repeated_calls_bitwise():
    """The batch-256 step three times from the same inputs: the same bits every time (the rows are
    written before the chunks holding them are read, on every call)."""
    w = _case("step256")
    first = _run(w, fused=True)
    for _ in range(3):
        again = _run(w, fused=True)
        assert all(np.array_equal(a, c) for a, c in zip(first, again))
    assert pa.pa_device_errors(clear=True) == 0


@pytest.mark.parametrize("name", ["step256", "decode64"])
def test_decode_write_flags_slots_it_cannot_place(name):
    """On the persistent grid (batch 256) and the dynamic grid (batch 64): a slot past the pool
    writes nothing and sets PA_DEVERR_SLOT, as the KV-write kernel does; an in-pool slot that is
    not the sequence's last token is still written (the caches match the separate write) and also
    sets PA_DEVERR_SLOT."""
    w = _case(name)
    p, b, wr = w.pool, w.decode, w.write
    slots = wr.slot_mapping.copy()
    live = np.flatnonzero(slots >= 0)
    slots[live[0]] = p.num_blocks * p.block_size + 5           # outside the pool
    s1 = int(live[1])
    L = int(b.context_lens[s1])
    assert L >= 2
    slots[s1] = int(b.block_tables[s1, (L - 2) // p.block_size]) * p.block_size + (L - 2) % p.block_size
    pa.pa_device_errors(clear=True)
    _, fk, fv = _run(w, fused=True, slots=slots)
    assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_SLOT
    _, sk, sv = _run(w, fused=False, slots=slots)
    assert pa.pa_device_errors(clear=True) & pa.PA_DEVERR_SLOT
    assert np.array_equal(fk, sk) and np.array_equal(fv, sv)


def test_decode_write_argument_errors():
    w = _case("decode64")
    p, b, wr = w.pool, w.decode, w.write
    kc, vc = to_dev(p.k_cache, p.dtype), to_dev(p.v_cache, p.dtype)
    q = to_dev(b.q, p.dtype)
    out = torch.empty_like(q)
    bt, cl = to_dev_i(b.block_tables, torch.int32), to_dev_i(b.context_lens, torch.int32)
    key, val = to_dev(wr.key, p.dtype), to_dev(wr.value, p.dtype)
    sm = to_dev_i(wr.slot_mapping, torch.int64)
    with pytest.raises(ValueError):
        pa.pa_decode_write(out, q, kc, vc, bt, cl, 2048, b.scale, key[:10], val, sm)
    with pytest.raises(ValueError):
        pa.pa_decode_write(out, q, kc, vc, bt, cl, 2048, b.scale, key, val, sm[:10])
    with pytest.raises(pa.PagedAttnError) as e:
        pa.pa_decode_write(out, q, kc, vc, bt, cl, 10 ** 6, b.scale, key, val, sm)
    assert e.value.status == -5
