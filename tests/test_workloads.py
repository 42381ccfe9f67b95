"""The seeded input generator: pinned to the published SplitMix64 outputs, to a
direct Box-Muller evaluation in Python, and to library fp16/bf16 rounding."""
import math

import numpy as np
import torch

import workloads as wl
from workloads import BF16, F16

MASK = 2**64 - 1


def splitmix_py(seed, n):
    """SplitMix64 written from its definition with Python integers."""
    out, s = [], seed
    for _ in range(n):
        s = (s + 0x9E3779B97F4A7C15) & MASK
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_vector():
    # first outputs of SplitMix64 seeded with 1234567, as printed with the reference implementation
    assert list(wl.splitmix64(1234567, 0, 3)) == [6457827717110365317, 3203168211198807973, 9817491932198370423]
    assert list(wl.splitmix64(42, 0, 50)) == splitmix_py(42, 50)
    assert list(wl.splitmix64(42, 20, 5)) == splitmix_py(42, 25)[20:]   # counter-based random access


def test_box_muller_normals():
    seed = 77
    u = splitmix_py(seed, 8)
    for e in range(8):
        u1 = ((u[2 * (e // 2)] >> 11) + 1) / 2.0**53
        u2 = ((u[2 * (e // 2) + 1] >> 11) + 1) / 2.0**53
        r = math.sqrt(-2.0 * math.log(u1))
        z = r * (math.sin if e % 2 else math.cos)(2 * math.pi * u2)
        assert abs(wl.lib().wl_normal_f64_at(seed, e) - z) < 1e-12
    x = wl.normal_f32(3, 400_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_narrowing_matches_library_rounding():
    f32 = wl.normal_f32(9, 100_000)
    assert np.array_equal(wl.normal_bits(9, 100_000, F16), f32.astype(np.float16).view(np.uint16))
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.normal_bits(9, 100_000, BF16), ref)
    # slices regenerate identically
    assert np.array_equal(wl.normal_bits(9, 10, BF16, start=500), wl.normal_bits(9, 600, BF16)[500:510])


def test_bounded_ints_and_permutations():
    x = wl.uniform_ints(5, 200_000, 100, 2048)
    assert x.min() == 100 and x.max() == 2048
    assert abs(x.mean() - 1074) < 10
    p = wl.permutation(6, 1000)
    assert np.array_equal(np.sort(p), np.arange(1000))
    assert not np.array_equal(p, np.arange(1000))


def test_workload_structure():
    w = wl.make_workload(1)
    assert w.pool.k_cache.shape == (64, 16, 2, 64) and w.decode.block_tables.shape == (1, 8)
    assert len(set(w.decode.block_tables[0].tolist())) == 8
    w = wl.make_workload(4)
    assert (w.write.slot_mapping == -1).sum() == 26
    s = w.write.slot_mapping
    assert len(set(s[s >= 0].tolist())) == (s >= 0).sum()        # distinct slots
    L = w.decode.context_lens.astype(np.int64)
    rows = np.nonzero(s >= 0)[0]
    # each written slot is the slot of position L-1 of its sequence
    assert np.array_equal(s[rows], w.decode.block_tables[rows, (L[rows] - 1) // 16].astype(np.int64) * 16
                          + (L[rows] - 1) % 16)
    w = wl.make_workload(5)
    assert np.all(w.decode.block_tables[:, :64] == w.decode.block_tables[0, :64])
    assert w.prefill.seq_lens[0] == 512 and w.prefill.seq_lens[7] == 4096 + 512
    # NaN canaries: every slot nobody owns is NaN, every owned slot finite
    nanbits = wl.NAN_BITS[BF16]
    assert np.all(w.pool.k_cache[~w.pool.valid] == nanbits)
    assert not np.any(w.pool.k_cache[w.pool.valid] == nanbits)
