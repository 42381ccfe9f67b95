"""The bench's algorithmic byte and flop counts (the roofline numerators), pinned on small
cases against the definitions they state: K/V over all contexts + q + out + block-table
entries (+ the context lengths) for decode, K and V rows read and written for the write,
4 D flops per visible (query row, key) pair and head for prefill."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def test_decode_bytes_single_request_workload():
    # 1 sequence, 2/2 heads, hd 64, fp16, 128 tokens in 8 blocks: K/V 65,536 B, q 256 B, out 256 B,
    # 8 table entries 32 B (66,080 B), plus the 4-byte context length
    w = wl.make_workload(1)
    assert bench.decode_bytes(w.decode, w.pool) == 65536 + 256 + 256 + 32 + 4


def test_decode_bytes_counts_each_context_token_once_per_kv_head():
    w = wl.build_workload("acc", 3, dtype=wl.BF16, n_q_heads=8, n_kv_heads=2, head_dim=128, decode_lens=[1, 17, 40])
    tokens = 1 + 17 + 40
    expect = tokens * 2 * 2 * 128 * 2 + 2 * w.decode.q.nbytes + (1 + 2 + 3) * 4 + 3 * 4
    assert bench.decode_bytes(w.decode, w.pool) == expect
    # no shared blocks: the unique count is the same
    assert bench.unique_decode_bytes(w.decode, w.pool) == expect


def test_unique_bytes_count_a_shared_prefix_once():
    w = wl.build_workload("shared", 4, dtype=wl.BF16, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          decode_lens=[40, 50, 33], shared_prefix_blocks=2)
    logical, unique = bench.decode_bytes(w.decode, w.pool), bench.unique_decode_bytes(w.decode, w.pool)
    per_token = 2 * 2 * 64 * 2
    assert logical - unique == 2 * 32 * per_token   # two of the three sequences re-read 32 prefix tokens


def test_write_bytes_batch_256_step():
    w = wl.make_workload(4)
    valid = int((w.write.slot_mapping >= 0).sum())
    assert valid == 256 - 26
    assert bench.write_bytes(w.write, w.pool) == 2 * valid * (8 * 128 * 2) * 2 + 256 * 8


def test_prefill_flops_against_the_mask():
    """Brute force: count the (row, key) pairs the bottom-right causal mask leaves visible."""
    w = wl.build_workload("pf", 5, dtype=wl.BF16, n_q_heads=4, n_kv_heads=2, head_dim=64,
                          prefill_q_lens=[1, 5, 3], prefill_ctx_lens=[0, 7, 2])
    pre = w.prefill
    pairs = 0
    for c in range(3):
        q_len = int(pre.query_start_loc[c + 1] - pre.query_start_loc[c])
        kv_len = int(pre.seq_lens[c])
        for j in range(q_len):
            pairs += sum(1 for t in range(kv_len) if t <= kv_len - q_len + j)
    assert bench.prefill_flops(pre, 4, 64) == 4 * 64 * 4 * pairs


def test_rope_write_bytes_counts_query_rows_and_table_rows():
    w = wl.write_rows_case(9, 40, pad_frac=0.25)
    n = 40
    w.rope = dict(q=np.zeros((n, 16, 128), np.uint16), positions=np.zeros(n, np.int64))
    valid = int((w.write.slot_mapping >= 0).sum())
    row = 8 * 128 * 2
    assert bench.rope_write_bytes(w) == 16 * n + 2 * n * 16 * 128 * 2 + valid * (4 * row + 128 * 4)
