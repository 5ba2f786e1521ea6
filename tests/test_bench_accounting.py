"""The benchmark's work accounting (algorithmic bytes and flops), checked by
brute-force counting on small workloads."""

import numpy as np

import bench
import workloads as W


def test_decode_bytes_counts_every_row_once_per_sequence():
    w = W.make_decode("acct", 901, [1, 255, 256, 257, 600], 16, 8, num_blocks=12, fill_caches=False)
    row = 8 * 128 * 2  # one token row of K (or V)
    kv = sum(int(L) * row * 2 for L in w.context_lens)
    qo = len(w.context_lens) * 16 * 128 * 2 * 2
    meta = sum(-(-int(L) // 256) for L in w.context_lens) * 4 + len(w.context_lens) * 4
    assert bench.decode_bytes(w.context_lens, 16, 8) == kv + qo + meta


def test_unique_bytes_count_shared_prefix_rows_once():
    w = W.graph_padded_decode(fill_caches=False)
    full = bench.decode_bytes(w.context_lens, 16, 8)
    uniq = bench.decode_unique_bytes(w.context_lens, w.block_tables, 16, 8)
    # brute force: the set of (physical block, offset) rows any sequence reads
    rows = set()
    for b, L in enumerate(w.context_lens):
        for t in range(int(L)):
            rows.add((int(w.block_tables[b, t // 256]), t % 256))
    row = 8 * 128 * 2 * 2
    assert uniq == full - int(w.context_lens.sum()) * row + len(rows) * row
    assert uniq < full  # the workload shares prefix blocks
    w2 = W.qwen3_0p6b_decode(fill_caches=False)  # no sharing
    assert bench.decode_unique_bytes(w2.context_lens, w2.block_tables, 16, 8) == \
        bench.decode_bytes(w2.context_lens, 16, 8)


def test_prefill_flops_by_counting_visible_pairs():
    w = W.make_prefill("acct", 902, [1, 5, 130, 300], [0, 2, 0, 44], 16, 8, num_blocks=6, fill_caches=False)
    pairs = 0
    for n, L in zip(w.seqlens_q, w.seqlens_k):
        c = int(L) - int(n)
        pairs += sum(c + j + 1 for j in range(int(n)))  # query j sees keys 0 .. c + j
    assert bench.prefill_flops(w) == 4 * 128 * 16 * pairs


def test_write_bytes_skip_padding():
    slots = np.array([5, -1, 7, -1, 300], np.int32)
    assert bench.write_bytes(slots, 8) == 3 * 8 * 128 * 2 * 2 * 2 + 5 * 4
