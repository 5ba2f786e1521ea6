"""Invariants of the seeded input generators (host logic, CPU only).

The rules checked here are the ones the pages state for the inputs of the
path: the slot formula and the decode-block rule (can_append), the
last-block-never-hit rule of the prefix cache, the token budget and
first-sequence-only chunking of the scheduler, and graph padding with slot -1.
"""

import os

import numpy as np
import pytest

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nano_vllm_constants.txt")


def golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split(None, 1)
                vals[k] = v
    return vals


def test_golden_constants_match_generators():
    g = golden()
    assert int(g["block_size"]) == W.BLOCK_SIZE
    assert int(g["pad_slot"]) == -1
    sizes = [int(x) for x in g["graph_batch_sizes"].split(",")]
    assert sizes == [1, 2, 4, 8] + list(range(16, 513, 16))
    assert int(g["max_num_seqs"]) >= 512


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1e-40], np.float32)
    b = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(b)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0 + 2**-6)
    assert back[3] == -2.5


def test_normal_bf16_deterministic_and_chunk_independent():
    a = W.normal_bf16((3, 1 << 21), 5, 1)
    b = W.normal_bf16((3, 1 << 21), 5, 1)
    assert np.array_equal(a, b)
    f = W.bf16_bits_to_f32(a)
    assert abs(f.mean()) < 0.01 and abs(f.std() - 1) < 0.01


def _check_decode(w: W.DecodeWorkload):
    bs = w.block_size
    shared = set(int(x) for x in w.shared_blocks)
    for b in range(w.batch):
        L = int(w.context_lens[b])
        row = w.block_tables[b]
        if b >= w.real_batch:
            assert L == 0 and w.slot_mapping[b] == -1 and (row == -1).all()
            continue
        nb = int((row >= 0).sum())
        assert nb == -(-L // bs)                       # ceil(L / bs) blocks
        assert (row[:nb] >= 0).all() and (row[nb:] == -1).all()
        s = int(w.slot_mapping[b])
        assert s == int(row[(L - 1) // bs]) * bs + (L - 1) % bs   # slot formula
        # can_append: a new block is needed exactly when len % bs == 1, i.e.
        # when the new token is the first of its block
        assert W.decode_needs_new_block(L, bs) == (s % bs == 0)
        assert int(row[(L - 1) // bs]) not in shared   # writes never hit shared blocks
    real = w.slot_mapping[: w.real_batch]
    assert len(set(real.tolist())) == real.size      # no duplicate slots


def test_tiny_decode():
    w = W.tiny_decode()
    assert w.batch == 4 and w.num_blocks == 16
    assert ((w.context_lens >= 1) & (w.context_lens <= 600)).all()
    _check_decode(w)


def test_qwen3_0p6b_decode_metadata():
    w = W.qwen3_0p6b_decode(fill_caches=False)
    assert w.batch == 256 and w.num_q_heads == 16 and w.num_kv_heads == 8
    assert ((w.context_lens >= 100) & (w.context_lens <= 2048)).all()
    need = sum(-(-int(L) // 256) for L in w.context_lens)
    assert w.num_blocks == int(np.ceil(need * 1.1))
    _check_decode(w)


def test_graph_padded_decode_metadata():
    w = W.graph_padded_decode(fill_caches=False)
    assert w.batch == 512 and w.real_batch == 500
    _check_decode(w)
    shared_rows = [b for b in range(500) if w.info["shared_counts"][b] > 0]
    assert 60 <= len(shared_rows) <= 100
    refs = np.bincount(w.block_tables[w.block_tables >= 0], minlength=w.num_blocks)
    assert refs.max() > 1                              # reference count above one
    assert set(np.nonzero(refs > 1)[0].tolist()) <= set(w.shared_blocks.tolist())


def test_qwen3_8b_decode_metadata():
    w = W.qwen3_8b_decode(fill_caches=False)
    assert w.batch == 64 and w.num_q_heads == 32 and w.num_blocks == 8192
    assert ((w.context_lens >= 8192) & (w.context_lens <= 32768)).all()
    _check_decode(w)


def test_chunked_prefill_prefix_rules():
    w = W.chunked_prefill_prefix(fill_caches=False)
    g = golden()
    budget = int(g["max_num_batched_tokens"])
    n = w.seqlens_q
    L = w.seqlens_k
    c = L - n
    assert n.sum() <= budget
    # the first candidate that was not admitted would have exceeded the budget
    assert w.info["admitted"] < 40
    # seq 0 continues a chunk split mid-prompt (not block aligned)
    assert c[0] > 0 and c[0] % 256 != 0
    # prefix hits are whole blocks, never the last block
    hits = np.array(w.info["shared_counts"])
    for i in range(1, w.num_seqs):
        if hits[i]:
            assert c[i] == 256 * hits[i]
            assert hits[i] <= -(-int(L[i]) // 256) - 1
            assert list(w.block_tables[i, :hits[i]]) == list(w.shared_blocks[:hits[i]])
        else:
            assert c[i] == 0
    # every new token's slot follows the formula and lands in a private block
    shared = set(w.shared_blocks.tolist())
    for i in range(w.num_seqs):
        for j in range(int(n[i])):
            p = int(c[i]) + j
            s = int(w.slot_mapping[w.cu_seqlens_q[i] + j])
            assert s == int(w.block_tables[i, p // 256]) * 256 + p % 256
            assert s // 256 not in shared


def test_prefill_8b_metadata():
    w = W.qwen3_8b_prefill(fill_caches=False)
    assert w.num_seqs == 4 and w.total_q == 32768 and (w.seqlens_k == 8192).all()


def test_cache_fill_history_and_stale():
    w = W.tiny_decode()
    for b in range(w.batch):
        L = int(w.context_lens[b])
        row = w.block_tables[b]
        for p in (0, L - 2, L - 1, L):
            if p < 0 or p >= 256 * int((row >= 0).sum()):
                continue
            blk, off = int(row[p // 256]), p % 256
            stale = p >= L - 1
            assert ((w.k_cache[blk, off] == W.SENTINEL_K).all()) == stale
            assert ((w.v_cache[blk, off] == W.SENTINEL_V).all()) == stale
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    for blk in set(range(w.num_blocks)) - used:
        assert (w.k_cache[blk] == W.SENTINEL_K).all()


def test_graph_bucket_sizes_match_the_page():
    from paged_kv_cache_304_gb300.graphs import graph_batch_sizes
    sizes = [int(x) for x in golden()["graph_batch_sizes"].split(",")]
    assert graph_batch_sizes(512) == sizes
    assert graph_batch_sizes(8) == [1, 2, 4, 8]
    assert graph_batch_sizes(40) == [1, 2, 4, 8, 16, 32, 40]
