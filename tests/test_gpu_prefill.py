"""Varlen causal prefill attention on the GPU vs the fp64 oracle.

Each case writes the step's new tokens with the library's KV write (checked
bit-exact), runs prefill through the C ABI and compares with the oracle:
every output element at sizes the oracle finishes quickly, sampled rows (the
first and last rows of every query tile plus 1024 seeded rows per sequence)
at the 8B-shaped 4 x 8192 size.  Bar: max-abs <= 2e-2, mean-abs <= 2e-3.

The library has two prefill kernels, chosen by the stated max_seqlen_q: a
persistent one for batches of short query tiles (<= 2048, e.g. the chunked
16384-token step and every edge case here) and one CTA per query tile above
that (4 x 8192).  Both are checked against the oracle, and against each other
bit for bit on the same inputs.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_304_gb300 as pkv
import workloads as W
from tests.gpu_util import check_close, i32, to_dev, to_host

pytestmark = pytest.mark.gpu


def run_prefill(w: W.PrefillWorkload, rows=None, cu_q=None, q=None):
    """Write + prefill on the GPU; compare with the oracle on `rows`."""
    cu_q = w.cu_seqlens_q if cu_q is None else cu_q
    q = w.q if q is None else q
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    nq = np.diff(cu_q)
    out = pkv.paged_attn_prefill(to_dev(q), kc, vc, i32(cu_q), i32(w.cu_seqlens_k), i32(w.block_tables), w.scale,
                                 int(nq.max()) if nq.size else 0, w.max_seqlen_k)
    torch.cuda.synchronize()
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    assert np.array_equal(to_host(kc), okc) and np.array_equal(to_host(vc), ovc), "kv write not bit-exact"
    ref = oracle.paged_attn_prefill(q, okc, ovc, cu_q, w.cu_seqlens_k, w.block_tables, w.scale, rows=rows)
    got = to_host(out)
    res = check_close(got, ref, w.name, rows=rows)
    assert pkv.device_error() == []
    return res, got, ref


def test_prefill_chunked_prefix_budget16384():
    """33 admitted prompts, a split first sequence, 9 prefix-cache hits."""
    run_prefill(W.chunked_prefill_prefix())


def config5_rows(w: W.PrefillWorkload) -> np.ndarray:
    """Rows checked at 4 x 8192: the first and last row of every 128-row query
    tile of every sequence (so every query tile a CTA can own is covered),
    plus 1024 distinct seeded rows per sequence (about 4550 rows in all)."""
    rng = np.random.default_rng(8192)
    rows = []
    for i in range(w.num_seqs):
        lo, hi = int(w.cu_seqlens_q[i]), int(w.cu_seqlens_q[i + 1])
        starts = np.arange(lo, hi, 128)
        rows += list(starts) + list(np.minimum(starts + 127, hi - 1))
        rows += list(rng.choice(np.arange(lo, hi), size=min(1024, hi - lo), replace=False))
    return np.unique(np.array(rows))


def test_prefill_qwen3_8b_4x8192_sampled_rows():
    """Every query tile's first and last rows plus 1024 seeded rows per
    sequence; the fp64 oracle takes about half a minute on 8-16 host cores."""
    w = W.qwen3_8b_prefill()
    rows = config5_rows(w)
    tiles = set()
    for r in rows:
        i = int(np.searchsorted(w.cu_seqlens_q, r, side="right")) - 1
        tiles.add((i, (int(r) - int(w.cu_seqlens_q[i])) // 128))
    assert len(tiles) == sum(-(-int(n) // 128) for n in w.seqlens_q)
    run_prefill(w, rows=rows)


EDGE = [
    # (lengths, cached)
    ([1], [0]),
    ([2, 1, 3], [1, 0, 0]),
    ([127, 128, 129], [0, 0, 0]),
    ([255, 256, 257], [0, 0, 0]),
    ([300, 600], [255, 256]),
    ([513, 700, 1000], [257, 1, 511]),
    ([1025, 40], [896, 0]),
    ([2000], [1000]),
]


@pytest.mark.parametrize("lens,cached", EDGE, ids=[f"case{i}" for i in range(len(EDGE))])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8)])
def test_prefill_edges(lens, cached, hq, hkv):
    need = sum(-(-L // 256) for L in lens)
    w = W.make_prefill("edge", 700 + sum(lens), lens, cached, hq, hkv, num_blocks=need + 3)
    run_prefill(w)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 1), (64, 8), (12, 4), (4, 2)])
def test_prefill_group_sizes(hq, hkv):
    lens, cached = [700, 130, 1], [300, 0, 0]
    w = W.make_prefill("groups", 800 + hq + hkv, lens, cached, hq, hkv, num_blocks=10)
    run_prefill(w)


def test_prefill_empty_sequence_in_batch():
    """A sequence with no new tokens (n = 0) in the middle of the batch."""
    w = W.make_prefill("empty_mid", 811, [300, 200, 150], [10, 0, 20], 16, 8, num_blocks=8)
    n = np.diff(w.cu_seqlens_q)
    keep = np.r_[np.arange(w.cu_seqlens_q[0], w.cu_seqlens_q[1]), np.arange(w.cu_seqlens_q[2], w.cu_seqlens_q[3])]
    cu_q = np.array([0, n[0], n[0], n[0] + n[2]], np.int32)
    # sequence 1 keeps its keys in the cache (written below) but asks for no rows
    run_prefill(w, cu_q=cu_q, q=w.q[keep])


def test_prefill_single_token_matches_decode():
    """A prefill of one new token per sequence is a decode step: both GPU
    paths agree with the oracle (and hence with each other)."""
    lens = [1, 257, 600, 1300]
    w = W.make_prefill("onetoken", 812, lens, [L - 1 for L in lens], 16, 8, num_blocks=12)
    _, got_p, ref = run_prefill(w)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    out_d = pkv.paged_attn_decode(to_dev(w.q), kc, vc, i32(np.array(lens, np.int32)), i32(w.block_tables), w.scale)
    check_close(to_host(out_d), ref, "decode on prefill inputs")


def test_prefill_scale_and_permuted_blocks():
    w = W.make_prefill("scale", 813, [900, 333], [0, 100], 16, 8, num_blocks=12)
    w.scale = 0.7 / math.sqrt(128)
    run_prefill(w)


def test_prefill_repeat_is_deterministic():
    w = W.make_prefill("repeat", 814, [1000, 500], [0, 0], 16, 8, num_blocks=8)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    args = (to_dev(w.q), kc, vc, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables), w.scale,
            w.max_seqlen_q, w.max_seqlen_k)
    a = to_host(pkv.paged_attn_prefill(*args))
    b = to_host(pkv.paged_attn_prefill(*args))
    assert np.array_equal(a, b)


def test_prefill_bad_block_ids_flag_without_fault():
    """Block-table entries outside the pool (the first entry of one sequence,
    the second of another) are read as block 0 and flagged in the device error
    word; a sequence whose table is intact still matches the oracle."""
    w = W.make_prefill("badblock", 815, [600, 300, 200], [0, 0, 0], 16, 8, num_blocks=8)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    tab = w.block_tables.copy()
    tab[0, 0] = 1_000_000
    tab[1, 1] = -5
    pkv.device_error(clear=True)
    out = pkv.paged_attn_prefill(to_dev(w.q), kc, vc, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(tab), w.scale,
                                 int(np.diff(w.cu_seqlens_q).max()), w.max_seqlen_k)
    torch.cuda.synchronize()
    assert "BLOCK_RANGE" in pkv.device_error(clear=True)
    rows = np.arange(w.cu_seqlens_q[2], w.cu_seqlens_q[3])
    ref = oracle.paged_attn_prefill(w.q, okc, ovc, w.cu_seqlens_q, w.cu_seqlens_k, w.block_tables, w.scale, rows=rows)
    check_close(to_host(out), ref, "intact sequence next to bad tables", rows=rows)


def test_prefill_understated_max_seqlen_q_is_flagged():
    """n_i above the stated max_seqlen_q: the launch covers too few query
    tiles, which the kernel reports in the device error word (no fault)."""
    w = W.make_prefill("understated", 816, [700, 90], [0, 0], 16, 8, num_blocks=6)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    pkv.device_error(clear=True)
    pkv.paged_attn_prefill(to_dev(w.q), kc, vc, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables),
                           w.scale, 128, w.max_seqlen_k)
    torch.cuda.synchronize()
    assert "LEN_RANGE" in pkv.device_error(clear=True)


def _prefill_both_kernels(w: W.PrefillWorkload):
    """Run one workload through the persistent kernel (stated max_seqlen_q at
    most 2048) and through the one-CTA-per-tile kernel (the same call with
    max_seqlen_q overstated to 4096, a legal upper bound)."""
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    args = (to_dev(w.q), kc, vc, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables), w.scale)
    a = to_host(pkv.paged_attn_prefill(*args, w.max_seqlen_q, w.max_seqlen_k))
    b = to_host(pkv.paged_attn_prefill(*args, 4096, max(4096, w.max_seqlen_k)))
    torch.cuda.synchronize()
    assert pkv.device_error() == []
    return a, b


@pytest.mark.parametrize("case", ["chunked", "edges", "groups12_4", "groups16_1"])
def test_prefill_persistent_and_grid_kernels_bit_identical(case):
    """Both prefill kernels compute every tile with the same steps in the same
    order: their outputs agree bit for bit (and the persistent one matches the
    oracle in the tests above)."""
    if case == "chunked":
        w = W.chunked_prefill_prefix()
    elif case == "edges":
        w = W.make_prefill("both_edges", 821, [1, 127, 129, 300, 1025, 40], [0, 0, 1, 255, 896, 0], 16, 8,
                           num_blocks=16)
    elif case == "groups12_4":
        w = W.make_prefill("both_g3", 822, [700, 130, 1], [300, 0, 0], 12, 4, num_blocks=10)
    else:
        w = W.make_prefill("both_g16", 823, [900, 257], [0, 100], 16, 1, num_blocks=10)
    a, b = _prefill_both_kernels(w)
    assert np.array_equal(a, b), "persistent and grid prefill kernels differ"


def test_prefill_understated_max_seqlen_q_long_prompt_is_flagged():
    """Above 2048 stated query tokens the one-CTA-per-tile kernel runs; a
    sequence longer than the stated bound is flagged there too (no fault)."""
    w = W.make_prefill("understated_long", 817, [2600, 300], [0, 0], 16, 8, num_blocks=14)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    pkv.device_error(clear=True)
    pkv.paged_attn_prefill(to_dev(w.q), kc, vc, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables),
                           w.scale, 2100, w.max_seqlen_k)
    torch.cuda.synchronize()
    assert "LEN_RANGE" in pkv.device_error(clear=True)


def test_prefill_many_sequences_fallback_order():
    """1100 sequences, one with 33,000 cached tokens: the sorted item order
    would take more than 8192 (level x 32-sequence) steps to enumerate, so the
    persistent kernel's scheduler falls back to the "last query tile of each
    sequence first" order.  Every row matches the oracle, and the output is
    bit-identical to the one-CTA-per-tile kernel's."""
    rng = np.random.default_rng(1100)
    lens = [int(x) for x in rng.integers(1, 41, size=1099)] + [33130]
    cached = [0] * 1099 + [33000]
    nch = -(-len(lens) // 32)
    vmax = -(-max(lens) // 128)
    assert vmax * nch > 8192  # the fallback order is the one under test
    need = sum(-(-L // 256) for L in lens)
    w = W.make_prefill("fallback_order", 1100, lens, cached, 16, 8, num_blocks=need + 4)
    run_prefill(w)
    a, b = _prefill_both_kernels(w)
    assert np.array_equal(a, b)
