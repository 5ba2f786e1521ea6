"""Device-side step metadata vs the oracle: bit-exact integers."""

import numpy as np
import pytest
import torch

import paged_kv_cache_304_gb300 as pkv
import workloads as W
from oracle.metadata import prepare_metadata
from tests.gpu_util import i32

pytestmark = pytest.mark.gpu


def _csr(tables):
    offs = np.zeros(len(tables) + 1, np.int32)
    offs[1:] = np.cumsum([len(t) for t in tables])
    ids = np.concatenate([np.asarray(t, np.int32) for t in tables]) if tables else np.zeros(0, np.int32)
    return ids, offs


def _run(tables, cached, lens, max_blocks, num_blocks, capacity=None):
    ids, offs = _csr(tables)
    total = int(np.sum(np.asarray(lens) - np.asarray(cached)))
    cap = total if capacity is None else capacity
    got = pkv.prepare_metadata(i32(ids), i32(offs), i32(cached), i32(lens), cap, max_blocks, num_blocks)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in got.items()}, total


def _check(tables, cached, lens, max_blocks, num_blocks, capacity=None):
    got, total = _run(tables, cached, lens, max_blocks, num_blocks, capacity)
    ref = prepare_metadata(tables, cached, lens, max_blocks)
    for k in ("cu_seqlens_q", "cu_seqlens_k", "context_lens", "block_tables"):
        assert np.array_equal(got[k], np.asarray(ref[k], np.int32)), k
    assert np.array_equal(got["slot_mapping"][:total], np.asarray(ref["slot_mapping"], np.int32))
    assert (got["slot_mapping"][total:] == -1).all()
    assert pkv.device_error() == []


def _tables_of(w, lens):
    return [list(w.block_tables[i, :-(-int(lens[i]) // 256)]) for i in range(len(lens))]


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0.6b_decode", "graph_padded_decode", "qwen3_8b_decode"])
def test_decode_metadata(name):
    w = W.ALL[name](fill_caches=False)
    L = w.context_lens[: w.real_batch]
    _check(_tables_of(w, L), L - 1, L, w.max_blocks_per_seq, w.num_blocks)


@pytest.mark.parametrize("name", ["chunked_prefill_prefix", "qwen3_8b_prefill"])
def test_prefill_metadata(name):
    w = W.ALL[name](fill_caches=False)
    L = w.seqlens_k
    _check(_tables_of(w, L), L - w.seqlens_q, L, w.max_blocks_per_seq, w.num_blocks)


def test_graph_padding_and_many_sequences():
    """Capacity beyond the real tokens is filled with -1 (the graph padding
    slot); 3000 sequences exercise the multi-chunk scan."""
    rng = np.random.default_rng(9)
    S = 3000
    L = rng.integers(1, 700, size=S)
    perm = rng.permutation(20000)
    tables, cur = [], 0
    for x in L:
        nb = -(-int(x) // 256)
        tables.append(list(perm[cur:cur + nb]))
        cur += nb
    _check(tables, L - 1, L, 3, 20000, capacity=S + 37)


def test_more_sequences_than_one_kernel_scans():
    """Above 16384 sequences the scan and the fill run as two kernels."""
    rng = np.random.default_rng(10)
    S = 17000
    L = rng.integers(1, 40, size=S)
    perm = rng.permutation(S + 10)
    tables = [[int(perm[i])] for i in range(S)]
    _check(tables, L - 1, L, 1, S + 10, capacity=S + 5)


def test_short_table_is_flagged_and_skipped():
    pkv.device_error(clear=True)
    got, _ = _run([[3], [5, 6]], [255, 0], [257, 300], 2, 8, capacity=300)
    assert "LEN_RANGE" in pkv.device_error()
    assert got["cu_seqlens_q"].tolist() == [0, 0, 300]  # sequence 0 contributes nothing


def test_graph_pad_rows_unflagged():
    """Pad rows (num_cached = length = 0, empty table) after the real rows of
    the padded decode workload: no flag, context length 0, -1 tables, and the
    real rows' slots followed by -1."""
    w = W.graph_padded_decode(fill_caches=False)
    L = w.context_lens.astype(np.int64)
    real = w.real_batch
    tables = _tables_of(w, L[:real]) + [[]] * (w.batch - real)
    cached = np.concatenate([L[:real] - 1, np.zeros(w.batch - real, np.int64)])
    pkv.device_error(clear=True)
    got, total = _run(tables, cached, L, w.max_blocks_per_seq, w.num_blocks, capacity=w.batch)
    assert total == real
    assert pkv.device_error() == []
    assert np.array_equal(got["slot_mapping"], w.slot_mapping)
    assert np.array_equal(got["context_lens"], w.context_lens)
    assert np.array_equal(got["block_tables"], w.block_tables)
