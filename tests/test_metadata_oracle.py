"""Pins for the step-metadata oracle (oracle/metadata.py), CPU only."""

import numpy as np
import pytest

import workloads as W
from oracle.metadata import prepare_metadata


def test_hand_worked_example():
    """Table [7, 2], block size 256, 250 tokens cached, 300 in total: the
    new positions 250..255 sit in physical block 7 (slots 2042..2047) and
    256..299 in block 2 (slots 512..555)."""
    m = prepare_metadata([[7, 2]], [250], [300], max_blocks=4)
    assert m["slot_mapping"] == list(range(2042, 2048)) + list(range(512, 556))
    assert m["cu_seqlens_q"] == [0, 50] and m["cu_seqlens_k"] == [0, 300]
    assert m["context_lens"] == [300]
    assert m["block_tables"] == [[7, 2, -1, -1]]


def test_decode_block_rule_and_invariants():
    rng = np.random.default_rng(5)
    S = 200
    L = rng.integers(1, 2000, size=S)
    perm = rng.permutation(2000)
    tables, cur = [], 0
    for x in L:
        nb = -(-int(x) // 256)
        tables.append(list(perm[cur:cur + nb]))
        cur += nb
    m = prepare_metadata(tables, L - 1, L, max_blocks=8)
    slots = np.array(m["slot_mapping"])
    assert slots.size == S and len(set(slots.tolist())) == S
    for i in range(S):
        # the new token opens a fresh block exactly when L % 256 == 1
        assert (L[i] % 256 == 1) == (slots[i] % 256 == 0)
        assert slots[i] // 256 == tables[i][(L[i] - 1) // 256]
    assert m["cu_seqlens_q"] == list(range(S + 1))
    assert m["cu_seqlens_k"][-1] == int(L.sum())


@pytest.mark.parametrize("name", ["chunked_prefill_prefix", "qwen3_8b_prefill"])
def test_prefill_workloads_agree_with_generator(name):
    w = W.ALL[name](fill_caches=False)
    L = w.seqlens_k
    c = L - w.seqlens_q
    tables = [list(w.block_tables[i, :-(-int(L[i]) // 256)]) for i in range(w.num_seqs)]
    m = prepare_metadata(tables, c, L, max_blocks=w.max_blocks_per_seq)
    assert m["slot_mapping"] == w.slot_mapping.tolist()
    assert m["cu_seqlens_q"] == w.cu_seqlens_q.tolist() and m["cu_seqlens_k"] == w.cu_seqlens_k.tolist()


def test_rejects_short_table():
    with pytest.raises(ValueError):
        prepare_metadata([[3]], [255], [257], max_blocks=2)  # position 256 needs a second block


def test_graph_pad_rows_reproduce_the_padded_decode_workload():
    """The CUDA-graph padded decode step (500 real rows padded to 512 with
    slot -1 and context length 0, built by the input generator): pad rows
    given as empty sequences (num_cached = length = 0, no table) add no
    tokens, get context length 0 and a -1 table row, so the real rows' slots
    followed by -1 up to the padded batch are exactly the generator's slot
    mapping."""
    w = W.graph_padded_decode(fill_caches=False)
    L = w.context_lens.astype(np.int64)
    real = w.real_batch
    tables = [list(w.block_tables[i, :-(-int(L[i]) // 256)]) for i in range(real)] + [[]] * (w.batch - real)
    cached = np.concatenate([L[:real] - 1, np.zeros(w.batch - real, np.int64)])
    m = prepare_metadata(tables, cached, L, max_blocks=w.max_blocks_per_seq)
    slots = m["slot_mapping"] + [-1] * (w.batch - len(m["slot_mapping"]))
    assert slots == w.slot_mapping.tolist()
    assert m["context_lens"] == w.context_lens.tolist()
    assert np.array_equal(np.array(m["block_tables"]), w.block_tables)
    assert m["cu_seqlens_q"][real:] == [real] * (w.batch - real + 1)


def test_rejects_empty_sequence_with_cached_tokens():
    with pytest.raises(ValueError):
        prepare_metadata([[3]], [5], [5], max_blocks=2)  # no new token but not a pad row
