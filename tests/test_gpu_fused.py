"""Decode with the KV write fused in vs the two separate calls and the oracle.

The fused call writes each sequence's new K/V row inside the decode kernel
(by the one CTA that then reads it).  It runs the same arithmetic on the same
work split as kv_cache_write + paged_attn_decode, so outputs and caches must
be bitwise identical to the separate calls.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_304_gb300 as pkv
import workloads as W
from tests.gpu_util import check_close, i32, to_dev, to_host

pytestmark = pytest.mark.gpu


def _both(w):
    kc1, vc1 = to_dev(w.k_cache), to_dev(w.v_cache)
    kc2, vc2 = to_dev(w.k_cache), to_dev(w.v_cache)
    q, kn, vn = to_dev(w.q), to_dev(w.k_new), to_dev(w.v_new)
    slots, ctx, tab = i32(w.slot_mapping), i32(w.context_lens), i32(w.block_tables)
    pkv.kv_cache_write(kn, vn, slots, kc1, vc1)
    o1 = pkv.paged_attn_decode(q, kc1, vc1, ctx, tab, w.scale, max_context_len=w.max_context_len)
    o2 = pkv.paged_attn_decode_fused_write(q, kn, vn, slots, kc2, vc2, ctx, tab, w.scale,
                                           max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    return o1, o2, (kc1, vc1), (kc2, vc2)


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0.6b_decode", "graph_padded_decode", "qwen3_8b_decode"])
def test_fused_equals_separate_and_oracle(name):
    w = W.ALL[name]()
    o1, o2, c1, c2 = _both(w)
    assert torch.equal(o1, o2)
    assert torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1])
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    assert np.array_equal(to_host(c2[0]), okc) and np.array_equal(to_host(c2[1]), ovc)
    ref = oracle.paged_attn_decode(w.q, okc, ovc, w.context_lens, w.block_tables, w.scale)
    real = np.nonzero(w.context_lens > 0)[0]
    check_close(to_host(o2), ref, name, rows=real)
    assert (to_host(o2)[w.context_lens == 0] == 0).all()
    assert pkv.device_error() == []


@pytest.mark.parametrize("hq,hkv", [(16, 8), (64, 8), (16, 1), (12, 4)])
def test_fused_edge_lengths(hq, hkv):
    lens = [1, 2, 16, 17, 255, 256, 257, 513, 1025, 3]
    w = W.make_decode("fused_edge", 1300 + hq, lens, hq, hkv, pool_factor=1.5, pad_to=len(lens) + 3)
    o1, o2, c1, c2 = _both(w)
    assert torch.equal(o1, o2) and torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1])
    assert pkv.device_error() == []


def test_fused_rejects_a_slot_that_is_not_the_new_token():
    """A slot other than position L-1's is neither written nor read as the
    new token; it is flagged in the device error word."""
    w = W.make_decode("fused_bad", 1310, [300, 40], 16, 8, num_blocks=4)
    slots = w.slot_mapping.copy()
    slots[0] = slots[0] - 5  # another (earlier) position of sequence 0
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.device_error(clear=True)
    pkv.paged_attn_decode_fused_write(to_dev(w.q), to_dev(w.k_new), to_dev(w.v_new), i32(slots), kc, vc,
                                      i32(w.context_lens), i32(w.block_tables), w.scale)
    assert pkv.device_error() == ["SLOT_RANGE"]
    got = to_host(kc).reshape(-1, 8, 128)
    base = w.k_cache.reshape(-1, 8, 128)
    assert np.array_equal(got[slots[0]], base[slots[0]])          # not written
    assert np.array_equal(got[w.slot_mapping[1]], w.k_new[1])     # the valid row was
