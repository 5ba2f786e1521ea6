"""Prefill with the KV write fused in vs the two separate calls and the oracle.

pkv_paged_attn_prefill_fused_write writes every new token's K/V row into the
cache (each SM a share), waits at a grid-wide barrier, then runs the
persistent prefill kernel; above a stated max_seqlen_q of 2048 it launches
the write kernel and then the long-prompt kernel.  The writes are the
standalone write's bytes and the attention is the same per-tile arithmetic
as either prefill kernel, so outputs and caches must be bitwise identical to
kv_cache_write followed by paged_attn_prefill, and within tolerance of the
fp64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_304_gb300 as pkv
import workloads as W
from tests.gpu_util import check_close, i32, to_dev, to_host
from tests.test_gpu_prefill import config5_rows

pytestmark = pytest.mark.gpu


def _both(w, slots=None, workspace=None):
    slots = w.slot_mapping if slots is None else slots
    kc1, vc1 = to_dev(w.k_cache), to_dev(w.v_cache)
    kc2, vc2 = to_dev(w.k_cache), to_dev(w.v_cache)
    q, kn, vn = to_dev(w.q), to_dev(w.k_new), to_dev(w.v_new)
    cq, ck, tab = i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables)
    sl = i32(slots)
    pkv.kv_cache_write(kn, vn, sl, kc1, vc1)
    o1 = pkv.paged_attn_prefill(q, kc1, vc1, cq, ck, tab, w.scale, w.max_seqlen_q, w.max_seqlen_k)
    o2 = pkv.paged_attn_prefill_fused_write(q, kn, vn, sl, kc2, vc2, cq, ck, tab, w.scale, w.max_seqlen_q,
                                            w.max_seqlen_k, workspace=workspace)
    torch.cuda.synchronize()
    return o1, o2, (kc1, vc1), (kc2, vc2)


@pytest.mark.parametrize("name", ["chunked_prefill_prefix", "qwen3_8b_prefill"])
def test_fused_prefill_equals_separate_and_oracle(name):
    """Chunked, prefix-cached 16384-token step and the 4 x 8192 prefill (where
    the separate call runs the one-CTA-per-tile kernel)."""
    w = W.ALL[name]()
    o1, o2, c1, c2 = _both(w)
    assert torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1]), "caches differ"
    assert torch.equal(o1, o2), "outputs differ"
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    assert np.array_equal(to_host(c2[0]), okc) and np.array_equal(to_host(c2[1]), ovc), "write not bit-exact"
    rows = config5_rows(w) if name == "qwen3_8b_prefill" else None
    ref = oracle.paged_attn_prefill(w.q, okc, ovc, w.cu_seqlens_q, w.cu_seqlens_k, w.block_tables, w.scale,
                                    rows=rows)
    check_close(to_host(o2), ref, f"fused prefill {name}", rows=rows)
    assert pkv.device_error() == []


@pytest.mark.parametrize("hq,hkv", [(12, 4), (8, 8), (16, 1)])
def test_fused_prefill_group_sizes(hq, hkv):
    """Groups of 3 (a head pair plus a lone head: items without slot B), 1
    and 16, with a continuation chunk, prefix hits and a 1-token sequence:
    bit-identical to the separate calls, caches bit-exact, close to the oracle."""
    w = W.make_prefill(f"fused_g{hq}_{hkv}", 933 + hq + hkv, [700, 300, 1000, 129, 1], [200, 0, 513, 0, 0], hq,
                       hkv, num_blocks=24)
    o1, o2, c1, c2 = _both(w)
    assert torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1]), "caches differ"
    assert torch.equal(o1, o2), "outputs differ"
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    assert np.array_equal(to_host(c2[0]), okc) and np.array_equal(to_host(c2[1]), ovc), "write not bit-exact"
    ref = oracle.paged_attn_prefill(w.q, okc, ovc, w.cu_seqlens_q, w.cu_seqlens_k, w.block_tables, w.scale)
    check_close(to_host(o2), ref, f"fused prefill hq={hq} hkv={hkv}")
    assert pkv.device_error() == []


def test_fused_prefill_reuses_its_workspace_and_skips_pad_slots():
    """One workspace across several calls (the barrier leaves it ready), a
    tiny batch (fewer work items than SMs), and slot -1 rows left unwritten."""
    ws = pkv.prefill_fused_workspace(torch.device("cuda:0"))
    w = W.make_prefill("fused_small", 931, [300, 1, 129], [0, 0, 100], 16, 8, num_blocks=8)
    for _ in range(3):
        o1, o2, c1, c2 = _both(w, workspace=ws)
        assert torch.equal(o1, o2) and torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1])
    slots = w.slot_mapping.copy()
    slots[5] = -1
    o1, o2, c1, c2 = _both(w, slots=slots, workspace=ws)
    assert torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1])
    assert torch.equal(o1, o2)
    assert pkv.device_error() == []


def test_fused_prefill_out_of_range_slot_is_flagged():
    w = W.make_prefill("fused_badslot", 932, [200, 300], [0, 0], 16, 8, num_blocks=6)
    slots = w.slot_mapping.copy()
    slots[7] = 6 * 256 + 3  # beyond the pool
    pkv.device_error(clear=True)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.paged_attn_prefill_fused_write(to_dev(w.q), to_dev(w.k_new), to_dev(w.v_new), i32(slots), kc, vc,
                                       i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables), w.scale,
                                       w.max_seqlen_q, w.max_seqlen_k)
    torch.cuda.synchronize()
    assert "SLOT_RANGE" in pkv.device_error(clear=True)


def test_fused_prefill_long_prompt_path_flags_bad_slot_and_leaves_workspace():
    """Above a stated max_seqlen_q of 2048 (two launches): bit-identical to the
    separate calls, an out-of-range slot is flagged by the write, and the
    workspace is not touched."""
    w = W.make_prefill("fused_long", 934, [3000, 700], [0, 100], 16, 8, num_blocks=20)
    ws = pkv.prefill_fused_workspace(torch.device("cuda:0"))
    ws.fill_(7)
    o1, o2, c1, c2 = _both(w, workspace=ws)
    assert torch.equal(c1[0], c2[0]) and torch.equal(c1[1], c2[1]) and torch.equal(o1, o2)
    assert bool((ws == 7).all())
    assert pkv.device_error() == []
    slots = w.slot_mapping.copy()
    slots[11] = 20 * 256 + 5  # beyond the pool
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.paged_attn_prefill_fused_write(to_dev(w.q), to_dev(w.k_new), to_dev(w.v_new), i32(slots), kc, vc,
                                       i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.block_tables), w.scale,
                                       w.max_seqlen_q, w.max_seqlen_k, workspace=ws)
    torch.cuda.synchronize()
    assert "SLOT_RANGE" in pkv.device_error(clear=True)
