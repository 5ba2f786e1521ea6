"""Paged decode attention on the GPU vs the fp64 oracle.

Each case writes the new tokens with the library's KV write (checked
bit-exact), then runs decode through the C ABI and compares every output
element of every real row with the oracle: max-abs <= 2e-2, mean-abs <= 2e-3.
Pad rows (context length 0) must be exactly zero.
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


def run_decode(w: W.DecodeWorkload, workspace=None, repeat: int = 1):
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    q, ctx, tab = to_dev(w.q), i32(w.context_lens), i32(w.block_tables)
    out = None
    for _ in range(repeat):
        out = pkv.paged_attn_decode(q, kc, vc, ctx, tab, w.scale, workspace=workspace,
                                    max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    ref = oracle.paged_attn_decode(w.q, okc, ovc, w.context_lens, w.block_tables, w.scale)
    got = to_host(out)
    assert np.array_equal(to_host(kc), okc) and np.array_equal(to_host(vc), ovc), "kv write not bit-exact"
    real = np.nonzero(w.context_lens > 0)[0]
    pad = np.nonzero(w.context_lens == 0)[0]
    res = check_close(got, ref, w.name, rows=real) if real.size else (0.0, 0.0)
    assert (got[pad] == 0).all(), "pad rows must be zero"
    assert pkv.device_error() == []
    return res


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0.6b_decode", "graph_padded_decode", "qwen3_8b_decode"])
def test_decode_workloads(name):
    run_decode(W.ALL[name]())


EDGE_LENS = [1, 2, 15, 16, 17, 255, 256, 257, 511, 512, 513, 769, 1025]


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (64, 8), (16, 1), (8, 8), (12, 4), (4, 2)])
def test_decode_edge_lengths_and_groups(hq, hkv):
    lens = EDGE_LENS + [3]
    w = W.make_decode(f"edge_{hq}_{hkv}", 900 + hq + hkv, lens, hq, hkv, pool_factor=1.5,
                      pad_to=len(lens) + 2)  # two pad rows (context length 0) at the end
    run_decode(w)


def test_decode_32768_context():
    w = W.make_decode("long", 901, [32768, 1, 32767, 257], 32, 8, num_blocks=300)
    run_decode(w)


def test_decode_pad_rows_only():
    w = W.make_decode("pads", 902, [300], 16, 8, num_blocks=4, pad_to=64)
    run_decode(w)


def test_decode_new_block_rule_lengths():
    """Lengths with L % 256 == 1: the new token opens a fresh block."""
    lens = [257, 513, 769, 1, 1025, 2049]
    w = W.make_decode("newblock", 903, lens, 16, 8, pool_factor=2.0)
    assert all((s % 256 == 0) for s in w.slot_mapping)
    run_decode(w)


@pytest.mark.parametrize("order", ["reversed", "random"])
def test_decode_block_permutation_and_shared_prefix(order):
    """Physical block order does not matter, and rows whose tables share
    prefix blocks (reference count 2) read them correctly.  (The two equal
    rows may be split differently across SMs, so they agree to rounding.)"""
    lens = [700, 700, 300, 1300]
    shared = [2, 2, 0, 0]
    w = W.make_decode("perm", 904, lens, 16, 8, num_blocks=16, shared_counts=shared, donor_blocks=2)
    # make row 1 a copy of row 0 (same q, same private tail contents)
    w.q[1] = w.q[0]
    w.k_new[1] = w.k_new[0]
    w.v_new[1] = w.v_new[0]
    t0, t1 = w.block_tables[0, 2], w.block_tables[1, 2]
    w.k_cache[t1] = w.k_cache[t0]
    w.v_cache[t1] = w.v_cache[t0]
    if order == "reversed":
        perm = np.arange(w.num_blocks)[::-1].copy()
    else:
        perm = np.random.default_rng(3).permutation(w.num_blocks)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    # relabel physical blocks: block p moves to position inv[p]
    w.k_cache = w.k_cache[perm].copy()
    w.v_cache = w.v_cache[perm].copy()
    w.block_tables = np.where(w.block_tables >= 0, inv[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    w.slot_mapping = np.array([w.block_tables[b, (L - 1) // 256] * 256 + (L - 1) % 256
                               for b, L in enumerate(lens)], np.int32)
    run_decode(w)


def test_decode_workspace_reuse_and_repeat():
    """Repeated calls with one caller-provided workspace give the same result."""
    w = W.qwen3_0p6b_decode()
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, torch.device("cuda:0"))
    ws.fill_(0xAB)  # contents need not be initialised
    run_decode(w, workspace=ws, repeat=3)


def test_decode_bad_block_id_flags_without_fault():
    """A block-table entry outside the pool is clamped on read (no fault)
    and flagged in the device error word."""
    w = W.make_decode("badblock", 905, [300, 40], 16, 8, num_blocks=4)
    tab = w.block_tables.copy()
    tab[0, 1] = 1000
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.device_error(clear=True)
    pkv.paged_attn_decode(to_dev(w.q), kc, vc, i32(w.context_lens), i32(tab), w.scale)
    assert "BLOCK_RANGE" in pkv.device_error()


def test_decode_scale_is_applied():
    """A different scale changes the output as the oracle says."""
    w = W.make_decode("scale", 906, [500, 77], 16, 8, num_blocks=6)
    w.scale = 0.5 / math.sqrt(128)
    run_decode(w)


def test_decode_understated_max_context_len_is_clamped_and_flagged():
    """A context length above the stated max_context_len is read only up to
    that bound and flagged; other sequences are unaffected."""
    w = W.make_decode("understated", 906, [300, 1000], 16, 8, num_blocks=8)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    pkv.device_error(clear=True)
    out = pkv.paged_attn_decode(to_dev(w.q), kc, vc, i32(w.context_lens), i32(w.block_tables), w.scale,
                                max_context_len=512)
    torch.cuda.synchronize()
    assert "LEN_RANGE" in pkv.device_error(clear=True)
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, okc, ovc)
    ref = oracle.paged_attn_decode(w.q, okc, ovc, w.context_lens, w.block_tables, w.scale)
    check_close(to_host(out), ref, "sequence within the bound", rows=np.array([0]))
