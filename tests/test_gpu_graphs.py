"""CUDA-graph bucketed decode: a replay of the captured write + decode step
for the smallest bucket >= batch equals direct calls on the real batch.

Pad rows (slot -1, context length 0) leave the token stream unchanged, so the
padded replay runs the same kernels on the same work split as the direct call:
outputs and caches must be bitwise identical.  One case is also checked
against the fp64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_304_gb300 as pkv
from paged_kv_cache_304_gb300.graphs import DecodeGraphRunner
import workloads as W
from tests.gpu_util import check_close, i32, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    # two layers over one seeded decode workload of 300 sequences
    w = W.make_decode("graphs", 1201, np.random.default_rng(1201).integers(1, 2000, size=300, endpoint=True),
                      16, 8, pool_factor=1.2)
    layers_host = [(w.k_cache, w.v_cache), (w.v_cache.copy(), w.k_cache.copy())]
    qs = [w.q, W.normal_bf16(w.q.shape, 1201, 50)]
    ks = [w.k_new, W.normal_bf16(w.k_new.shape, 1201, 51)]
    vs = [w.v_new, W.normal_bf16(w.v_new.shape, 1201, 52)]
    return w, layers_host, qs, ks, vs


def _dev_layers(layers_host):
    return [(to_dev(k), to_dev(v)) for k, v in layers_host]


@pytest.mark.parametrize("B", [1, 3, 17, 100, 256, 300])
def test_graph_replay_equals_direct_calls(setup, B):
    w, layers_host, qs, ks, vs = setup
    g_layers = _dev_layers(layers_host)
    d_layers = _dev_layers(layers_host)
    runner = DecodeGraphRunner(g_layers, 16, w.max_blocks_per_seq, w.scale, max_batch=512,
                               max_context_len=w.max_context_len)
    assert runner.bucket(B) >= B
    q = torch.stack([to_dev(x[:B]) for x in qs])
    k = torch.stack([to_dev(x[:B]) for x in ks])
    v = torch.stack([to_dev(x[:B]) for x in vs])
    slots, ctx, tab = i32(w.slot_mapping[:B]), i32(w.context_lens[:B]), i32(w.block_tables[:B])
    out_g = runner.run(q, k, v, slots, ctx, tab).clone()
    outs_d = []
    for li, (kc, vc) in enumerate(d_layers):
        pkv.kv_cache_write(k[li], v[li], slots, kc, vc)
        outs_d.append(pkv.paged_attn_decode(q[li], kc, vc, ctx, tab, w.scale, max_context_len=w.max_context_len))
    torch.cuda.synchronize()
    for li in range(2):
        assert torch.equal(out_g[li], outs_d[li]), f"layer {li}"
        assert torch.equal(g_layers[li][0], d_layers[li][0]) and torch.equal(g_layers[li][1], d_layers[li][1])
    b = runner.bucket(B)
    assert bool((runner.static.out[:, B:b] == 0).all()), "pad rows must be zero"
    assert pkv.device_error() == []


@pytest.mark.parametrize("B", [5, 256])
def test_fused_graph_replay_equals_direct_fused_calls(setup, B):
    """The runner capturing paged_attn_decode_fused_write (write inside the
    decode kernel) replays to the direct fused calls, bit for bit."""
    w, layers_host, qs, ks, vs = setup
    g_layers = _dev_layers(layers_host)
    d_layers = _dev_layers(layers_host)
    runner = DecodeGraphRunner(g_layers, 16, w.max_blocks_per_seq, w.scale, max_batch=512,
                               max_context_len=w.max_context_len, fused=True)
    q = torch.stack([to_dev(x[:B]) for x in qs])
    k = torch.stack([to_dev(x[:B]) for x in ks])
    v = torch.stack([to_dev(x[:B]) for x in vs])
    slots, ctx, tab = i32(w.slot_mapping[:B]), i32(w.context_lens[:B]), i32(w.block_tables[:B])
    out_g = runner.run(q, k, v, slots, ctx, tab).clone()
    outs_d = [pkv.paged_attn_decode_fused_write(q[li], k[li], v[li], slots, kc, vc, ctx, tab, w.scale,
                                                max_context_len=w.max_context_len)
              for li, (kc, vc) in enumerate(d_layers)]
    torch.cuda.synchronize()
    for li in range(2):
        assert torch.equal(out_g[li], outs_d[li]), f"layer {li}"
        assert torch.equal(g_layers[li][0], d_layers[li][0]) and torch.equal(g_layers[li][1], d_layers[li][1])
    assert bool((runner.static.out[:, B:runner.bucket(B)] == 0).all()), "pad rows must be zero"
    assert pkv.device_error() == []


def test_graph_replays_repeat_and_match_oracle(setup):
    w, layers_host, qs, ks, vs = setup
    B = 77
    layers = _dev_layers(layers_host[:1])
    runner = DecodeGraphRunner(layers, 16, w.max_blocks_per_seq, w.scale, max_batch=128,
                               max_context_len=w.max_context_len)
    args = (to_dev(qs[0][:B])[None], to_dev(ks[0][:B])[None], to_dev(vs[0][:B])[None], i32(w.slot_mapping[:B]),
            i32(w.context_lens[:B]), i32(w.block_tables[:B]))
    first = runner.run(*args).clone()
    for _ in range(3):
        again = runner.run(*args)
    torch.cuda.synchronize()
    assert torch.equal(first, again)
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new[:B], w.v_new[:B], w.slot_mapping[:B], okc, ovc)
    ref = oracle.paged_attn_decode(w.q[:B], okc, ovc, w.context_lens[:B], w.block_tables[:B], w.scale)
    check_close(to_host(first[0]), ref, "graph decode vs oracle")
