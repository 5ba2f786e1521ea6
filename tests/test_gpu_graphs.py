"""CUDA-graph bucketed decode: a replay of the captured write + decode step
for the smallest bucket >= batch equals direct calls on the real batch; the
device-chained step (metadata on the device, then every layer's fused write +
decode, the sampler after the replay) equals the same calls made directly.

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


# ---------------------------------------------------------------- device-chained step
from paged_kv_cache_304_gb300.graphs import DecodeStepGraph  # noqa: E402
from oracle.metadata import prepare_metadata as oracle_metadata  # noqa: E402


def _csr_of(w, B):
    """The B sequences' block lists (just the blocks their lengths use) as a
    CSR pair, with num_cached = L - 1 and length L (a decode step)."""
    L = w.context_lens[:B].astype(np.int64)
    lists = [w.block_tables[i, :-(-int(L[i]) // 256)] for i in range(B)]
    offs = np.zeros(B + 1, np.int32)
    offs[1:] = np.cumsum([x.size for x in lists])
    ids = np.concatenate(lists).astype(np.int32)
    return ids, offs, (L - 1).astype(np.int32), L.astype(np.int32)


@pytest.mark.parametrize("B", [1, 17, 256, 300])
def test_chained_step_equals_separate_calls(setup, B):
    """Metadata on the device then the layers' fused write + decode, replayed
    from one graph for the bucket: bit for bit the same outputs, caches and
    metadata as calling pkv_prepare_metadata and the fused calls directly on
    the real batch, with the pad rows zero and no flag raised."""
    w, layers_host, qs, ks, vs = setup
    g_layers = _dev_layers(layers_host)
    d_layers = _dev_layers(layers_host)
    runner = DecodeStepGraph(g_layers, 16, w.max_blocks_per_seq, w.scale, w.num_blocks, max_batch=512,
                             max_context_len=w.max_context_len)
    ids, offs, cached, lens = _csr_of(w, B)
    q = torch.stack([to_dev(x[:B]) for x in qs])
    k = torch.stack([to_dev(x[:B]) for x in ks])
    v = torch.stack([to_dev(x[:B]) for x in vs])
    out_g = runner.run(q, k, v, i32(ids), i32(offs), i32(cached), i32(lens)).clone()
    meta_g = {kk: t.clone() for kk, t in runner.metadata(B).items()}
    meta_d = pkv.prepare_metadata(i32(ids), i32(offs), i32(cached), i32(lens), B, w.max_blocks_per_seq,
                                  w.num_blocks)
    outs_d = [pkv.paged_attn_decode_fused_write(q[li], k[li], v[li], meta_d["slot_mapping"], kc, vc,
                                                meta_d["context_lens"], meta_d["block_tables"], w.scale,
                                                max_context_len=w.max_context_len)
              for li, (kc, vc) in enumerate(d_layers)]
    torch.cuda.synchronize()
    for kk in ("slot_mapping", "context_lens", "block_tables"):
        assert torch.equal(meta_g[kk], meta_d[kk]), kk
    for li in range(2):
        assert torch.equal(out_g[li], outs_d[li]), f"layer {li}"
        assert torch.equal(g_layers[li][0], d_layers[li][0]) and torch.equal(g_layers[li][1], d_layers[li][1])
    b = runner.bucket(B)
    assert bool((runner.sets[0].out[:, B:b] == 0).all()), "pad rows must be zero"
    assert pkv.device_error() == []


def test_chained_step_matches_oracles(setup):
    """One chained replay against the oracles: the metadata oracle (slots,
    context lengths, packed tables) and the fp64 write + decode oracle."""
    w, layers_host, qs, ks, vs = setup
    B = 45
    layers = _dev_layers(layers_host[:1])
    runner = DecodeStepGraph(layers, 16, w.max_blocks_per_seq, w.scale, w.num_blocks, max_batch=64,
                             max_context_len=w.max_context_len, buffer_sets=2)
    ids, offs, cached, lens = _csr_of(w, B)
    n = runner.stage(to_dev(qs[0][:B])[None], to_dev(ks[0][:B])[None], to_dev(vs[0][:B])[None], i32(ids),
                     i32(offs), i32(cached), i32(lens), buffer_set=1)
    out = runner.replay(n, buffer_set=1).clone()
    meta = {kk: t.cpu().numpy() for kk, t in runner.metadata(B, 1).items()}
    torch.cuda.synchronize()
    ref_meta = oracle_metadata([ids[offs[i]:offs[i + 1]].tolist() for i in range(B)], cached, lens,
                               w.max_blocks_per_seq)
    assert meta["slot_mapping"].tolist() == ref_meta["slot_mapping"]
    assert meta["context_lens"].tolist() == ref_meta["context_lens"]
    assert np.array_equal(meta["block_tables"], np.array(ref_meta["block_tables"]))
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_cache_write(w.k_new[:B], w.v_new[:B], w.slot_mapping[:B], okc, ovc)
    ref = oracle.paged_attn_decode(w.q[:B], okc, ovc, w.context_lens[:B], w.block_tables[:B], w.scale)
    check_close(to_host(out[0]), ref, "chained decode step vs oracle")
    assert np.array_equal(to_host(layers[0][0]), okc) and np.array_equal(to_host(layers[0][1]), ovc)
    assert pkv.device_error() == []


def test_chained_step_then_sampler(setup):
    """The sampler after a chained replay draws the tokens the fp64 sampler
    oracle draws for the same logits, temperatures, seed and offset (up to
    near-ties of the oracle's own scores)."""
    w, layers_host, qs, ks, vs = setup
    B, V = 16, 5000
    layers = _dev_layers(layers_host[:1])
    runner = DecodeStepGraph(layers, 16, w.max_blocks_per_seq, w.scale, w.num_blocks, max_batch=16,
                             max_context_len=w.max_context_len)
    ids, offs, cached, lens = _csr_of(w, B)
    runner.run(to_dev(qs[0][:B])[None], to_dev(ks[0][:B])[None], to_dev(vs[0][:B])[None], i32(ids), i32(offs),
               i32(cached), i32(lens))
    rng = np.random.default_rng(77)
    logits = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    temps = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    tok = runner.sample(torch.from_numpy(logits).cuda(), torch.from_numpy(temps).cuda(), 1234, 9).cpu().numpy()
    ref, scores = oracle.default().sample(logits, temps, 1234, 9, with_scores=True)
    for b in np.nonzero(tok != ref)[0]:  # allowed only for a near-tie of the oracle's race scores
        gap = abs(scores[b, ref[b]] - scores[b, tok[b]])
        assert gap <= 1e-4 * max(1.0, abs(scores[b, ref[b]])), (b, ref[b], tok[b], gap)
    assert pkv.device_error() == []
