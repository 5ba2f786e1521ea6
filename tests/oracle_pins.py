"""Pins for the fp64 oracle: checks against facts other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError if that oracle disagrees with what the pages or mathematics
fix.  ``test_oracle.py`` runs them on the real oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with planted mistakes and requires that
some pin fails for every mutant.

Sources (page "13. 读一个最小推理引擎：nano-vllm"):
  store kernel skips slot -1 and copies whole K/V rows ("第六站：注意力层");
  slot = block_table[pos // bs] * bs + pos % bs ("第五站：执行准备与 KV 容量");
  every step computes from num_cached_tokens onward ("第二站：一个请求的状态");
  prefix blocks are shared by reference count ("第四站：块管理与前缀缓存");
  freed blocks are not cleared ("第四站", release without clearing).
"""

from __future__ import annotations

import math

import numpy as np

from workloads import f32_to_bf16_bits, bf16_bits_to_f32, normal_bf16

BS = 256


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def paged_from_logical(Ks, Vs, num_blocks, rng, bs=BS, sentinel=(0x461C, 0xC61C), perm=None):
    """Scatter per-sequence logical K/V ([L, Hkv, D] uint16) into a paged cache.

    Blocks are taken from a permutation of the pool (random unless given);
    every unused slot holds a large finite sentinel.  Returns
    (k_cache, v_cache, tables [S, max_blocks] int32).
    """
    Hkv, D = Ks[0].shape[1:]
    if perm is None:
        perm = rng.permutation(num_blocks)
    need = [max(1, -(-k.shape[0] // bs)) for k in Ks]
    tables = np.full((len(Ks), max(need)), -1, dtype=np.int32)
    kc = np.full((num_blocks * bs, Hkv, D), sentinel[0], dtype=np.uint16)
    vc = np.full((num_blocks * bs, Hkv, D), sentinel[1], dtype=np.uint16)
    cur = 0
    for i, (K, V) in enumerate(zip(Ks, Vs)):
        tables[i, :need[i]] = perm[cur:cur + need[i]]
        cur += need[i]
        L = K.shape[0]
        pos = np.arange(L)
        slots = tables[i][pos // bs].astype(np.int64) * bs + pos % bs
        kc[slots] = K
        vc[slots] = V
    return kc.reshape(num_blocks, bs, Hkv, D), vc.reshape(num_blocks, bs, Hkv, D), tables


def _rand_seqs(rng_seed, lens, Hkv, D):
    Ks = [normal_bf16((L, Hkv, D), rng_seed, 100 + i) for i, L in enumerate(lens)]
    Vs = [normal_bf16((L, Hkv, D), rng_seed, 200 + i) for i, L in enumerate(lens)]
    return Ks, Vs


# --------------------------------------------------------------------------
# KV write
# --------------------------------------------------------------------------

def pin_write_scatter(orc):
    """Write == numpy scatter of whole rows; -1 rows skipped; rest untouched."""
    rng = np.random.default_rng(11)
    nb, Hkv, D, N = 6, 2, 16, 40
    row = Hkv * D
    stride = row + 8  # token stride larger than the row
    kbuf = normal_bf16((N, stride), 11, 1)
    vbuf = normal_bf16((N, stride), 11, 2)
    slots = rng.choice(nb * BS, size=N, replace=False).astype(np.int32)
    slots[rng.choice(N, size=7, replace=False)] = -1
    kc = np.full((nb, BS, Hkv, D), 0x7777, dtype=np.uint16)
    vc = np.full((nb, BS, Hkv, D), 0x3333, dtype=np.uint16)
    orc.kv_cache_write(kbuf, vbuf, slots, kc, vc)
    ek = np.full((nb * BS, row), 0x7777, dtype=np.uint16)
    ev = np.full((nb * BS, row), 0x3333, dtype=np.uint16)
    keep = slots >= 0
    ek[slots[keep]] = kbuf[keep, :row]
    ev[slots[keep]] = vbuf[keep, :row]
    assert np.array_equal(kc.reshape(nb * BS, row), ek)
    assert np.array_equal(vc.reshape(nb * BS, row), ev)


def pin_write_all_padding(orc):
    """A batch made only of padding rows (slot -1) changes nothing."""
    kc = np.full((2, BS, 2, 16), 0x1234, dtype=np.uint16)
    vc = kc.copy()
    k = normal_bf16((5, 2, 16), 12, 1)
    orc.kv_cache_write(k, k, np.full(5, -1, np.int32), kc, vc)
    assert (kc == 0x1234).all() and (vc == 0x1234).all()


# --------------------------------------------------------------------------
# Attention: closed forms
# --------------------------------------------------------------------------

def pin_single_key(orc):
    """L = 1: softmax of one score is 1, so o = v_0 of kv head h // G exactly."""
    Hq, Hkv, D = 8, 2, 32
    rng = np.random.default_rng(13)
    Ks, Vs = _rand_seqs(13, [1, 1, 1], Hkv, D)
    kc, vc, tab = paged_from_logical(Ks, Vs, 5, rng)
    q = normal_bf16((3, Hq, D), 13, 7)
    out = orc.paged_attn_decode(q, kc, vc, np.array([1, 1, 1], np.int32), tab, 0.125)
    G = Hq // Hkv
    for b in range(3):
        for h in range(Hq):
            assert np.array_equal(out[b, h], _f64(Vs[b][0, h // G]))


def pin_zero_query(orc):
    """q = 0: every score is 0, so o = mean of the L value rows."""
    Hq, Hkv, D = 4, 4, 16
    rng = np.random.default_rng(14)
    lens = [300, 513]
    Ks, Vs = _rand_seqs(14, lens, Hkv, D)
    kc, vc, tab = paged_from_logical(Ks, Vs, 6, rng)
    q = np.zeros((2, Hq, D), np.uint16)
    out = orc.paged_attn_decode(q, kc, vc, np.array(lens, np.int32), tab, 0.3)
    for b in range(2):
        expect = _f64(Vs[b]).mean(axis=0)  # [Hkv, D]
        assert np.allclose(out[b], expect, rtol=0, atol=1e-12)


def pin_equal_keys(orc):
    """All keys equal: scores are equal whatever q is, so o = mean of V."""
    Hq, Hkv, D = 4, 2, 16
    rng = np.random.default_rng(15)
    L = 257
    Ks, Vs = _rand_seqs(15, [L], Hkv, D)
    Ks[0][:] = Ks[0][0]
    kc, vc, tab = paged_from_logical(Ks, Vs, 3, rng)
    q = normal_bf16((1, Hq, D), 15, 9)
    out = orc.paged_attn_decode(q, kc, vc, np.array([L], np.int32), tab, 0.25)
    mean = _f64(Vs[0]).mean(axis=0)
    for h in range(Hq):
        assert np.allclose(out[0, h], mean[h // (Hq // Hkv)], rtol=0, atol=1e-12)


def pin_two_keys_logistic(orc):
    """Two keys: softmax over two logits is the logistic function, so
    o = v0 + (v1 - v0) * sigma(scale * (q.k1 - q.k0))."""
    Hq, Hkv, D = 2, 1, 8
    rng = np.random.default_rng(16)
    K = np.zeros((2, Hkv, D), np.float32)
    K[1, 0, 0] = 2.0
    K[0, 0, 1] = 1.0
    V = np.zeros((2, Hkv, D), np.float32)
    V[0, 0, :] = 1.0
    V[1, 0, :] = -3.0
    q = np.zeros((1, Hq, D), np.float32)
    q[0, 0, 0] = 1.0   # head 0: q.k1 = 2, q.k0 = 0
    q[0, 1, 1] = 1.5   # head 1: q.k1 = 0, q.k0 = 1.5
    Kb, Vb, qb = f32_to_bf16_bits(K), f32_to_bf16_bits(V), f32_to_bf16_bits(q)
    kc, vc, tab = paged_from_logical([Kb], [Vb], 2, rng)
    scale = 0.5
    out = orc.paged_attn_decode(qb, kc, vc, np.array([2], np.int32), tab, scale)
    for h, delta in ((0, 2.0), (1, -1.5)):
        w1 = 1.0 / (1.0 + math.exp(-scale * delta))
        expect = 1.0 + (-3.0 - 1.0) * w1
        assert abs(out[0, h, 0] - expect) < 1e-14, (h, out[0, h, 0], expect)


def pin_dominant_key(orc):
    """One key whose score exceeds every other by >= 60 takes all the mass."""
    Hq, Hkv, D = 2, 1, 16
    rng = np.random.default_rng(17)
    L = 600
    K = np.zeros((L, Hkv, D), np.float32)
    K[:, 0, :] = rng.uniform(-0.1, 0.1, size=(L, D))
    star = 437
    K[star, 0, 0] = 64.0
    V = rng.standard_normal((L, Hkv, D)).astype(np.float32)
    q = np.zeros((1, Hq, D), np.float32)
    q[0, :, 0] = 8.0
    Kb, Vb, qb = f32_to_bf16_bits(K), f32_to_bf16_bits(V), f32_to_bf16_bits(q)
    kc, vc, tab = paged_from_logical([Kb], [Vb], 4, rng)
    out = orc.paged_attn_decode(qb, kc, vc, np.array([L], np.int32), tab, 1.0 / 8.0)
    expect = _f64(Vb[star, 0])
    for h in range(Hq):
        assert np.allclose(out[0, h], expect, rtol=1e-20, atol=1e-20)


def pin_shift_invariance(orc):
    """Softmax is invariant to a common shift of all logits: adding a
    component that raises every score by 1000 leaves the output unchanged
    (this also needs the maximum to be subtracted before exponentiating,
    since exp(1000) overflows a double)."""
    Hq, Hkv, D = 2, 1, 16
    rng = np.random.default_rng(26)
    L = 300
    K = rng.standard_normal((L, Hkv, D)).astype(np.float32)
    K[:, :, D - 1] = 0.0
    V = rng.standard_normal((L, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    q[:, :, D - 1] = 1.0
    Ks = K.copy()
    Ks[:, :, D - 1] = 1000.0
    Vb, qb = f32_to_bf16_bits(V), f32_to_bf16_bits(q)
    a = paged_from_logical([f32_to_bf16_bits(K)], [Vb], 2, None, perm=np.array([1, 0]))
    b = paged_from_logical([f32_to_bf16_bits(Ks)], [Vb], 2, None, perm=np.array([1, 0]))
    oa = orc.paged_attn_decode(qb, a[0], a[1], np.array([L], np.int32), a[2], 1.0)
    ob = orc.paged_attn_decode(qb, b[0], b[1], np.array([L], np.int32), b[2], 1.0)
    assert np.isfinite(ob).all() and np.allclose(oa, ob, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Attention: a library routine (torch SDPA in float64)
# --------------------------------------------------------------------------

def _sdpa(qh, kh, vh, scale, causal):
    import torch
    import torch.nn.functional as F
    q = torch.from_numpy(qh).permute(1, 0, 2)[None]  # [1, Hq, n, D]
    k = torch.from_numpy(kh).permute(1, 0, 2)[None]  # [1, Hkv, L, D]
    v = torch.from_numpy(vh).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


def pin_sdpa_prefill(orc):
    """Full-prompt prefill (nothing cached) equals causal SDPA in float64 on
    the contiguous sequences, with GQA head sharing as torch defines it."""
    Hq, Hkv, D = 8, 2, 32
    rng = np.random.default_rng(18)
    lens = [1, 255, 256, 257, 600]
    Ks, Vs = _rand_seqs(18, lens, Hkv, D)
    kc, vc, tab = paged_from_logical(Ks, Vs, 12, rng)
    T = sum(lens)
    q = normal_bf16((T, Hq, D), 18, 5)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    out = orc.paged_attn_prefill(q, kc, vc, cu, cu, tab, scale)
    for i, L in enumerate(lens):
        ref = _sdpa(_f64(q[cu[i]:cu[i + 1]]), _f64(Ks[i]), _f64(Vs[i]), scale, True)
        assert np.allclose(out[cu[i]:cu[i + 1]], ref, rtol=0, atol=1e-12), i


def pin_sdpa_decode(orc):
    """Decode equals SDPA in float64 of the single query over all L keys."""
    Hq, Hkv, D = 16, 8, 128
    rng = np.random.default_rng(19)
    lens = [1, 255, 256, 257, 511, 512, 513]
    Ks, Vs = _rand_seqs(19, lens, Hkv, D)
    kc, vc, tab = paged_from_logical(Ks, Vs, 20, rng)
    q = normal_bf16((len(lens), Hq, D), 19, 5)
    scale = 1.0 / math.sqrt(D)
    out = orc.paged_attn_decode(q, kc, vc, np.array(lens, np.int32), tab, scale)
    for b in range(len(lens)):
        ref = _sdpa(_f64(q[b:b + 1]), _f64(Ks[b]), _f64(Vs[b]), scale, False)
        assert np.allclose(out[b], ref[0], rtol=0, atol=1e-12), b


# --------------------------------------------------------------------------
# Attention: invariants the pages fix
# --------------------------------------------------------------------------

def pin_block_permutation(orc):
    """Where the blocks sit physically does not matter: two different
    permutations of the pool give bitwise identical results."""
    Hq, Hkv, D = 4, 2, 16
    lens = [700, 300, 45]
    Ks, Vs = _rand_seqs(20, lens, Hkv, D)
    q = normal_bf16((3, Hq, D), 20, 5)
    outs = []
    for perm in (np.arange(8), np.arange(8)[::-1].copy(), np.random.default_rng(20).permutation(8)):
        kc, vc, tab = paged_from_logical(Ks, Vs, 8, None, perm=perm)
        outs.append(orc.paged_attn_decode(q, kc, vc, np.array(lens, np.int32), tab, 0.25))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_chunk_consistency(orc):
    """Computing from num_cached_tokens onward gives the same rows as
    computing the whole prompt: a prefix-cached or chunked prefill of rows
    c..L-1 equals rows c..L-1 of the full prefill (bottom-right causal)."""
    Hq, Hkv, D = 4, 2, 16
    rng = np.random.default_rng(21)
    lens = [600, 300]
    cached = [257, 256]
    Ks, Vs = _rand_seqs(21, lens, Hkv, D)
    kc, vc, tab = paged_from_logical(Ks, Vs, 6, rng)
    T = sum(lens)
    q = normal_bf16((T, Hq, D), 21, 5)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    full = orc.paged_attn_prefill(q, kc, vc, cu, cu, tab, 0.25)
    n = [L - c for L, c in zip(lens, cached)]
    cuq = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    qc = np.concatenate([q[cu[i] + cached[i]:cu[i + 1]] for i in range(2)])
    part = orc.paged_attn_prefill(qc, kc, vc, cuq, cu, tab, 0.25)
    for i in range(2):
        assert np.array_equal(part[cuq[i]:cuq[i + 1]], full[cu[i] + cached[i]:cu[i + 1]]), i
    # and decode at length L is the last row of the prefill of length L
    dec = orc.paged_attn_decode(q[cu[1:] - 1], kc, vc, np.array(lens, np.int32), tab, 0.25)
    assert np.array_equal(dec, full[cu[1:] - 1])


def pin_causality(orc):
    """Changing K/V at positions > c + j leaves query row j unchanged, and
    changing position c + j itself changes it."""
    Hq, Hkv, D = 2, 1, 16
    rng = np.random.default_rng(22)
    L, c = 520, 200
    Ks, Vs = _rand_seqs(22, [L], Hkv, D)
    q = normal_bf16((L - c, Hq, D), 22, 5)
    cuq = np.array([0, L - c], np.int32)
    cuk = np.array([0, L], np.int32)
    kc, vc, tab = paged_from_logical(Ks, Vs, 3, rng, perm=np.array([2, 0, 1]))
    base = orc.paged_attn_prefill(q, kc, vc, cuq, cuk, tab, 0.3)
    j = 100
    K2, V2 = Ks[0].copy(), Vs[0].copy()
    K2[c + j + 1:] = normal_bf16(K2[c + j + 1:].shape, 22, 9)
    V2[c + j + 1:] = normal_bf16(V2[c + j + 1:].shape, 22, 10)
    kc2, vc2, _ = paged_from_logical([K2], [V2], 3, rng, perm=np.array([2, 0, 1]))
    pert = orc.paged_attn_prefill(q, kc2, vc2, cuq, cuk, tab, 0.3)
    assert np.array_equal(pert[:j + 1], base[:j + 1])
    assert not np.array_equal(pert[j + 1], base[j + 1])
    V3 = Vs[0].copy()
    V3[c + j] = normal_bf16(V3[c + j].shape, 22, 11)
    kc3, vc3, _ = paged_from_logical([Ks[0]], [V3], 3, rng, perm=np.array([2, 0, 1]))
    pert3 = orc.paged_attn_prefill(q, kc3, vc3, cuq, cuk, tab, 0.3)
    assert np.array_equal(pert3[:j], base[:j]) and not np.array_equal(pert3[j], base[j])


def pin_shared_prefix(orc):
    """Two sequences whose tables reference the same physical prefix blocks
    (reference count 2), with equal queries and equal private tails, give
    identical outputs; a third with a different tail differs."""
    Hq, Hkv, D = 4, 2, 16
    rng = np.random.default_rng(23)
    L = 600
    Ks, Vs = _rand_seqs(23, [L], Hkv, D)
    kc, vc, tab0 = paged_from_logical(Ks, Vs, 8, rng, perm=np.array([5, 1, 6, 0, 2, 3, 4, 7]))
    tail = tab0[0, 2]
    # seq 1: shares blocks 5, 1 and has its own copy of the tail in block 3
    kc[3] = kc[tail]
    vc[3] = vc[tail]
    tables = np.array([[5, 1, tail], [5, 1, 3], [5, 1, 4]], np.int32)
    kc[4] = kc[tail]
    vc[4, :] = vc[tail]
    vc[4, 10] = f32_to_bf16_bits(np.full((Hkv, D), 5.0, np.float32))
    q = np.repeat(normal_bf16((1, Hq, D), 23, 5), 3, axis=0)
    out = orc.paged_attn_decode(q, kc, vc, np.full(3, L, np.int32), tables, 0.25)
    assert np.array_equal(out[0], out[1])
    assert not np.array_equal(out[0], out[2])


def pin_stale_ignored(orc):
    """Slots past the context length (stale data from freed blocks) do not
    affect the result: sentinel values +-9984 or zeros give identical output."""
    Hq, Hkv, D = 4, 2, 16
    lens = [300, 5]
    Ks, Vs = _rand_seqs(24, lens, Hkv, D)
    q = normal_bf16((2, Hq, D), 24, 5)
    perm = np.random.default_rng(24).permutation(5)
    a = paged_from_logical(Ks, Vs, 5, None, perm=perm)
    b = paged_from_logical(Ks, Vs, 5, None, perm=perm, sentinel=(0, 0))
    oa = orc.paged_attn_decode(q, a[0], a[1], np.array(lens, np.int32), a[2], 0.25)
    ob = orc.paged_attn_decode(q, b[0], b[1], np.array(lens, np.int32), b[2], 0.25)
    assert np.array_equal(oa, ob)
    cu = np.array([0, 300, 305], np.int32)
    qp = normal_bf16((305, Hq, D), 24, 6)
    pa = orc.paged_attn_prefill(qp, a[0], a[1], cu, cu, a[2], 0.25)
    pb = orc.paged_attn_prefill(qp, b[0], b[1], cu, cu, b[2], 0.25)
    assert np.array_equal(pa, pb)


def pin_pad_rows(orc):
    """CUDA-graph pad rows (context length 0, table row of -1) give zeros."""
    Hq, Hkv, D = 4, 2, 16
    Ks, Vs = _rand_seqs(25, [40], Hkv, D)
    kc, vc, tab = paged_from_logical(Ks, Vs, 2, np.random.default_rng(25))
    tables = np.full((3, tab.shape[1]), -1, np.int32)
    tables[1] = tab[0]
    q = normal_bf16((3, Hq, D), 25, 5)
    out = orc.paged_attn_decode(q, kc, vc, np.array([0, 40, 0], np.int32), tables, 0.25)
    assert (out[0] == 0).all() and (out[2] == 0).all() and np.abs(out[1]).sum() > 0


# --------------------------------------------------------------------------
# Exponential-race sampler
# --------------------------------------------------------------------------

def pin_philox_known_answer(orc):
    """Philox4x32-10 of the zero counter under the zero key: the published
    known answer of the generator."""
    assert orc.philox4x32_10([0, 0, 0, 0], [0, 0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]


def pin_race_distribution(orc):
    """The race winner is distributed as softmax(logits / T) (chi-square,
    60000 independent rows, p-value > 1e-4)."""
    from scipy.stats import chisquare
    V, B, T = 8, 60000, 0.7
    base = np.array([1.0, 0.5, -0.3, 2.0, 0.0, -1.0, 1.5, 0.2], np.float32)
    tok = orc.sample(np.tile(base, (B, 1)), np.full(B, T, np.float32), seed=99, offset=0)
    z = base.astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    counts = np.bincount(tok, minlength=V)
    assert chisquare(counts, p * counts.sum()).pvalue > 1e-4


def pin_low_temperature_is_argmax(orc):
    """As T -> 0 the race always picks the largest logit."""
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((40, 500)).astype(np.float32)
    tok = orc.sample(logits, np.full(40, 1e-3, np.float32), seed=5, offset=3)
    assert (tok == logits.argmax(axis=1)).all()


ALL_PINS = [
    pin_write_scatter, pin_write_all_padding, pin_single_key, pin_zero_query, pin_equal_keys,
    pin_two_keys_logistic, pin_dominant_key, pin_shift_invariance, pin_sdpa_prefill, pin_sdpa_decode, pin_block_permutation,
    pin_chunk_consistency, pin_causality, pin_shared_prefix, pin_stale_ignored, pin_pad_rows,
    pin_philox_known_answer, pin_race_distribution, pin_low_temperature_is_argmax,
]
