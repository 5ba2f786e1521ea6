"""Seeded synthetic inputs for the paged-KV attention path.

This module only *builds inputs*: Qwen3-shaped q/k/v tensors, per-sequence
block tables, slot mappings, context lengths and cu_seqlens, and paged K/V
caches whose unused slots hold stale sentinel data.  It holds none of the
attention arithmetic, so both the fp64 oracle (in tests) and the CUDA path
(in tests and in the benchmark) can take their inputs from here.

Sources for the shapes and rules used here (nano-vllm as described on the
page "13. 读一个最小推理引擎：nano-vllm", commit bb823b3):

* the cache is one preallocated tensor of shape
  (num_blocks, block_size, num_kv_heads, head_dim) per layer and per K/V
  ("第五站：执行准备与 KV 容量", the KV-capacity paragraph);
* block_size defaults to 256 ("第二站：一个请求的状态");
* slot = block_table[pos // block_size] * block_size + pos % block_size, and a
  prefill step only feeds tokens from num_cached_tokens onward
  ("第五站", the slot-mapping paragraph);
* a decode step needs a fresh block exactly when len % block_size == 1
  ("第四站：块管理与前缀缓存", can_append);
* prefix-cache lookups stop before the last block, so the last block is never
  a hit ("第四站", the prefix-hit paragraph);
* freed blocks keep their contents until reallocated ("第四站", free without
  clearing), which is why unreferenced slots hold stale finite data here;
* CUDA-graph padding rows carry slot -1 ("第五站", the CUDA Graph paragraph);
* the scheduler admits sequences first-come-first-served under a token budget
  of 16384 and only the first sequence of a step may be split
  ("第三站：调度器").

Random values are N(0, 1) drawn as float32 from numpy's default_rng and
rounded to bfloat16 (round to nearest, ties to even).  bf16 tensors are held
as numpy uint16 arrays of raw bit patterns.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 256
HEAD_DIM = 128

# Large finite stale value (bf16 bit patterns of +9984.0 and -9984.0).  Slots
# that no sequence may read are filled with these so that a kernel which reads
# past a context length, or reads an unreferenced block, produces a visibly
# wrong result instead of a plausible one.
SENTINEL_K = np.uint16(0x461C)
SENTINEL_V = np.uint16(0xC61C)

_CHUNK = 1 << 22


# ---------------------------------------------------------------------------
# bf16 helpers (input construction only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, stream: int) -> np.ndarray:
    """N(0,1) bf16 bits of the given shape, deterministic in (seed, stream).

    The values are generated in fixed chunks of 4 Mi elements; chunk i uses
    the generator default_rng([seed, stream, i]), so the result does not depend
    on the number of threads used to fill it.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(i: int) -> None:
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        rng = np.random.default_rng([seed, stream, i])
        out[lo:hi] = f32_to_bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))

    if nchunks <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# Workload containers
# ---------------------------------------------------------------------------

@dataclass
class DecodeWorkload:
    """One decode step of one layer: write the new token, then attend.

    context_lens[b] counts the new token (it is written first, then read).
    Pad rows (CUDA-graph padding) have slot -1, context length 0 and a block
    table row of -1.
    """
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q: np.ndarray             # uint16 [B, Hq, D]
    k_new: np.ndarray         # uint16 [B, Hkv, D]
    v_new: np.ndarray         # uint16 [B, Hkv, D]
    slot_mapping: np.ndarray  # int32 [B]
    context_lens: np.ndarray  # int32 [B]
    block_tables: np.ndarray  # int32 [B, max_blocks_per_seq], -1 padded
    k_cache: np.ndarray | None  # uint16 [num_blocks, bs, Hkv, D] (before the write)
    v_cache: np.ndarray | None
    scale: float
    real_batch: int
    shared_blocks: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    info: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0


@dataclass
class PrefillWorkload:
    """One (possibly chunked, possibly prefix-cached) varlen prefill step.

    Sequence i contributes n_i = cu_seqlens_q[i+1]-cu_seqlens_q[i] new tokens
    and has L_i = cu_seqlens_k[i+1]-cu_seqlens_k[i] tokens in total; its first
    c_i = L_i - n_i tokens (num_cached_tokens) are already in the cache.
    """
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q: np.ndarray             # uint16 [T, Hq, D], packed over sequences
    k_new: np.ndarray         # uint16 [T, Hkv, D]
    v_new: np.ndarray         # uint16 [T, Hkv, D]
    slot_mapping: np.ndarray  # int32 [T]
    cu_seqlens_q: np.ndarray  # int32 [S+1]
    cu_seqlens_k: np.ndarray  # int32 [S+1]
    block_tables: np.ndarray  # int32 [S, max_blocks_per_seq]
    k_cache: np.ndarray | None
    v_cache: np.ndarray | None
    scale: float
    shared_blocks: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    info: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens_q.shape[0] - 1)

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def seqlens_q(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)

    @property
    def seqlens_k(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_k)

    @property
    def max_seqlen_q(self) -> int:
        return int(self.seqlens_q.max()) if self.num_seqs else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seqlens_k.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


# ---------------------------------------------------------------------------
# Block tables, slots and cache contents
# ---------------------------------------------------------------------------

def blocks_needed(length: int, block_size: int = BLOCK_SIZE) -> int:
    return (int(length) + block_size - 1) // block_size


def slot_of(table_row: np.ndarray, pos: int, block_size: int = BLOCK_SIZE) -> int:
    """Physical slot of logical position `pos` (the pages' slot formula)."""
    return int(table_row[pos // block_size]) * block_size + pos % block_size


def decode_needs_new_block(length: int, block_size: int = BLOCK_SIZE) -> bool:
    """nano-vllm's can_append rule: appending made len % bs == 1."""
    return length % block_size == 1


def build_block_tables(lengths, shared_counts, num_blocks: int, rng: np.random.Generator,
                       donor_blocks: int = 0, block_size: int = BLOCK_SIZE):
    """Assign physical blocks to sequences from a seeded permutation.

    The first `donor_blocks` entries of the permutation form a shared prefix
    (a block chain left in the cache by an earlier request); sequence b takes
    its first shared_counts[b] blocks from it, so those blocks have a
    reference count above one.  Every other block of every sequence is
    private.  Returns (tables [B, max_blocks] int32 -1 padded, donor ids).
    """
    lengths = [int(x) for x in lengths]
    need = [blocks_needed(L, block_size) for L in lengths]
    private = sum(n - s for n, s in zip(need, shared_counts))
    if private + donor_blocks > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {private + donor_blocks}")
    perm = rng.permutation(num_blocks).astype(np.int32)
    donor = perm[:donor_blocks]
    free = list(perm[donor_blocks:])
    max_blocks = max([1] + need)
    tables = np.full((len(lengths), max_blocks), -1, dtype=np.int32)
    cursor = 0
    for b, (n, s) in enumerate(zip(need, shared_counts)):
        if s > n:
            raise ValueError("shared prefix longer than the sequence")
        tables[b, :s] = donor[:s]
        tables[b, s:n] = free[cursor:cursor + n - s]
        cursor += n - s
    return tables, donor


def _fill_cache(num_blocks: int, Hkv: int, D: int, referenced: np.ndarray, seed: int,
                stream: int, sentinel: np.uint16, block_size: int) -> np.ndarray:
    """Cache with N(0,1) data in the referenced blocks and sentinels elsewhere."""
    cache = np.full((num_blocks, block_size, Hkv, D), sentinel, dtype=np.uint16)
    if referenced.size:
        cache[referenced] = normal_bf16((referenced.size, block_size, Hkv, D), seed, stream)
    return cache


def _stamp_stale_all(k_cache, v_cache, tables, valid, shared, block_size):
    """Stamp stale tails; shared (donor) blocks are always fully valid."""
    for b in range(tables.shape[0]):
        row = tables[b]
        if valid[b] <= 0 and not (row >= 0).any():
            continue
        nb = int((row >= 0).sum())
        for lb in range(valid[b] // block_size, nb):
            p = int(row[lb])
            if p in shared:
                continue
            start = max(0, int(valid[b]) - lb * block_size)
            k_cache[p, start:] = SENTINEL_K
            v_cache[p, start:] = SENTINEL_V


# ---------------------------------------------------------------------------
# Generic builders
# ---------------------------------------------------------------------------

def make_decode(name: str, seed: int, lengths, num_q_heads: int, num_kv_heads: int,
                num_blocks: int | None = None, pool_factor: float = 1.1, shared_counts=None,
                donor_blocks: int = 0, pad_to: int | None = None, head_dim: int = HEAD_DIM,
                block_size: int = BLOCK_SIZE, fill_caches: bool = True) -> DecodeWorkload:
    """Decode step: each sequence of length L writes its new token at L-1."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    B = int(lengths.size)
    if shared_counts is None:
        shared_counts = np.zeros(B, dtype=np.int64)
    shared_counts = np.asarray(shared_counts, dtype=np.int64)
    need = sum(blocks_needed(L, block_size) - s for L, s in zip(lengths, shared_counts)) + donor_blocks
    if num_blocks is None:
        num_blocks = int(math.ceil(need * pool_factor))
    tables, donor = build_block_tables(lengths, shared_counts, num_blocks, rng, donor_blocks, block_size)
    Bp = B if pad_to is None else int(pad_to)
    if Bp < B:
        raise ValueError("pad_to smaller than the batch")
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    q = normal_bf16((Bp, Hq, D), seed, 1)
    k_new = normal_bf16((Bp, Hkv, D), seed, 2)
    v_new = normal_bf16((Bp, Hkv, D), seed, 3)
    slots = np.full(Bp, -1, dtype=np.int32)
    ctx = np.zeros(Bp, dtype=np.int32)
    tab = np.full((Bp, tables.shape[1]), -1, dtype=np.int32)
    tab[:B] = tables
    for b in range(B):
        L = int(lengths[b])
        ctx[b] = L
        slots[b] = slot_of(tables[b], L - 1, block_size)
    k_cache = v_cache = None
    if fill_caches:
        referenced = np.unique(tables[tables >= 0])
        k_cache = _fill_cache(num_blocks, Hkv, D, referenced, seed, 4, SENTINEL_K, block_size)
        v_cache = _fill_cache(num_blocks, Hkv, D, referenced, seed, 5, SENTINEL_V, block_size)
        # history occupies positions [0, L-1); the new token's slot and the rest
        # of its block hold stale data until the write.
        _stamp_stale_all(k_cache, v_cache, tables, lengths - 1, set(int(x) for x in donor), block_size)
    return DecodeWorkload(
        name=name, seed=seed, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        block_size=block_size, num_blocks=num_blocks, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=slots, context_lens=ctx, block_tables=tab, k_cache=k_cache, v_cache=v_cache,
        scale=1.0 / math.sqrt(D), real_batch=B, shared_blocks=donor.astype(np.int32),
        info={"lengths": lengths.tolist(), "shared_counts": shared_counts.tolist()})


def make_prefill(name: str, seed: int, lengths, cached, num_q_heads: int, num_kv_heads: int,
                 num_blocks: int, shared_counts=None, donor_blocks: int = 0,
                 head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE,
                 fill_caches: bool = True) -> PrefillWorkload:
    """Prefill step: sequence i has L_i tokens of which c_i are cached."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    cached = np.asarray(cached, dtype=np.int64)
    S = int(lengths.size)
    if shared_counts is None:
        shared_counts = np.zeros(S, dtype=np.int64)
    shared_counts = np.asarray(shared_counts, dtype=np.int64)
    if np.any(cached < 0) or np.any(cached >= np.maximum(lengths, 1)):
        raise ValueError("need 0 <= num_cached < L for every sequence")
    tables, donor = build_block_tables(lengths, shared_counts, num_blocks, rng, donor_blocks, block_size)
    n = lengths - cached
    cu_q = np.zeros(S + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(n)
    cu_k = np.zeros(S + 1, dtype=np.int32)
    cu_k[1:] = np.cumsum(lengths)
    T = int(cu_q[-1])
    Hq, Hkv, D = num_q_heads, num_kv_heads, head_dim
    q = normal_bf16((T, Hq, D), seed, 1)
    k_new = normal_bf16((T, Hkv, D), seed, 2)
    v_new = normal_bf16((T, Hkv, D), seed, 3)
    slots = np.empty(T, dtype=np.int32)
    for i in range(S):
        for j in range(int(n[i])):
            slots[cu_q[i] + j] = slot_of(tables[i], int(cached[i]) + j, block_size)
    k_cache = v_cache = None
    if fill_caches:
        referenced = np.unique(tables[tables >= 0])
        k_cache = _fill_cache(num_blocks, Hkv, D, referenced, seed, 4, SENTINEL_K, block_size)
        v_cache = _fill_cache(num_blocks, Hkv, D, referenced, seed, 5, SENTINEL_V, block_size)
        _stamp_stale_all(k_cache, v_cache, tables, cached, set(int(x) for x in donor), block_size)
    return PrefillWorkload(
        name=name, seed=seed, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
        block_size=block_size, num_blocks=num_blocks, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=slots, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, block_tables=tables,
        k_cache=k_cache, v_cache=v_cache, scale=1.0 / math.sqrt(D),
        shared_blocks=donor.astype(np.int32),
        info={"lengths": lengths.tolist(), "cached": cached.tolist(),
              "shared_counts": shared_counts.tolist()})


# ---------------------------------------------------------------------------
# The five named workloads (seed = 3040 + config number)
# ---------------------------------------------------------------------------

def tiny_decode(fill_caches: bool = True) -> DecodeWorkload:
    """4 sequences, L ~ U[1, 600], 16 q / 8 kv heads, 16 physical blocks."""
    seed = 3041
    rng = np.random.default_rng([seed, 0])
    lengths = rng.integers(1, 600, size=4, endpoint=True)
    return make_decode("tiny_decode_b4", seed, lengths, 16, 8, num_blocks=16, fill_caches=fill_caches)


def qwen3_0p6b_decode(fill_caches: bool = True, batch: int = 256) -> DecodeWorkload:
    """Qwen3-0.6B-shaped decode: B=256, L ~ U[100, 2048], 16/8 heads."""
    seed = 3042
    rng = np.random.default_rng([seed, 0])
    lengths = rng.integers(100, 2048, size=batch, endpoint=True)
    return make_decode("qwen3_0.6b_decode_b256", seed, lengths, 16, 8, pool_factor=1.1,
                       fill_caches=fill_caches)


def chunked_prefill_prefix(fill_caches: bool = True) -> PrefillWorkload:
    """Chunked varlen prefill with prefix-cache hits under a 16384-token budget.

    40 candidate prompts with L ~ U[100, 1024].  The first is a continuation
    chunk (its first c0 tokens, not block aligned, were computed by an earlier
    step).  12 of the others (30%) with L > 256 reuse h = min(U{1,3},
    ceil(L/256) - 1) leading blocks of a 3-block donor prefix, so
    num_cached = 256 h (the last block is never a hit).  Sequences are
    admitted first-come-first-served while the new-token total stays within
    16384; the first that does not fit ends the step.
    """
    seed = 3043
    rng = np.random.default_rng([seed, 0])
    budget = 16384
    L = rng.integers(100, 1024, size=40, endpoint=True)
    c = np.zeros(40, dtype=np.int64)
    h = np.zeros(40, dtype=np.int64)
    while True:
        c0 = int(rng.integers(1, L[0] - 1, endpoint=True))
        if c0 % BLOCK_SIZE:
            break
    c[0] = c0
    eligible = [i for i in range(1, 40) if L[i] > BLOCK_SIZE]
    sharers = rng.choice(eligible, size=min(12, len(eligible)), replace=False)
    for i in sharers:
        hi = min(int(rng.integers(1, 3, endpoint=True)), blocks_needed(L[i]) - 1)
        h[i] = hi
        c[i] = BLOCK_SIZE * hi
    admitted = []
    used = 0
    for i in range(40):
        need = int(L[i] - c[i])
        if used + need > budget:
            break
        admitted.append(i)
        used += need
    idx = np.asarray(admitted)
    w = make_prefill("chunked_prefill_prefix_budget16384", seed, L[idx], c[idx], 16, 8, num_blocks=1024,
                     shared_counts=h[idx], donor_blocks=3, fill_caches=fill_caches)
    # seq0's earlier chunk is in the cache: its own (private) blocks before c0
    w.info.update({"candidates": 40, "admitted": len(admitted), "budget": budget,
                   "new_tokens": used, "sharers": int((h[idx] > 0).sum())})
    return w


def graph_padded_decode(fill_caches: bool = True) -> DecodeWorkload:
    """Real batch 500 padded to 512 (slot -1, context 0), L ~ U[256, 4096],
    20% of sequences share 1-3 leading blocks of a donor prefix (clamped so
    that the block receiving the new token stays private)."""
    seed = 3044
    rng = np.random.default_rng([seed, 0])
    B = 500
    L = rng.integers(256, 4096, size=B, endpoint=True)
    shared = np.zeros(B, dtype=np.int64)
    sharers = rng.choice(B, size=B // 5, replace=False)
    for i in sharers:
        shared[i] = min(int(rng.integers(1, 3, endpoint=True)), (int(L[i]) - 1) // BLOCK_SIZE)
    return make_decode("graph_padded_decode_b500_pad512", seed, L, 16, 8, pool_factor=1.1,
                       shared_counts=shared, donor_blocks=3, pad_to=512, fill_caches=fill_caches)


def qwen3_8b_decode(fill_caches: bool = True, batch: int = 64) -> DecodeWorkload:
    """Qwen3-8B-shaped long-context decode: B=64, L ~ U[8192, 32768], 32/8
    heads, 8192-block pool."""
    seed = 3045
    rng = np.random.default_rng([seed, 0])
    L = rng.integers(8192, 32768, size=batch, endpoint=True)
    return make_decode("qwen3_8b_decode_b64", seed, L, 32, 8, num_blocks=8192, fill_caches=fill_caches)


def qwen3_8b_prefill(fill_caches: bool = True, num_seqs: int = 4, seqlen: int = 8192) -> PrefillWorkload:
    """Qwen3-8B-shaped prefill: 4 sequences x 8192 tokens, nothing cached."""
    seed = 3045
    L = np.full(num_seqs, seqlen, dtype=np.int64)
    c = np.zeros(num_seqs, dtype=np.int64)
    return make_prefill("qwen3_8b_prefill_4x8192", seed, L, c, 32, 8, num_blocks=8192,
                        fill_caches=fill_caches)


ALL = {
    "tiny_decode": tiny_decode,
    "qwen3_0.6b_decode": qwen3_0p6b_decode,
    "chunked_prefill_prefix": chunked_prefill_prefix,
    "graph_padded_decode": graph_padded_decode,
    "qwen3_8b_decode": qwen3_8b_decode,
    "qwen3_8b_prefill": qwen3_8b_prefill,
}
