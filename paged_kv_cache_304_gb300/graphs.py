"""CUDA-graph bucketed decode: capture the decode step once per batch bucket
and replay it.

nano-vllm captures its decode step as CUDA graphs for batch sizes 1, 2, 4, 8
and then 16 to 512 in steps of 16, largest first, all sharing one memory pool;
at run time it picks the smallest graph not smaller than the real batch,
copies the real inputs into the graph's static buffers, fills the slots of
the extra rows with -1 and replays (page "13. 读一个最小推理引擎：nano-vllm",
section "第五站：执行准备与 KV 容量", CUDA Graph paragraph).

DecodeGraphRunner does the same for the paged-KV attention path of any number
of layers: each captured graph holds, per layer, kv_cache_write followed by
paged_attn_decode (three library kernels), all reading static input buffers
and sharing one decode workspace sized for the largest bucket.  Pad rows get
slot -1 (the write skips them) and context length 0 (decode writes zeros and
reads nothing for them), so a padded replay gives exactly the rows a direct
call on the real batch gives.

DecodeStepGraph goes one step further: its graphs also derive the step
metadata on the device from what each sequence holds (block list, cached
tokens, length), so the host sends only those, and the sampler runs after the
replay.

This module is host plumbing around the C-ABI calls: it allocates the static
buffers with torch and captures/replays graphs; every step of the path runs in
the library's kernels.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (decode_workspace, kv_cache_write, paged_attn_decode, paged_attn_decode_fused_write,
               prepare_metadata, sample_exponential_race)


def graph_batch_sizes(max_batch: int = 512) -> list[int]:
    """Bucket sizes nano-vllm captures: 1, 2, 4, 8, then 16..max in steps of 16."""
    sizes = [b for b in (1, 2, 4, 8) if b <= max_batch]
    sizes += list(range(16, max_batch + 1, 16))
    if not sizes or sizes[-1] < max_batch:
        sizes.append(max_batch)
    return sizes


@dataclass
class _Static:
    q: torch.Tensor        # [layers, max_batch, Hq, D]
    k_new: torch.Tensor    # [layers, max_batch, Hkv, D]
    v_new: torch.Tensor
    out: torch.Tensor      # [layers, max_batch, Hq, D]
    slots: torch.Tensor    # [max_batch] int32
    ctx: torch.Tensor      # [max_batch] int32
    tables: torch.Tensor   # [max_batch, max_blocks] int32


class DecodeGraphRunner:
    """Replays a captured write + decode step for the smallest bucket >= batch.

    layers: list of (k_cache, v_cache) pairs, one per decoder layer.
    max_blocks_per_seq: width of the block-table rows.
    max_context_len: host-known bound of the context lengths (captured into
    the graphs, so it must hold for every replay).
    fused: capture paged_attn_decode_fused_write (write inside the decode
    kernel) instead of kv_cache_write followed by paged_attn_decode.
    """

    def __init__(self, layers, num_q_heads: int, max_blocks_per_seq: int, scale: float,
                 max_batch: int = 512, max_context_len: int | None = None, buckets=None, fused: bool = False):
        if not layers:
            raise ValueError("need at least one layer")
        k0 = layers[0][0]
        self.device = k0.device
        self.layers = list(layers)
        nb, bs, hkv, d = (int(x) for x in k0.shape)
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, hkv, d
        self.max_batch = max_batch
        self.max_blocks = max_blocks_per_seq
        self.scale = float(scale)
        self.fused = fused
        self.max_context_len = max_context_len if max_context_len is not None else max_blocks_per_seq * bs
        self.buckets = sorted(buckets or graph_batch_sizes(max_batch))
        nl = len(layers)
        dev, bf = self.device, torch.bfloat16
        self.static = _Static(
            q=torch.zeros((nl, max_batch, num_q_heads, d), dtype=bf, device=dev),
            k_new=torch.zeros((nl, max_batch, hkv, d), dtype=bf, device=dev),
            v_new=torch.zeros((nl, max_batch, hkv, d), dtype=bf, device=dev),
            out=torch.zeros((nl, max_batch, num_q_heads, d), dtype=bf, device=dev),
            slots=torch.full((max_batch,), -1, dtype=torch.int32, device=dev),
            ctx=torch.zeros((max_batch,), dtype=torch.int32, device=dev),
            tables=torch.full((max_batch, max_blocks_per_seq), -1, dtype=torch.int32, device=dev),
        )
        self.workspace = decode_workspace(max_batch, num_q_heads, dev)
        self.graphs: dict[int, torch.cuda.CUDAGraph] = {}
        self._capture()

    def _step(self, b: int) -> None:
        st = self.static
        for li, (kc, vc) in enumerate(self.layers):
            if self.fused:
                paged_attn_decode_fused_write(st.q[li, :b], st.k_new[li, :b], st.v_new[li, :b], st.slots[:b], kc, vc,
                                              st.ctx[:b], st.tables[:b], self.scale, out=st.out[li, :b],
                                              workspace=self.workspace, max_context_len=self.max_context_len)
                continue
            kv_cache_write(st.k_new[li, :b], st.v_new[li, :b], st.slots[:b], kc, vc)
            paged_attn_decode(st.q[li, :b], kc, vc, st.ctx[:b], st.tables[:b], self.scale, out=st.out[li, :b],
                              workspace=self.workspace, max_context_len=self.max_context_len)

    def _capture(self) -> None:
        # Static inputs are all pad rows during capture, so the captured
        # launches read and write nothing; the largest bucket is captured first
        # (nano-vllm's order) and all graphs share one pool.
        torch.cuda.synchronize(self.device)
        pool = None
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self._step(self.buckets[-1])  # warm-up outside capture
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        for b in reversed(self.buckets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, pool=pool, capture_error_mode="relaxed"):
                self._step(b)
            if pool is None:
                pool = g.pool()
            self.graphs[b] = g
        torch.cuda.synchronize(self.device)

    def bucket(self, batch: int) -> int:
        for b in self.buckets:
            if b >= batch:
                return b
        raise ValueError(f"batch {batch} exceeds the largest captured bucket {self.buckets[-1]}")

    def run(self, q, k_new, v_new, slot_mapping, context_lens, block_tables) -> torch.Tensor:
        """One decode step of every layer for a real batch of B sequences.

        q: [layers, B, Hq, D]; k_new, v_new: [layers, B, Hkv, D]; slot_mapping,
        context_lens: [B] int32; block_tables: [B, <= max_blocks] int32.
        Returns out[:, :B] (a view of the static output buffer, valid until the
        next run).
        """
        B = int(context_lens.shape[0])
        b = self.bucket(B)
        st = self.static
        st.q[:, :B].copy_(q)
        st.k_new[:, :B].copy_(k_new)
        st.v_new[:, :B].copy_(v_new)
        st.slots[:B].copy_(slot_mapping)
        st.ctx[:B].copy_(context_lens)
        st.tables[:B, :block_tables.shape[1]].copy_(block_tables)
        if b > B:
            st.slots[B:b].fill_(-1)
            st.ctx[B:b].fill_(0)
        self.graphs[b].replay()
        return st.out[:, :B]


@dataclass
class _StepBuffers:
    q: torch.Tensor              # [layers, max_batch, Hq, D]
    k_new: torch.Tensor          # [layers, max_batch, Hkv, D]
    v_new: torch.Tensor
    out: torch.Tensor            # [layers, max_batch, Hq, D]
    block_ids: torch.Tensor      # [max_batch * max_blocks] int32, the CSR block lists
    table_offsets: torch.Tensor  # [max_batch + 1] int32
    num_cached: torch.Tensor     # [max_batch] int32
    seq_lens: torch.Tensor       # [max_batch] int32
    meta: dict                   # prepare_metadata outputs sized for max_batch


class DecodeStepGraph:
    """The decode step chained on the device and replayed from one CUDA graph
    per batch bucket: step metadata, then every layer's KV write + decode.

    nano-vllm's prepare_decode turns each running sequence's block table and
    length into the slot of the new token, the context length and the padded
    block-table tensor on the host, copies them into the graph's buffers
    (pad rows: slot -1, context length 0) and replays the captured step (page
    "13. 读一个最小推理引擎：nano-vllm", section "第五站：执行准备与 KV 容量",
    slot-mapping and CUDA Graph paragraphs).  Here the host hands over only
    what each sequence holds -- its block list (a CSR pair), num_cached and
    length -- and the captured graph derives the rest on the device
    (pkv_prepare_metadata) before the layers' fused write + decode calls read
    it.  Pad rows are empty sequences (num_cached = length = 0, no blocks),
    which the metadata turns into slot -1 and context length 0.

    Sampling is not captured: as in nano-vllm, the sampler runs after the
    replay (sample() below), so each step can draw new random numbers.

    `buffer_sets` > 1 captures the graphs once per set of static buffers, so
    a caller can stage step s+1's inputs (stage() on a copy stream) while
    step s replays from the other set.
    """

    def __init__(self, layers, num_q_heads: int, max_blocks_per_seq: int, scale: float, num_blocks: int,
                 max_batch: int = 512, max_context_len: int | None = None, buckets=None, buffer_sets: int = 1):
        if not layers:
            raise ValueError("need at least one layer")
        k0 = layers[0][0]
        self.device = k0.device
        self.layers = list(layers)
        nb, bs, hkv, d = (int(x) for x in k0.shape)
        self.num_q_heads, self.num_kv_heads, self.head_dim, self.block_size = num_q_heads, hkv, d, bs
        self.num_blocks = int(num_blocks)
        self.max_batch = max_batch
        self.max_blocks = max_blocks_per_seq
        self.scale = float(scale)
        self.max_context_len = max_context_len if max_context_len is not None else max_blocks_per_seq * bs
        self.buckets = sorted(buckets or graph_batch_sizes(max_batch))
        nl = len(layers)
        dev, bf, i32 = self.device, torch.bfloat16, torch.int32

        def buffers():
            return _StepBuffers(
                q=torch.zeros((nl, max_batch, num_q_heads, d), dtype=bf, device=dev),
                k_new=torch.zeros((nl, max_batch, hkv, d), dtype=bf, device=dev),
                v_new=torch.zeros((nl, max_batch, hkv, d), dtype=bf, device=dev),
                out=torch.zeros((nl, max_batch, num_q_heads, d), dtype=bf, device=dev),
                block_ids=torch.zeros(max(1, max_batch * max_blocks_per_seq), dtype=i32, device=dev),
                table_offsets=torch.zeros(max_batch + 1, dtype=i32, device=dev),
                num_cached=torch.zeros(max_batch, dtype=i32, device=dev),
                seq_lens=torch.zeros(max_batch, dtype=i32, device=dev),
                meta={"cu_seqlens_q": torch.zeros(max_batch + 1, dtype=i32, device=dev),
                      "cu_seqlens_k": torch.zeros(max_batch + 1, dtype=i32, device=dev),
                      "context_lens": torch.zeros(max_batch, dtype=i32, device=dev),
                      "slot_mapping": torch.full((max_batch,), -1, dtype=i32, device=dev),
                      "block_tables": torch.full((max_batch, max_blocks_per_seq), -1, dtype=i32, device=dev)},
            )

        self.sets = [buffers() for _ in range(max(1, buffer_sets))]
        self.workspace = decode_workspace(max_batch, num_q_heads, dev)
        self.graphs: list[dict[int, torch.cuda.CUDAGraph]] = [{} for _ in self.sets]
        self._capture()

    def _step(self, st: _StepBuffers, b: int) -> None:
        m = st.meta
        view = {"cu_seqlens_q": m["cu_seqlens_q"][:b + 1], "cu_seqlens_k": m["cu_seqlens_k"][:b + 1],
                "context_lens": m["context_lens"][:b], "slot_mapping": m["slot_mapping"][:b],
                "block_tables": m["block_tables"][:b]}
        prepare_metadata(st.block_ids, st.table_offsets[:b + 1], st.num_cached[:b], st.seq_lens[:b], b,
                         self.max_blocks, self.num_blocks, self.block_size, out=view)
        for li, (kc, vc) in enumerate(self.layers):
            paged_attn_decode_fused_write(st.q[li, :b], st.k_new[li, :b], st.v_new[li, :b], view["slot_mapping"],
                                          kc, vc, view["context_lens"], view["block_tables"], self.scale,
                                          out=st.out[li, :b], workspace=self.workspace,
                                          max_context_len=self.max_context_len)

    def _capture(self) -> None:
        # The static inputs are all pad rows during capture (empty sequences),
        # so the captured launches write and read nothing; the largest bucket
        # is captured first and all graphs share one pool.
        torch.cuda.synchronize(self.device)
        pool = None
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self._step(self.sets[0], self.buckets[-1])  # warm-up outside capture
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        for si, st in enumerate(self.sets):
            for b in reversed(self.buckets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, pool=pool, capture_error_mode="relaxed"):
                    self._step(st, b)
                if pool is None:
                    pool = g.pool()
                self.graphs[si][b] = g
        torch.cuda.synchronize(self.device)

    def bucket(self, batch: int) -> int:
        for b in self.buckets:
            if b >= batch:
                return b
        raise ValueError(f"batch {batch} exceeds the largest captured bucket {self.buckets[-1]}")

    def stage(self, q, k_new, v_new, block_ids, table_offsets, num_cached, seq_lens, buffer_set: int = 0) -> int:
        """Copy one step's inputs into a buffer set (on the current stream;
        non-blocking from pinned host memory) and pad it to its bucket.

        q: [layers, B, Hq, D]; k_new, v_new: [layers, B, Hkv, D] bf16;
        block_ids [nnz] / table_offsets [B+1]: the B sequences' block lists as
        a CSR pair (int32); num_cached, seq_lens: [B] int32 (L - 1 and L for a
        decode step).  Returns B.
        """
        B = int(seq_lens.shape[0])
        b = self.bucket(B)
        nnz = int(block_ids.shape[0])
        if nnz > self.sets[0].block_ids.numel():
            raise ValueError("more block-list entries than max_batch * max_blocks_per_seq")
        st = self.sets[buffer_set]
        st.q[:, :B].copy_(q, non_blocking=True)
        st.k_new[:, :B].copy_(k_new, non_blocking=True)
        st.v_new[:, :B].copy_(v_new, non_blocking=True)
        st.block_ids[:nnz].copy_(block_ids, non_blocking=True)
        st.table_offsets[:B + 1].copy_(table_offsets, non_blocking=True)
        st.num_cached[:B].copy_(num_cached, non_blocking=True)
        st.seq_lens[:B].copy_(seq_lens, non_blocking=True)
        if b > B:  # pad rows: empty sequences
            st.table_offsets[B + 1:b + 1].fill_(nnz)
            st.num_cached[B:b].fill_(0)
            st.seq_lens[B:b].fill_(0)
        return B

    def replay(self, B: int, buffer_set: int = 0) -> torch.Tensor:
        """Replay the step for the staged batch of B sequences; returns
        out[:, :B] (a view of the set's static output, valid until its next
        replay)."""
        self.graphs[buffer_set][self.bucket(B)].replay()
        return self.sets[buffer_set].out[:, :B]

    def run(self, q, k_new, v_new, block_ids, table_offsets, num_cached, seq_lens) -> torch.Tensor:
        """stage() into buffer set 0 and replay()."""
        B = self.stage(q, k_new, v_new, block_ids, table_offsets, num_cached, seq_lens, 0)
        return self.replay(B, 0)

    def metadata(self, B: int, buffer_set: int = 0) -> dict:
        """Views of the device metadata of the last replay's real rows."""
        m = self.sets[buffer_set].meta
        return {"slot_mapping": m["slot_mapping"][:B], "context_lens": m["context_lens"][:B],
                "block_tables": m["block_tables"][:B]}

    def sample(self, logits: torch.Tensor, temperatures: torch.Tensor, seed: int, offset: int) -> torch.Tensor:
        """Next tokens from the LM head's logits [B, V] (after the replay)."""
        return sample_exponential_race(logits, temperatures, seed, offset)
