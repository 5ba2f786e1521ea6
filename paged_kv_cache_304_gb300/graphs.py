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

This module is host plumbing around the C-ABI calls: it allocates the static
buffers with torch and captures/replays graphs; every step of the path runs in
the library's kernels.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import decode_workspace, kv_cache_write, paged_attn_decode, paged_attn_decode_fused_write


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
