#!/usr/bin/env python
"""Benchmark of the paged-KV attention path on GB300.

One step = one Qwen3-0.6B-shaped decode step of every decoder layer: for each
of 28 layers, write the 256 new tokens' K/V into that layer's paged cache and
run decode attention over batch 256 with context lengths uniform in
[100, 2048], in one call (paged_attn_decode_fused_write; the separate
kv_cache_write + paged_attn_decode step is reported too); 16 query / 8 kv
heads, head_dim 128, block_size 256, shuffled block tables.  Inputs are synthetic
and seeded (seed 3042); every layer has its own cache, so each layer's
working set (about 1.2 GB) is far larger than L2 and no flush is needed.

Printed: one JSON line (rank 0).  `value` is the algorithmic HBM bytes of the
whole step (decode K/V/q/out/metadata plus the KV write's reads and writes)
divided by the step time.  `roofline` reports the dominant call
(paged_attn_decode_fused_write) against the measured HBM copy bandwidth.  Extra lines of
the same object report other workloads (graph-padded decode, 8B-shaped
decode, prefill TFLOP/s, the 32768-token KV write).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

`--impl reference` times the fp64 CPU oracle (the only reference
implementation of this path) on a bounded sample of the same workload.
Multi-GPU runs are independent replicas (the path has no exchange step).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attn HBM GB/s (% of 8 TB/s); prefill TFLOP/s; KV-write GB/s"
LAYERS = 28
NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


def recorded_traffic():
    """DRAM bytes per decode_kernel launch from the committed ncu capture,
    or None if the kernel's sources changed since it was taken."""
    import hashlib
    rec = os.path.join(ROOT, "profiles", "decode_kernel_traffic.txt")
    srcs = [os.path.join(ROOT, "paged_kv_cache_304_gb300", "csrc", f) for f in ("decode.cu", "pkv_device.cuh")]
    try:
        vals = {}
        with open(rec) as f:
            for line in f:
                if line.strip() and not line.startswith("#"):
                    k, v = line.split(None, 1)
                    vals[k] = v.strip()
        h = hashlib.sha256(b"".join(open(p, "rb").read() for p in srcs)).hexdigest()
        return int(vals["bytes_per_launch"]) if vals.get("sources_sha256") == h else None
    except (OSError, KeyError, ValueError):
        return None


def decode_bytes(ctx: np.ndarray, hq: int, hkv: int, d: int = 128, bs: int = 256) -> int:
    """Algorithmic bytes of one decode call: K and V rows of every context
    token, q in, out back, block-table entries and context lengths."""
    L = ctx.astype(np.int64)
    kv = int(L.sum()) * hkv * d * 2 * 2
    qo = ctx.size * hq * d * 2 * 2
    meta = int(((L + bs - 1) // bs).sum()) * 4 + ctx.size * 4
    return kv + qo + meta


def decode_unique_bytes(ctx: np.ndarray, tables: np.ndarray, hq: int, hkv: int, d: int = 128,
                        bs: int = 256) -> int:
    """decode_bytes with every cache row counted once: a block that several
    sequences share (a common prefix) is read from HBM once per call at best."""
    used = {}
    for b, L in enumerate(ctx.astype(np.int64)):
        for lb in range(int((L + bs - 1) // bs)):
            phys = int(tables[b, lb])
            used[phys] = max(used.get(phys, 0), int(min(bs, L - bs * lb)))
    kv = sum(used.values()) * hkv * d * 2 * 2
    return kv + decode_bytes(ctx, hq, hkv, d, bs) - int(ctx.astype(np.int64).sum()) * hkv * d * 2 * 2


def write_bytes(slots: np.ndarray, hkv: int, d: int = 128) -> int:
    """Algorithmic bytes of one KV write: K and V rows read and written for
    every non-padding token, plus the slot mapping."""
    n = int((slots >= 0).sum())
    return n * hkv * d * 2 * 2 * 2 + slots.size * 4


def prefill_flops(w: W.PrefillWorkload) -> int:
    """4 * D * Hq flops per (query, visible key) pair (QK^T and PV)."""
    n = w.seqlens_q.astype(np.int64)
    L = w.seqlens_k.astype(np.int64)
    c = L - n
    pairs = int((n * c + n * (n + 1) // 2).sum())
    return 4 * w.head_dim * w.num_q_heads * pairs


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms.

    Started before the warm-up (nvidia-smi takes a while to come up) and
    summarised over the samples whose timestamps fall inside the timed
    region (mark_start / mark_end); if none does, over the nearest ones.
    """

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
            deadline = time.time() + 8.0
            while time.time() < deadline and os.path.getsize(self.file.name) == 0:
                time.sleep(0.05)
        except (OSError, ValueError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _ts(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append((self._ts(parts[0]), parts[1:]))
        os.unlink(self.file.name)
        if not rows:
            return None
        inside = [r for t, r in rows if t is not None and self.t0 is not None and self.t0 <= t <= (self.t1 or t)]
        if not inside and self.t0 is not None:
            mid = (self.t0 + (self.t1 or self.t0)) / 2
            timed = [(abs(t - mid), r) for t, r in rows if t is not None]
            inside = [r for _, r in sorted(timed, key=lambda x: x[0])[:2]] if timed else [r for _, r in rows]
        use = inside or [r for _, r in rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in use) if v is not None]
        mx = [v for v in (num(r[2]) for r in use) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle
def oracle_decode_layer_rate(min_seconds: float = 10.0, max_reps: int = 20):
    """Time the fp64 oracle (write + decode) on one layer of the decode
    workload on the host cores; returns (GB/s of the same algorithmic bytes,
    threads, description)."""
    import oracle
    w = W.qwen3_0p6b_decode()
    nbytes = decode_bytes(w.context_lens, w.num_q_heads, w.num_kv_heads) + write_bytes(w.slot_mapping, w.num_kv_heads)
    reps, t_total = 0, 0.0
    while reps < max_reps and (t_total < min_seconds or reps == 0):
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        t0 = time.perf_counter()
        oracle.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, kc, vc)
        oracle.paged_attn_decode(w.q, kc, vc, w.context_lens, w.block_tables, w.scale)
        t_total += time.perf_counter() - t0
        reps += 1
    gbs = nbytes * reps / t_total / 1e9
    desc = (f"one of the 28 layers (batch 256, full KV write + decode), repeated {reps}x in "
            f"{t_total:.1f} s; GB/s of the same algorithmic bytes")
    return gbs, oracle.num_threads(), desc


def cpu_model() -> str:
    """The host CPU's model name as lscpu reports it (best effort)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def step_config(w, world: int) -> dict:
    """The `config` of the benchmark step (the same for both arms)."""
    return {"workload": "qwen3_0.6b_decode_b256: 28 layers x paged_attn_decode_fused_write (KV write + decode)",
            "batch": w.batch, "context_lens": "U[100, 2048], seed 3042", "layers": LAYERS,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": 128, "block_size": 256,
            "num_blocks_per_layer": w.num_blocks,
            "l2": "inputs larger than L2 (about 1.2 GB per layer, a different cache per layer)",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, timed on the host cores."""
    if rank != 0:
        return 0
    import oracle
    w = W.qwen3_0p6b_decode()
    # Bounded sample: the first 32 sequences of one layer (write + decode).
    B = 32
    nbytes = decode_bytes(w.context_lens[:B], w.num_q_heads, w.num_kv_heads) + \
        write_bytes(w.slot_mapping[:B], w.num_kv_heads)

    def step():
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        t0 = time.perf_counter()
        oracle.kv_cache_write(w.k_new[:B], w.v_new[:B], w.slot_mapping[:B], kc, vc)
        oracle.paged_attn_decode(w.q[:B], kc, vc, w.context_lens[:B], w.block_tables[:B], w.scale)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "each step: the KV write and decode of 32 of the 256 sequences of one of the "
                                   "28 layers, GB/s of those algorithmic bytes", "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm
def make_cache(torch, num_layers, nb, hkv, gen, device):
    """The global cache (2, layers, num_blocks, 256, hkv, 128), N(0,1) bf16."""
    kv = torch.empty((2, num_layers, nb, 256, hkv, 128), dtype=torch.bfloat16, device=device)
    flat = kv.view(-1)
    chunk = 1 << 28
    for lo in range(0, flat.numel(), chunk):
        hi = min(flat.numel(), lo + chunk)
        flat[lo:hi] = torch.randn(hi - lo, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return kv


def run_pkv(args, rank, world, local):
    global LAYERS
    LAYERS = args.layers
    import torch
    import paged_kv_cache_304_gb300 as pkv

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    pk, peak_kind = peaks()
    gen = torch.Generator(device=device)
    gen.manual_seed(3042 + rank)

    w = W.qwen3_0p6b_decode(fill_caches=False)
    B, hq, hkv, d = w.batch, w.num_q_heads, w.num_kv_heads, 128
    kv = make_cache(torch, LAYERS, w.num_blocks, hkv, gen, device)
    qs = torch.randn((LAYERS, B, hq, d), generator=gen, device=device).to(torch.bfloat16)
    ks = torch.randn((LAYERS, B, hkv, d), generator=gen, device=device).to(torch.bfloat16)
    vs = torch.randn((LAYERS, B, hkv, d), generator=gen, device=device).to(torch.bfloat16)
    outs = torch.empty_like(qs)
    slots = torch.from_numpy(w.slot_mapping).to(device)
    ctx = torch.from_numpy(w.context_lens).to(device)
    tab = torch.from_numpy(w.block_tables).to(device)
    ws = pkv.decode_workspace(B, hq, device)
    maxctx = w.max_context_len
    stream = torch.cuda.current_stream(device)

    def step():
        # one layer = the KV write fused into decode (rows a1 + a2 in one call);
        # nothing else runs in the step, so no event sits between the launches
        # (an event record would break the programmatic-dependent-launch overlap)
        for l in range(LAYERS):
            pkv.paged_attn_decode_fused_write(qs[l], ks[l], vs[l], slots, kv[0, l], kv[1, l], ctx, tab, w.scale,
                                              out=outs[l], workspace=ws, max_context_len=maxctx)

    step_bytes = LAYERS * (decode_bytes(w.context_lens, hq, hkv) + write_bytes(w.slot_mapping, hkv))
    dec_bytes = decode_bytes(w.context_lens, hq, hkv) + write_bytes(w.slot_mapping, hkv)

    with ClockSampler(local) as clocks:
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        assert pkv.device_error() == [], "device error during warm-up"
        barrier(world)
        torch.cuda.synchronize()
        clocks.mark_start()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        barrier(world)
    ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(ms, world, device)
    # average duration of one fused call over the timed region: the region
    # holds only these calls, back to back, so launch gaps count against it
    dec_ms = ms / LAYERS
    clk = clocks.summary()

    # end to end, through the device-chained step graph (DecodeStepGraph): per
    # step the host sends each layer's q, k_new, v_new and, for the step
    # metadata, only what each sequence holds -- its block list (a CSR pair),
    # num_cached and length -- from pinned memory; the replayed graph derives
    # the slots, context lengths and packed tables on the device and runs the
    # 28 fused write + decode calls; every layer's output comes back to pinned
    # host memory.  Two buffer sets: a copy stream stages step s+1 while step
    # s replays and drains step s-1's outputs.
    from paged_kv_cache_304_gb300.graphs import DecodeStepGraph

    L_host = w.context_lens.astype(np.int64)
    lists = [w.block_tables[i, :-(-int(L_host[i]) // 256)] for i in range(B)]
    offs = np.zeros(B + 1, np.int32)
    offs[1:] = np.cumsum([x.size for x in lists])
    h_q = qs.cpu().pin_memory()
    h_k = ks.cpu().pin_memory()
    h_v = vs.cpu().pin_memory()
    h_meta = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).pin_memory()
              for a in (np.concatenate(lists), offs, L_host - 1, L_host)]
    h_src = (h_q, h_k, h_v, *h_meta)
    h_out = torch.empty(outs.shape, dtype=outs.dtype, pin_memory=True)
    step_graph = DecodeStepGraph([(kv[0, l], kv[1, l]) for l in range(LAYERS)], hq, w.max_blocks_per_seq, w.scale,
                                 w.num_blocks, max_batch=B, max_context_len=maxctx, buckets=[B], buffer_sets=2)
    copy = torch.cuda.Stream(device)

    def run_e2e(nsteps):
        ev = lambda: [torch.cuda.Event() for _ in range(nsteps)]
        in_ready, in_free, done, out_free = ev(), ev(), ev(), ev()

        def load(s):
            with torch.cuda.stream(copy):
                if s >= 2:
                    copy.wait_event(in_free[s - 2])   # step s-2 has finished reading this set
                    copy.wait_event(out_free[s - 2])  # and its outputs have left it
                step_graph.stage(*h_src, buffer_set=s % 2)
                in_ready[s].record(copy)

        copy.wait_stream(stream)
        load(0)
        for s in range(nsteps):
            if s + 1 < nsteps:
                load(s + 1)
            stream.wait_event(in_ready[s])
            out = step_graph.replay(B, buffer_set=s % 2)
            in_free[s].record(stream)
            done[s].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(done[s])
                h_out.copy_(out, non_blocking=True)
                out_free[s].record(copy)
        stream.wait_stream(copy)

    run_e2e(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 50))
    barrier(world)
    e0.record(stream)
    run_e2e(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, device)
    h2d = sum(t.numel() * t.element_size() for t in h_src)
    d2h = h_out.numel() * h_out.element_size()
    e2e_out_ok = bool(torch.equal(h_out.to(device), outs))  # the chained step gives the eager step's outputs
    del step_graph

    # the same step with the write fused into decode, and both captured once
    # as a CUDA graph (bucket = batch) and replayed
    from paged_kv_cache_304_gb300.graphs import DecodeGraphRunner

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)

    extra = {}
    for name, fused in (("decode_step_cuda_graph", False), ("decode_step_fused_write_cuda_graph", True)):
        runner = DecodeGraphRunner([(kv[0, l], kv[1, l]) for l in range(LAYERS)], hq, w.max_blocks_per_seq, w.scale,
                                   max_batch=B, max_context_len=maxctx, buckets=[B], fused=fused)
        runner.run(qs, ks, vs, slots, ctx, tab)
        gms = timed(runner.graphs[B].replay)
        extra[name] = {"ms_per_step": round(gms, 4), "GB/s": round(step_bytes * world / (gms / 1e3) / 1e9, 2)}
        del runner
    # the runner as a caller uses it: a real batch that is not a bucket size,
    # copied into the static buffers and padded (slot -1, length 0) to the
    # next bucket, then replayed
    Bp = B - 6
    runner = DecodeGraphRunner([(kv[0, l], kv[1, l]) for l in range(LAYERS)], hq, w.max_blocks_per_seq, w.scale,
                               max_batch=B, max_context_len=maxctx, buckets=[Bp - Bp % 16, B], fused=True)
    real = (qs[:, :Bp], ks[:, :Bp], vs[:, :Bp], slots[:Bp], ctx[:Bp], tab[:Bp])
    rms = timed(lambda: runner.run(*real))
    rbytes = LAYERS * (decode_bytes(w.context_lens[:Bp], hq, hkv) + write_bytes(w.slot_mapping[:Bp], hkv))
    extra[f"decode_step_graph_runner_b{Bp}_bucket{B}"] = {
        "ms_per_step": round(rms, 4), "GB/s": round(rbytes * world / (rms / 1e3) / 1e9, 2),
        "note": "DecodeGraphRunner.run: input copies, pad rows and the replay of the fused 28-layer graph"}
    del runner
    def unfused_step():
        for l in range(LAYERS):
            pkv.kv_cache_write(ks[l], vs[l], slots, kv[0, l], kv[1, l])
            pkv.paged_attn_decode(qs[l], kv[0, l], kv[1, l], ctx, tab, w.scale, out=outs[l], workspace=ws,
                                  max_context_len=maxctx)

    ums = timed(unfused_step)
    extra["decode_step_separate_write"] = {"ms_per_step": round(ums, 4),
                                           "GB/s": round(step_bytes * world / (ums / 1e3) / 1e9, 2),
                                           "note": "kv_cache_write then paged_attn_decode per layer (eager)"}
    if not args.no_extra:
        extra.update(run_extras(torch, pkv, device, gen, pk))
    assert pkv.device_error() == [], "device error during the benchmark"

    value = step_bytes * world / (ms / 1e3) / 1e9
    dec_gbs = dec_bytes / (dec_ms / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": step_config(w, world),
        "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(dec_gbs / pk["hbm_gbs"], 4), "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(dec_gbs / NOMINAL_HBM_GBS, 4),
                     "kernel": "paged_attn_decode_fused_write call (decode_kernel with the KV write, then "
                               "decode_combine_kernel); time per call = timed region / calls",
                     "bytes_per_launch": dec_bytes, "ms_per_launch": round(dec_ms, 5),
                     "traffic": recorded_traffic() if LAYERS == 28 or LAYERS == 1 else None},
        "clocks": clk,
        "e2e": {"value": round(step_bytes * world / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "DecodeStepGraph: per-sequence block lists and lengths in, metadata on the device, "
                        "28 fused write+decode calls replayed from one graph",
                "outputs_equal_eager_step": e2e_out_ok},
        "gpu_launches": args.steps * LAYERS * 2,
        "extra": extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, cores, desc = oracle_decode_layer_rate()
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "cpu_model": cpu_model()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _time_calls(torch, fn, reps: int, warm: int = 3, per_graph: int = 10):
    """Median per-call device time of `fn`, from CUDA-graph replays of
    `per_graph` back-to-back calls (so host-side argument marshalling is not
    timed); falls back to event-bracketed calls if capture fails."""
    stream = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for _ in range(per_graph):
                fn()
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(max(1, reps)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) for x, y in times) / per_graph
    except RuntimeError:
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) for x, y in times)


def _l2_evictor(torch, device):
    """A callable that evicts L2 by reading a 256 MB buffer (a read leaves
    clean lines; a write would leave dirty lines whose write-back would be
    charged to whatever runs next)."""
    src = torch.ones(64 << 20, dtype=torch.float32, device=device)
    dst = torch.empty(1, dtype=torch.float32, device=device)
    return lambda: torch.sum(src, dim=0, keepdim=True, out=dst)


def _time_cold(torch, fn, reps: int, evict):
    """Median device time of one call of `fn` (replayed from a CUDA graph)
    with L2 evicted before each rep; the eviction is outside the events."""
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        fn()
    times = []
    for _ in range(reps):
        evict()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) for x, y in times)


def _decode_extra(torch, pkv, device, gen, w: W.DecodeWorkload, pk, reps=20, cold_too=False):
    kv = make_cache(torch, 1, w.num_blocks, w.num_kv_heads, gen, device)
    q = torch.randn(w.q.shape, generator=gen, device=device).to(torch.bfloat16)
    ctx = torch.from_numpy(w.context_lens).to(device)
    tab = torch.from_numpy(w.block_tables).to(device)
    ws = pkv.decode_workspace(w.batch, w.num_q_heads, device)
    out = torch.empty_like(q)

    def call():
        pkv.paged_attn_decode(q, kv[0, 0], kv[1, 0], ctx, tab, w.scale, out=out, workspace=ws,
                              max_context_len=w.max_context_len)
    ms = _time_calls(torch, call, reps)
    nbytes = decode_bytes(w.context_lens, w.num_q_heads, w.num_kv_heads)
    gbs = nbytes / (ms / 1e3) / 1e9
    res = {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 4),
           "bytes": nbytes}
    ubytes = decode_unique_bytes(w.context_lens, w.block_tables, w.num_q_heads, w.num_kv_heads)
    if ubytes != nbytes:
        res["unique_bytes"] = ubytes
        res["GB/s_unique"] = round(ubytes / (ms / 1e3) / 1e9, 1)
    if cold_too:
        # back-to-back replays keep a small working set in L2; this is the
        # latency of one call whose K/V must come from HBM
        res["ms_cold_l2"] = round(_time_cold(torch, call, reps, _l2_evictor(torch, device)), 4)
    del kv
    return res


def _write_extra(torch, pkv, device, gen, w, pk, reps=20):
    kv = make_cache(torch, 1, w.num_blocks, w.num_kv_heads, gen, device)
    k = torch.randn(w.k_new.shape, generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn(w.v_new.shape, generator=gen, device=device).to(torch.bfloat16)
    slots = torch.from_numpy(w.slot_mapping).to(device)
    # the write's own working set is about the size of L2: evict L2 between reps
    evict = _l2_evictor(torch, device)

    def fn():
        pkv.kv_cache_write(k, v, slots, kv[0, 0], kv[1, 0])

    for _ in range(3):
        fn()
    times = []
    stream = torch.cuda.current_stream()
    for _ in range(reps):
        evict()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.median(x.elapsed_time(y) for x, y in times)
    nbytes = write_bytes(w.slot_mapping, w.num_kv_heads)
    gbs = nbytes / (ms / 1e3) / 1e9
    del kv
    return {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 4),
            "bytes": nbytes, "l2": "evicted between reps (256 MB read)"}


def _prefill_extra(torch, pkv, device, gen, w: W.PrefillWorkload, pk, reps=10, step_too=False):
    kv = make_cache(torch, 1, w.num_blocks, w.num_kv_heads, gen, device)
    q = torch.randn(w.q.shape, generator=gen, device=device).to(torch.bfloat16)
    cq = torch.from_numpy(w.cu_seqlens_q).to(device)
    ck = torch.from_numpy(w.cu_seqlens_k).to(device)
    tab = torch.from_numpy(w.block_tables).to(device)
    out = torch.empty_like(q)
    try:
        ms = _time_calls(torch, lambda: pkv.paged_attn_prefill(q, kv[0, 0], kv[1, 0], cq, ck, tab, w.scale,
                                                               w.max_seqlen_q, w.max_seqlen_k, out=out), reps)
    except pkv.PkvError as e:
        return {"unavailable": str(e)}
    flops = prefill_flops(w)
    tf = flops / (ms / 1e3) / 1e12
    res = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_of_measured_bf16": round(tf / pk["bf16_tflops"], 4),
           "flops": flops}
    if step_too:
        # the whole prefill step of one layer: the KV write of the new tokens
        # then attention, as two calls and as the one fused call
        kn = torch.randn(w.k_new.shape, generator=gen, device=device).to(torch.bfloat16)
        vn = torch.randn(w.v_new.shape, generator=gen, device=device).to(torch.bfloat16)
        slots = torch.from_numpy(w.slot_mapping).to(device)
        ws = pkv.prefill_fused_workspace(device)

        def separate():
            pkv.kv_cache_write(kn, vn, slots, kv[0, 0], kv[1, 0])
            pkv.paged_attn_prefill(q, kv[0, 0], kv[1, 0], cq, ck, tab, w.scale, w.max_seqlen_q, w.max_seqlen_k,
                                   out=out)

        def fused():
            pkv.paged_attn_prefill_fused_write(q, kn, vn, slots, kv[0, 0], kv[1, 0], cq, ck, tab, w.scale,
                                               w.max_seqlen_q, w.max_seqlen_k, out=out, workspace=ws)

        res["step_write_then_prefill_ms"] = round(_time_calls(torch, separate, reps), 4)
        res["step_fused_write_prefill_ms"] = round(_time_calls(torch, fused, reps), 4)
    del kv
    return res


def _metadata_extra(torch, pkv, device, w, reps=20):
    """Device-side step metadata (slot mapping, cu_seqlens, packed tables)."""
    if isinstance(w, W.DecodeWorkload):
        L = w.context_lens[: w.real_batch].astype(np.int64)
        c = L - 1
    else:
        L = w.seqlens_k.astype(np.int64)
        c = L - w.seqlens_q
    tabs = [w.block_tables[i, : -(-int(L[i]) // 256)] for i in range(L.size)]
    offs = np.zeros(L.size + 1, np.int32)
    offs[1:] = np.cumsum([t.size for t in tabs])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    args = (dev(np.concatenate(tabs)), dev(offs), dev(c), dev(L), int((L - c).sum()), w.max_blocks_per_seq,
            w.num_blocks)
    ms = _time_calls(torch, lambda: pkv.prepare_metadata(*args), reps)
    return {"us": round(ms * 1e3, 2), "sequences": int(L.size), "new_tokens": int((L - c).sum())}


def _sampler_extra(torch, pkv, device, gen, pk, B=256, V=151936, reps=20):
    """Exponential-race sampling over a Qwen3-sized vocabulary (4 bytes of
    fp32 logits per token read once)."""
    logits = torch.randn((B, V), generator=gen, device=device, dtype=torch.float32) * 2
    temps = torch.full((B,), 0.7, device=device, dtype=torch.float32)
    out = torch.empty(B, dtype=torch.int32, device=device)
    ws = torch.empty(max(256, int(pkv.load().pkv_sample_workspace_bytes(B, V))), dtype=torch.uint8, device=device)
    ms = _time_calls(torch, lambda: pkv.sample_exponential_race(logits, temps, 1, 2, out=out, workspace=ws), reps)
    nbytes = B * V * 4 + B * 8
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / pk["hbm_gbs"], 4),
            "batch": B, "vocab": V}


def run_extras(torch, pkv, device, gen, pk):
    out = {}
    out["sampler_b256_vocab151936"] = _sampler_extra(torch, pkv, device, gen, pk)
    out["metadata_qwen3_0.6b_decode_b256"] = _metadata_extra(torch, pkv, device, W.qwen3_0p6b_decode(fill_caches=False))
    out["metadata_chunked_prefill_prefix"] = _metadata_extra(torch, pkv, device,
                                                             W.chunked_prefill_prefix(fill_caches=False))
    out["metadata_qwen3_8b_prefill_4x8192"] = _metadata_extra(torch, pkv, device, W.qwen3_8b_prefill(fill_caches=False))
    out["graph_padded_decode_b500_pad512"] = _decode_extra(torch, pkv, device, gen,
                                                            W.graph_padded_decode(fill_caches=False), pk)
    out["qwen3_8b_decode_b64"] = _decode_extra(torch, pkv, device, gen, W.qwen3_8b_decode(fill_caches=False), pk)
    out["tiny_decode_b4_latency"] = _decode_extra(torch, pkv, device, gen, W.tiny_decode(fill_caches=False), pk,
                                                  cold_too=True)
    out["kv_write_qwen3_8b_prefill_32768_tokens"] = _write_extra(torch, pkv, device, gen,
                                                                 W.qwen3_8b_prefill(fill_caches=False), pk)
    out["chunked_prefill_prefix_budget16384"] = _prefill_extra(torch, pkv, device, gen,
                                                               W.chunked_prefill_prefix(fill_caches=False), pk,
                                                               step_too=True)
    out["qwen3_8b_prefill_4x8192"] = _prefill_extra(torch, pkv, device, gen, W.qwen3_8b_prefill(fill_caches=False),
                                                    pk, step_too=True)
    torch.cuda.empty_cache()
    return out


CASES = ("step", "prefill_8b", "prefill_chunked", "decode_8b", "decode_padded", "decode_tiny", "write_32768",
         "sampler", "metadata")


def run_case(args, local):
    """One workload on its own (for profiling): time it and print one JSON line."""
    import torch
    import paged_kv_cache_304_gb300 as pkv
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    pk, peak_kind = peaks()
    gen = torch.Generator(device=device)
    gen.manual_seed(3040)
    reps = max(1, args.steps)
    if args.case == "prefill_8b":
        n = args.prefill_seqs
        if n == 4:
            w = W.qwen3_8b_prefill(fill_caches=False)
        else:  # a smaller pool for profiling runs
            w = W.make_prefill(f"qwen3_8b_prefill_{n}x8192", 3045, [8192] * n, [0] * n, 32, 8,
                               num_blocks=32 * n + 8, fill_caches=False)
        res = _prefill_extra(torch, pkv, device, gen, w, pk, reps=reps, step_too=True)
    elif args.case == "prefill_chunked":
        w = W.chunked_prefill_prefix(fill_caches=False)
        res = _prefill_extra(torch, pkv, device, gen, w, pk, reps=reps, step_too=True)
    elif args.case == "decode_8b":
        w = W.qwen3_8b_decode(fill_caches=False)
        res = _decode_extra(torch, pkv, device, gen, w, pk, reps=reps)
    elif args.case == "decode_padded":
        w = W.graph_padded_decode(fill_caches=False)
        res = _decode_extra(torch, pkv, device, gen, w, pk, reps=reps)
    elif args.case == "decode_tiny":
        w = W.tiny_decode(fill_caches=False)
        res = _decode_extra(torch, pkv, device, gen, w, pk, reps=reps, cold_too=True)
    elif args.case == "sampler":
        res = _sampler_extra(torch, pkv, device, gen, pk, reps=reps)
        print(json.dumps({"case": args.case, "workload": "sampler_b256_vocab151936", "peak_kind": peak_kind, **res}),
              flush=True)
        return 0
    elif args.case == "metadata":
        w = W.qwen3_0p6b_decode(fill_caches=False)
        res = _metadata_extra(torch, pkv, device, w, reps=reps)
    else:
        w = W.qwen3_8b_prefill(fill_caches=False)
        res = _write_extra(torch, pkv, device, gen, w, pk, reps=reps)
    assert pkv.device_error() == [], "device error"
    print(json.dumps({"case": args.case, "workload": w.name, "peak_kind": peak_kind, **res}), flush=True)
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--case", choices=CASES, default="step",
                    help="step (the benchmark) or one workload on its own, for profiling")
    ap.add_argument("--prefill-seqs", type=int, default=4, help="sequences of 8192 tokens for --case prefill_8b")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="decoder layers per step (28 for the benchmark; 1 for a small profiling case)")
    args = ap.parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.case != "step":
        return run_case(args, local)
    return run_pkv(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
