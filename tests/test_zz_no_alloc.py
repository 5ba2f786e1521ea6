"""The decode entry point that allocates nothing (pkv_paged_attn_decode_noalloc).

Some callers cannot allocate device memory -- a plugin whose host engine owns
every device allocation, or a C caller that only holds the tensor pointers it
was handed -- so they cannot supply the workspace pkv_paged_attn_decode needs.
pkv_paged_attn_decode_noalloc keeps its scratch in a fixed array inside the
library instead.  These tests call it through the C ABI and check it against
pkv_paged_attn_decode on the same inputs, twice in a row (the array keeps the
first call's contents when the second starts), and check that a batch too
large for the fixed array is refused without a launch.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_304_gb300 as pkv
import workloads as W
from tests.gpu_util import check_close, i32, to_dev, to_host

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20


def _noalloc_fn():
    lib = pkv.load()
    fn = lib.pkv_paged_attn_decode_noalloc
    vp, i32t = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, vp, vp, vp, vp, i32t, i32t, i32t, i32t, i32t, i32t, i32t, i32t, ctypes.c_float, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(fn, q, kc, vc, ctx, tab, w, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ctx.data_ptr(), tab.data_ptr(), int(tab.shape[1]),
              w.batch, w.num_q_heads, w.num_kv_heads, 128, 256, w.num_blocks, w.max_context_len, float(w.scale),
              out.data_ptr(), stream)


@pytest.mark.parametrize("make", [W.qwen3_0p6b_decode, W.graph_padded_decode], ids=["b256", "b500_pad512"])
def test_noalloc_matches_workspace_decode_twice(make):
    w = make()
    fn = _noalloc_fn()
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    q, ctx, tab = to_dev(w.q), i32(w.context_lens), i32(w.block_tables)
    ref = pkv.paged_attn_decode(q, kc, vc, ctx, tab, w.scale, max_context_len=w.max_context_len)
    ref_bits = to_host(ref)
    ref64 = W.bf16_bits_to_f32(ref_bits).astype(np.float64)
    real = np.nonzero(w.context_lens > 0)[0]
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _call_noalloc(fn, q, kc, vc, ctx, tab, w, out)
        assert rc == 0, pkv.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        got = to_host(out)
        check_close(got, ref64, f"noalloc call {call + 1}", rows=real)
        assert (got[w.context_lens == 0] == 0).all()
    assert pkv.device_error() == []


def test_noalloc_rejects_batch_beyond_fixed_scratch():
    fn = _noalloc_fn()
    hq = 16
    need = pkv.decode_workspace_bytes(1024, hq)
    assert need > STATIC_SCRATCH_BYTES
    w = W.make_decode("big", 1, [5] * 1024, hq, 8, num_blocks=1100, fill_caches=False)
    kc = torch.zeros((w.num_blocks, 256, 8, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1024, hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 7.0)
    rc = _call_noalloc(fn, q, kc, kc, i32(w.context_lens), i32(w.block_tables), w, out)
    assert rc == -4  # PKV_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def _largest_batch_fitting(hq: int) -> int:
    """Largest batch whose decode scratch fits the fixed array on this GPU,
    from the library's own size query (so no SM count is assumed)."""
    lo, hi = 0, 1
    while pkv.decode_workspace_bytes(hi, hq) <= STATIC_SCRATCH_BYTES:
        lo, hi = hi, hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if pkv.decode_workspace_bytes(mid, hq) <= STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_batch_limit_exact():
    """At the largest batch whose scratch fits, the call runs and matches
    pkv_paged_attn_decode; one sequence more is refused before any launch."""
    hq = 16
    bmax = _largest_batch_fitting(hq)
    assert pkv.decode_workspace_bytes(bmax, hq) <= STATIC_SCRATCH_BYTES < pkv.decode_workspace_bytes(bmax + 1, hq)
    fn = _noalloc_fn()
    rng = np.random.default_rng(855)
    lens = rng.integers(1, 700, size=bmax)
    w = W.make_decode("limit", 855, lens, hq, 8)
    kc, vc = to_dev(w.k_cache), to_dev(w.v_cache)
    pkv.kv_cache_write(to_dev(w.k_new), to_dev(w.v_new), i32(w.slot_mapping), kc, vc)
    q, ctx, tab = to_dev(w.q), i32(w.context_lens), i32(w.block_tables)
    ref = to_host(pkv.paged_attn_decode(q, kc, vc, ctx, tab, w.scale, max_context_len=w.max_context_len))
    out = torch.full_like(q, float("nan"))
    rc = _call_noalloc(fn, q, kc, vc, ctx, tab, w, out)
    assert rc == 0, pkv.STATUS.get(rc, rc)
    torch.cuda.synchronize()
    check_close(to_host(out), W.bf16_bits_to_f32(ref).astype(np.float64), "noalloc at the batch limit")
    # One more sequence (a pad row) no longer fits: refused, nothing launched.
    w2 = W.make_decode("limit_plus_one", 856, lens, hq, 8, pad_to=bmax + 1, fill_caches=False)
    q2 = torch.zeros((bmax + 1, hq, 128), dtype=torch.bfloat16, device="cuda")
    out2 = torch.full_like(q2, 7.0)
    rc = _call_noalloc(fn, q2, kc, vc, i32(w2.context_lens), i32(w2.block_tables), w2, out2)
    assert rc == -4  # PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out2 == 7.0).all())
    assert pkv.device_error() == []
