"""KV-cache write on the GPU vs the oracle: bit-exact, untouched elsewhere."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_304_gb300 as pkv
import workloads as W
from tests.gpu_util import assert_equal_chunks, i32, to_dev, to_host

pytestmark = pytest.mark.gpu


def _run(k_new, v_new, slots, k_cache, v_cache):
    kc, vc = to_dev(k_cache), to_dev(v_cache)
    pkv.kv_cache_write(to_dev(k_new), to_dev(v_new), i32(slots), kc, vc)
    torch.cuda.synchronize()
    okc, ovc = k_cache.copy(), v_cache.copy()
    oracle.kv_cache_write(k_new, v_new, slots, okc, ovc)
    assert_equal_chunks(to_host(kc), okc, "k_cache")
    assert_equal_chunks(to_host(vc), ovc, "v_cache")
    assert pkv.device_error() == []


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0.6b_decode", "graph_padded_decode",
                                  "chunked_prefill_prefix"])
def test_write_workloads(name):
    w = W.ALL[name]()
    _run(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)


def test_write_qwen3_8b_prefill_32768_tokens():
    w = W.qwen3_8b_prefill()
    _run(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)


def test_write_all_padding_is_noop():
    kc = np.full((4, 256, 8, 128), 0x1234, np.uint16)
    k = W.normal_bf16((7, 8, 128), 1, 1)
    _run(k, k, np.full(7, -1, np.int32), kc, kc.copy())


@pytest.mark.parametrize("hkv", [1, 2, 8])
def test_write_strided_rows(hkv):
    """Token rows with a stride larger than the row (a view into a fused qkv buffer)."""
    n, nb = 300, 6
    rng = np.random.default_rng(5)
    row = hkv * 128
    buf = W.normal_bf16((n, row * 3), 5, 1)
    slots = rng.choice(nb * 256, size=n, replace=False).astype(np.int32)
    slots[::7] = -1
    kc = np.full((nb, 256, hkv, 128), 0x7F7F, np.uint16)
    vc = np.full((nb, 256, hkv, 128), 0x3F3F, np.uint16)
    dbuf = to_dev(buf)
    dk, dv = dbuf[:, row:2 * row].view(n, hkv, 128), dbuf[:, 2 * row:].view(n, hkv, 128)
    dkc, dvc = to_dev(kc), to_dev(vc)
    pkv.kv_cache_write(dk, dv, i32(slots), dkc, dvc)
    torch.cuda.synchronize()
    oracle.kv_cache_write(buf[:, row:2 * row], buf[:, 2 * row:], slots, kc, vc)
    assert np.array_equal(to_host(dkc), kc) and np.array_equal(to_host(dvc), vc)


def test_write_out_of_range_slot_flags_and_skips():
    """A slot beyond the cache is skipped (no fault) and flagged on the device."""
    kc = np.full((2, 256, 8, 128), 0x1111, np.uint16)
    k = W.normal_bf16((3, 8, 128), 2, 1)
    slots = np.array([5, 2 * 256 + 9, 300], np.int32)
    dkc, dvc = to_dev(kc), to_dev(kc)
    pkv.device_error(clear=True)
    pkv.kv_cache_write(to_dev(k), to_dev(k), i32(slots), dkc, dvc)
    assert pkv.device_error() == ["SLOT_RANGE"]
    exp = kc.copy().reshape(512, 8, 128)
    exp[5], exp[300] = k[0], k[2]
    assert np.array_equal(to_host(dkc).reshape(512, 8, 128), exp)
