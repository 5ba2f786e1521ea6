"""fp64 CPU oracle for the paged-KV attention path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its binding)
never imports it and shares no code with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, IEEE double, OpenMP over
output rows); this module compiles it with gcc and marshals numpy arrays.
bf16 tensors are numpy uint16 arrays of raw bit patterns.

Every function is pinned by ``tests/test_oracle.py`` against closed forms,
torch's scaled_dot_product_attention in float64, and invariants the pages
fix (block-permutation invariance, causality, chunk consistency, shared
prefixes, slot -1 skipping).  ``tests/test_oracle_mutants.py`` plants
mistakes in copies of the C source and checks that the pins catch them.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libpkv_oracle.so")
_lock = threading.Lock()
_default = None

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source file into a shared library at `out`."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (only when the source is newer than the library)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: oracle returned {rc}")


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.pkv_oracle_kv_cache_write.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i64, i64]
        lib.pkv_oracle_kv_cache_write.restype = ctypes.c_int
        lib.pkv_oracle_paged_attn_decode.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                                     ctypes.c_double, vp]
        lib.pkv_oracle_paged_attn_decode.restype = ctypes.c_int
        lib.pkv_oracle_paged_attn_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
                                                      ctypes.c_double, vp, i64, vp]
        lib.pkv_oracle_paged_attn_prefill.restype = ctypes.c_int
        lib.pkv_oracle_philox4x32_10.argtypes = [vp, vp, vp]
        lib.pkv_oracle_philox4x32_10.restype = None
        lib.pkv_oracle_uniform.argtypes = [i64, i64, ctypes.c_uint64, ctypes.c_uint64]
        lib.pkv_oracle_uniform.restype = ctypes.c_double
        lib.pkv_oracle_sample.argtypes = [vp, i64, vp, i64, i64, ctypes.c_uint64, ctypes.c_uint64, vp, vp]
        lib.pkv_oracle_sample.restype = ctypes.c_int
        lib.pkv_oracle_num_threads.restype = ctypes.c_int
        lib.pkv_oracle_set_num_threads.argtypes = [ctypes.c_int]
        self.lib = lib
        self.path = lib_path

    def num_threads(self) -> int:
        """Number of OpenMP threads the oracle runs on."""
        return int(self.lib.pkv_oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.lib.pkv_oracle_set_num_threads(int(n))

    def kv_cache_write(self, k, v, slot_mapping, k_cache, v_cache) -> None:
        """Scatter each token's K/V row into the caches in place; skip slot -1.

        k, v: uint16 [N, Hkv, D] (or [N, row_stride] 2-D, row_stride >= Hkv*D);
        slot_mapping: int32 [N]; k_cache, v_cache: uint16
        [num_blocks, bs, Hkv, D], C-contiguous, modified in place.
        """
        if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
            raise ValueError("caches must be C-contiguous")
        n = int(slot_mapping.shape[0])
        row = int(np.prod(k_cache.shape[2:]))
        k2 = _c(k, np.uint16).reshape(n, -1)
        v2 = _c(v, np.uint16).reshape(n, -1)
        slots = _c(slot_mapping, np.int32)
        num_slots = int(k_cache.shape[0] * k_cache.shape[1])
        _check(self.lib.pkv_oracle_kv_cache_write(_ptr(k2), k2.shape[1], _ptr(v2), v2.shape[1], _ptr(slots), n,
                                                  _ptr(k_cache), _ptr(v_cache), num_slots, row),
               "kv_cache_write")

    def paged_attn_decode(self, q, k_cache, v_cache, context_lens, block_tables, scale) -> np.ndarray:
        """Decode attention in fp64.  Returns float64 [B, Hq, D]."""
        q = _c(q, np.uint16)
        B, Hq, D = q.shape
        nb, bs, Hkv, D2 = k_cache.shape
        if D2 != D or not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
            raise ValueError("cache shape/layout mismatch")
        ctx = _c(context_lens, np.int32)
        tab = _c(block_tables, np.int32).reshape(B, -1)
        out = np.empty((B, Hq, D), dtype=np.float64)
        _check(self.lib.pkv_oracle_paged_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(ctx), _ptr(tab),
                                                     tab.shape[1], B, Hq, Hkv, D, bs, nb, float(scale),
                                                     _ptr(out)),
               "paged_attn_decode")
        return out

    def paged_attn_prefill(self, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale,
                           rows=None) -> np.ndarray:
        """Varlen causal prefill attention in fp64.  Returns float64 [T, Hq, D].

        With `rows` (global query row indices) only those rows are computed
        and every other row of the result is NaN.
        """
        q = _c(q, np.uint16)
        T, Hq, D = q.shape
        nb, bs, Hkv, D2 = k_cache.shape
        if D2 != D or not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
            raise ValueError("cache shape/layout mismatch")
        cq = _c(cu_seqlens_q, np.int32)
        ck = _c(cu_seqlens_k, np.int32)
        tab = _c(block_tables, np.int32).reshape(cq.size - 1, -1)
        out = np.full((T, Hq, D), np.nan, dtype=np.float64)
        if rows is None:
            rp, nr = None, 0
        else:
            r = _c(rows, np.int64)
            rp, nr = _ptr(r), int(r.size)
        _check(self.lib.pkv_oracle_paged_attn_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cq), _ptr(ck),
                                                      _ptr(tab), tab.shape[1], int(cq.size - 1), Hq, Hkv, D, bs,
                                                      nb, float(scale), rp, nr, _ptr(out)),
               "paged_attn_prefill")
        return out


    def philox4x32_10(self, counter, key) -> list[int]:
        """Philox4x32-10 block: four 32-bit words for a 4-word counter and 2-word key."""
        c = np.ascontiguousarray(counter, dtype=np.uint32)
        k = np.ascontiguousarray(key, dtype=np.uint32)
        out = np.zeros(4, dtype=np.uint32)
        self.lib.pkv_oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
        return [int(x) for x in out]

    def uniform(self, b: int, i: int, seed: int, offset: int) -> float:
        return float(self.lib.pkv_oracle_uniform(b, i, seed, offset))

    def sample(self, logits, temperatures, seed: int, offset: int = 0, with_scores: bool = False):
        """Exponential-race sampling in fp64.  logits float32 [B, V].

        Returns tokens int32 [B] (and float64 scores [B, V] = log p - log E)."""
        lg = _c(logits, np.float32)
        B, V = lg.shape
        t = _c(temperatures, np.float32)
        tokens = np.empty(B, dtype=np.int32)
        scores = np.empty((B, V), dtype=np.float64) if with_scores else None
        _check(self.lib.pkv_oracle_sample(_ptr(lg), V, _ptr(t), B, V, seed, offset, _ptr(tokens),
                                          _ptr(scores) if with_scores else None), "sample")
        return (tokens, scores) if with_scores else tokens


def default() -> Oracle:
    """The oracle built from ``pkv_oracle.c``."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def kv_cache_write(*a, **kw):
    return default().kv_cache_write(*a, **kw)


def paged_attn_decode(*a, **kw):
    return default().paged_attn_decode(*a, **kw)


def paged_attn_prefill(*a, **kw):
    return default().paged_attn_prefill(*a, **kw)


def num_threads() -> int:
    return default().num_threads()


def set_num_threads(n: int) -> None:
    default().set_num_threads(n)
