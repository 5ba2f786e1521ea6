"""Python binding of libpkv.so, the sm_103a paged-KV attention library.

Argument marshalling only: every function below derives the C-ABI arguments
(device pointers, sizes, strides, the current CUDA stream) from torch
tensors and calls the library.  All computation runs in the library's CUDA
kernels; there is no other code path.  If the compiled library cannot be
loaded, importing works but every call raises ``PkvLibraryError``.

The three calls follow nano-vllm's attention layer (page "13. 读一个最小推理引擎：
nano-vllm", section "第六站：注意力层"): write the step's K/V into the paged
cache, then attend -- varlen prefill or one-token decode -- through block
tables.  See ``include/pkv.h`` for the exact contract of each call.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pkv.h")

PKV_OK = 0
STATUS = {
    0: "PKV_OK", -1: "PKV_ERR_NULL", -2: "PKV_ERR_SHAPE", -3: "PKV_ERR_UNSUPPORTED",
    -4: "PKV_ERR_WORKSPACE", -5: "PKV_ERR_CUDA", -6: "PKV_ERR_ALIGN",
}
DEVERR = {0x1: "SLOT_RANGE", 0x2: "BLOCK_RANGE", 0x4: "LEN_RANGE", 0x8: "WAIT_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class PkvLibraryError(RuntimeError):
    """The compiled CUDA library is missing or could not be loaded."""


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def exported_functions() -> list[str]:
    """Names of the functions declared in include/pkv.h."""
    import re
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def load(path: str | None = None):
    """Load (once) and return the ctypes handle of libpkv.so."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise PkvLibraryError(f"{p} not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        try:
            lib = ctypes.CDLL(p)
        except OSError as e:  # pragma: no cover
            raise PkvLibraryError(f"cannot load {p}: {e}") from e
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_version.restype = ctypes.c_int
        lib.pkv_kv_cache_write.argtypes = [vp, i64, vp, i64, vp, i32, vp, vp, i32, i32, i32, i32, vp]
        lib.pkv_kv_cache_write.restype = ctypes.c_int
        lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32]
        lib.pkv_decode_workspace_bytes.restype = sz
        lib.pkv_paged_attn_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp,
                                              vp, sz, vp]
        lib.pkv_paged_attn_decode.restype = ctypes.c_int
        lib.pkv_paged_attn_decode_fused_write.argtypes = [vp, vp, i64, vp, i64, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                          i32, i32, i32, i32, f32, vp, vp, sz, vp]
        lib.pkv_paged_attn_decode_fused_write.restype = ctypes.c_int
        lib.pkv_paged_attn_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                               i32, f32, vp, vp]
        lib.pkv_paged_attn_prefill.restype = ctypes.c_int
        lib.pkv_prepare_metadata.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.pkv_prepare_metadata.restype = ctypes.c_int
        lib.pkv_sample_workspace_bytes.argtypes = [i32, i32]
        lib.pkv_sample_workspace_bytes.restype = sz
        lib.pkv_sample_exponential_race.argtypes = [vp, i64, vp, i32, i32, ctypes.c_uint64, ctypes.c_uint64, vp, vp,
                                                    sz, vp]
        lib.pkv_sample_exponential_race.restype = ctypes.c_int
        lib.pkv_prefill_fused_workspace_bytes.argtypes = []
        lib.pkv_prefill_fused_workspace_bytes.restype = sz
        lib.pkv_paged_attn_prefill_fused_write.argtypes = [vp, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                           i32, i32, i32, i32, i32, i32, i32, f32, vp, vp, sz, vp]
        lib.pkv_paged_attn_prefill_fused_write.restype = ctypes.c_int
        lib.pkv_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        lib.pkv_device_error.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(fn: str, status: int) -> None:
    if status != PKV_OK:
        raise PkvError(fn, status)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _cache_dims(k_cache: torch.Tensor):
    if k_cache.dim() != 4 or not k_cache.is_contiguous():
        raise ValueError("caches must be contiguous (num_blocks, block_size, num_kv_heads, head_dim)")
    return tuple(int(x) for x in k_cache.shape)


def kv_cache_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor) -> None:
    """Scatter k, v [N, Hkv, D] (bf16) into the caches at slot_mapping [N] (int32); -1 is skipped."""
    lib = load()
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, n, torch.bfloat16)
    _dev(slot_mapping, "slot_mapping", torch.int32)
    nb, bs, hkv, d = _cache_dims(k_cache)
    if tuple(v_cache.shape) != tuple(k_cache.shape) or not v_cache.is_contiguous():
        raise ValueError("v_cache must match k_cache")
    n = int(slot_mapping.shape[0])
    for t, name in ((k, "k"), (v, "v")):
        if t.shape[0] != n or t[0].numel() != hkv * d or (n and not t[0].is_contiguous()):
            raise ValueError(f"{name} must be [N, {hkv}, {d}] with contiguous rows")
    if not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous")
    _check("pkv_kv_cache_write", lib.pkv_kv_cache_write(
        k.data_ptr(), k.stride(0) if n else hkv * d, v.data_ptr(), v.stride(0) if n else hkv * d,
        slot_mapping.data_ptr(), n, k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, d, _stream(k_cache)))


def decode_workspace_bytes(batch: int, num_q_heads: int, max_context_len: int = 0) -> int:
    """Scratch bytes of paged_attn_decode on the current device (depends on its SM count)."""
    return int(load().pkv_decode_workspace_bytes(batch, num_q_heads, max_context_len))


def decode_workspace(batch: int, num_q_heads: int, device, max_context_len: int = 0) -> torch.Tensor:
    """A workspace tensor for paged_attn_decode (uninitialised bytes)."""
    with torch.cuda.device(device):
        n = decode_workspace_bytes(batch, num_q_heads, max_context_len)
    return torch.empty(max(256, n), dtype=torch.uint8, device=device)


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, context_lens: torch.Tensor,
                      block_tables: torch.Tensor, scale: float, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, max_context_len: int | None = None) -> torch.Tensor:
    """Decode attention.  q [B, Hq, D] bf16; context_lens [B] int32; block_tables [B, max_blocks] int32.

    ``max_context_len`` is a host-known upper bound of context_lens (default:
    block_tables.shape[1] * block_size); it is never read back from the device.
    """
    lib = load()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, n, torch.bfloat16)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(block_tables, "block_tables", torch.int32)
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, dq = (int(x) for x in q.shape)
    if dq != d or not q.is_contiguous():
        raise ValueError("q must be contiguous [B, Hq, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous [B, max_blocks]")
    if context_lens.shape != (B,) or not context_lens.is_contiguous():
        raise ValueError("context_lens must be contiguous [B]")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if workspace is None:
        workspace = decode_workspace(B, hq, q.device)
    maxb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = maxb * bs
    _check("pkv_paged_attn_decode", lib.pkv_paged_attn_decode(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), context_lens.data_ptr(), block_tables.data_ptr(), maxb,
        B, hq, hkv, d, bs, nb, int(max_context_len), float(scale), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(q)))
    return out


def paged_attn_decode_fused_write(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                  slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  context_lens: torch.Tensor, block_tables: torch.Tensor, scale: float,
                                  out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                  max_context_len: int | None = None) -> torch.Tensor:
    """kv_cache_write(k_new, v_new, slot_mapping, ...) + paged_attn_decode(...) in one call.

    slot_mapping[b] must be the slot of position context_lens[b] - 1 or -1.
    """
    lib = load()
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, n, torch.bfloat16)
    for t, n in ((slot_mapping, "slot_mapping"), (context_lens, "context_lens"), (block_tables, "block_tables")):
        _dev(t, n, torch.int32)
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, dq = (int(x) for x in q.shape)
    if dq != d or not q.is_contiguous():
        raise ValueError("q must be contiguous [B, Hq, head_dim]")
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if t.shape[0] != B or t[0].numel() != hkv * d or (B and not t[0].is_contiguous()):
            raise ValueError(f"{name} must be [B, {hkv}, {d}] with contiguous rows")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous [B, max_blocks]")
    if context_lens.shape != (B,) or slot_mapping.shape != (B,):
        raise ValueError("context_lens and slot_mapping must be [B]")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, hq, q.device)
    maxb = int(block_tables.shape[1])
    if max_context_len is None:
        max_context_len = maxb * bs
    _check("pkv_paged_attn_decode_fused_write", lib.pkv_paged_attn_decode_fused_write(
        q.data_ptr(), k_new.data_ptr(), k_new.stride(0) if B else hkv * d, v_new.data_ptr(),
        v_new.stride(0) if B else hkv * d, slot_mapping.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        context_lens.data_ptr(), block_tables.data_ptr(), maxb, B, hq, hkv, d, bs, nb, int(max_context_len),
        float(scale), out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(q)))
    return out


def paged_attn_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, cu_seqlens_q: torch.Tensor,
                       cu_seqlens_k: torch.Tensor, block_tables: torch.Tensor, scale: float, max_seqlen_q: int,
                       max_seqlen_k: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """Varlen causal prefill attention through block tables (bottom-right causal alignment).

    q [T, Hq, D] bf16 packed by cu_seqlens_q [S+1]; cu_seqlens_k [S+1] gives each
    sequence's total length in the cache; max_seqlen_q/k are host-known bounds.
    """
    lib = load()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, n, torch.bfloat16)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k"), (block_tables, "block_tables")):
        _dev(t, n, torch.int32)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    nb, bs, hkv, d = _cache_dims(k_cache)
    T, hq, dq = (int(x) for x in q.shape)
    if dq != d or not q.is_contiguous():
        raise ValueError("q must be contiguous [T, Hq, head_dim]")
    S = int(cu_seqlens_q.shape[0]) - 1
    if cu_seqlens_k.shape[0] != S + 1 or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("cu_seqlens_k must be [S+1] and block_tables [S, max_blocks]")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    _check("pkv_paged_attn_prefill", lib.pkv_paged_attn_prefill(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
        block_tables.data_ptr(), int(block_tables.shape[1]), S, T, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
        bs, nb, float(scale), out.data_ptr(), _stream(q)))
    return out


def prefill_fused_workspace(device) -> torch.Tensor:
    """A zeroed workspace for paged_attn_prefill_fused_write (reusable by the
    calls of one stream)."""
    n = int(load().pkv_prefill_fused_workspace_bytes())
    return torch.zeros(max(256, n), dtype=torch.uint8, device=device)


def paged_attn_prefill_fused_write(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                   slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                                   block_tables: torch.Tensor, scale: float, max_seqlen_q: int, max_seqlen_k: int,
                                   out: torch.Tensor | None = None,
                                   workspace: torch.Tensor | None = None) -> torch.Tensor:
    """kv_cache_write of the step's new tokens then paged_attn_prefill, in one call.

    k_new, v_new [T, Hkv, D] bf16 with rows 16-byte aligned; slot_mapping [T]
    int32; workspace: from prefill_fused_workspace() (zeroed once, then reused).
    """
    lib = load()
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, n, torch.bfloat16)
    for t, n in ((slot_mapping, "slot_mapping"), (cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k"),
                 (block_tables, "block_tables")):
        _dev(t, n, torch.int32)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    nb, bs, hkv, d = _cache_dims(k_cache)
    T, hq, dq = (int(x) for x in q.shape)
    if dq != d or not q.is_contiguous():
        raise ValueError("q must be contiguous [T, Hq, head_dim]")
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if t.dim() != 3 or tuple(t.shape) != (T, hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{n} must be [T, Hkv, head_dim] with contiguous rows")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [T]")
    S = int(cu_seqlens_q.shape[0]) - 1
    if cu_seqlens_k.shape[0] != S + 1 or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise ValueError("cu_seqlens_k must be [S+1] and block_tables [S, max_blocks]")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if workspace is None:
        workspace = prefill_fused_workspace(q.device)
    _check("pkv_paged_attn_prefill_fused_write", lib.pkv_paged_attn_prefill_fused_write(
        q.data_ptr(), k_new.data_ptr(), k_new.stride(0), v_new.data_ptr(), v_new.stride(0), slot_mapping.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
        block_tables.data_ptr(), int(block_tables.shape[1]), S, T, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d,
        bs, nb, float(scale), out.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream(q)))
    return out


def prepare_metadata(block_ids: torch.Tensor, table_offsets: torch.Tensor, num_cached: torch.Tensor,
                     seq_lens: torch.Tensor, token_capacity: int, max_blocks_per_seq: int, num_blocks: int,
                     block_size: int = 256, out: dict | None = None) -> dict:
    """Step metadata on the device from per-sequence (block table, num_cached, length).

    block_ids/table_offsets: the block tables as a CSR pair (int32); num_cached,
    seq_lens: [S] int32 (num_cached = seq_len = 0 marks a CUDA-graph pad row).
    Returns device tensors cu_seqlens_q, cu_seqlens_k, context_lens,
    slot_mapping [token_capacity] (-1 past the real tokens) and block_tables
    [S, max_blocks_per_seq]; `out` may hold preallocated tensors of those
    names and shapes (int32, contiguous) to write into instead.
    """
    lib = load()
    for t, n in ((block_ids, "block_ids"), (table_offsets, "table_offsets"), (num_cached, "num_cached"),
                 (seq_lens, "seq_lens")):
        _dev(t, n, torch.int32)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    S = int(seq_lens.shape[0])
    if num_cached.shape != (S,) or table_offsets.shape != (S + 1,):
        raise ValueError("num_cached must be [S] and table_offsets [S+1]")
    dev = seq_lens.device
    shapes = {"cu_seqlens_q": (S + 1,), "cu_seqlens_k": (S + 1,), "context_lens": (S,),
              "slot_mapping": (max(token_capacity, 0),), "block_tables": (S, max_blocks_per_seq)}
    if out is None:
        out = {k: torch.empty(v, dtype=torch.int32, device=dev) for k, v in shapes.items()}
    else:
        for k, v in shapes.items():
            t = out[k]
            _dev(t, k, torch.int32)
            if tuple(t.shape) != v or not t.is_contiguous():
                raise ValueError(f"out[{k!r}] must be a contiguous int32 tensor of shape {v}")
    _check("pkv_prepare_metadata", lib.pkv_prepare_metadata(
        block_ids.data_ptr(), table_offsets.data_ptr(), num_cached.data_ptr(), seq_lens.data_ptr(), S,
        int(token_capacity), int(max_blocks_per_seq), int(block_size), int(num_blocks),
        out["cu_seqlens_q"].data_ptr(), out["cu_seqlens_k"].data_ptr(), out["context_lens"].data_ptr(),
        out["slot_mapping"].data_ptr(), out["block_tables"].data_ptr(), _stream(seq_lens)))
    return out


def sample_exponential_race(logits: torch.Tensor, temperatures: torch.Tensor, seed: int, offset: int = 0,
                            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Next token per row: argmax softmax(logits / T) / Exp(1) noise (Philox, seed/offset).

    logits [B, V] float32 with contiguous rows; temperatures [B] float32 > 0.
    Returns int32 [B].
    """
    lib = load()
    _dev(logits, "logits", torch.float32)
    _dev(temperatures, "temperatures", torch.float32)
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [B, V] with contiguous rows")
    B, V = (int(x) for x in logits.shape)
    if temperatures.shape != (B,) or not temperatures.is_contiguous():
        raise ValueError("temperatures must be contiguous [B]")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=logits.device)
    if workspace is None:
        workspace = torch.empty(max(256, int(lib.pkv_sample_workspace_bytes(B, V))), dtype=torch.uint8,
                                device=logits.device)
    _check("pkv_sample_exponential_race", lib.pkv_sample_exponential_race(
        logits.data_ptr(), logits.stride(0), temperatures.data_ptr(), B, V, int(seed) & (2**64 - 1),
        int(offset) & (2**64 - 1), out.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(logits)))
    return out


def device_error(clear: bool = True) -> list[str]:
    """Names of the device error bits set since the last clear (synchronises)."""
    lib = load()
    v = ctypes.c_uint32(0)
    _check("pkv_device_error", lib.pkv_device_error(ctypes.byref(v), 1 if clear else 0))
    return [name for bit, name in DEVERR.items() if v.value & bit]
