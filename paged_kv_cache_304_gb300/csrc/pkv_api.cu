// pkv_api.cu -- the C ABI declared in include/pkv.h: host-side argument
// validation, TMA tensor-map construction and kernel launch.  Nothing here
// allocates device memory or synchronises the host (pkv_device_error aside).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kDecodeTileTokens = 16;    // must match kT in decode.cu
constexpr int kPrefillTileTokens = 128;  // must match kTileN in prefill.cu
constexpr size_t kPrefillFusedWorkspaceBytes = 256;  // grid-barrier words of the fused-write prefill

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor maps over one layer's K and V caches, (num_blocks, 256, Hkv, 128)
// bf16, for tiles of `tile_tokens` consecutive tokens of one block and
// `heads_per_box` kv heads (all heads for decode, one for prefill).  The
// preferred map is 5-D over (dim within half, token, head, dim half, block)
// so that one copy brings the whole tile, laid out as
// [half][head][token][64 dims] with 128-byte swizzled rows.  If the driver
// refuses that stride order, a 3-D map over (dim, head, slot) is used and
// the kernel issues one copy per (half, head) into the same layout.
bool encode_cache_maps(const void* k_cache, const void* v_cache, int num_blocks, int hkv,
                       int tile_tokens, int heads_per_box, CacheMaps* maps) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(hkv) * kHeadDim * 2;  // bytes per token row
  {
    cuuint64_t dims[5] = {64, kBlockSize, static_cast<cuuint64_t>(hkv), 2, static_cast<cuuint64_t>(num_blocks)};
    cuuint64_t strides[4] = {row, kHeadDim * 2, 128, row * kBlockSize};
    cuuint32_t box[5] = {64, static_cast<cuuint32_t>(tile_tokens), static_cast<cuuint32_t>(heads_per_box), 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r1 = enc(&maps->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(k_cache), dims, strides,
                      box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = enc(&maps->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(v_cache), dims, strides,
                      box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 == CUDA_SUCCESS && r2 == CUDA_SUCCESS) {
      maps->per_head = 0;
      return true;
    }
  }
  cuuint64_t dims[3] = {kHeadDim, static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  cuuint64_t strides[2] = {kHeadDim * 2, row};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(tile_tokens)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r1 = enc(&maps->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k_cache), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  CUresult r2 = enc(&maps->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v_cache), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  maps->per_head = 1;
  return r1 == CUDA_SUCCESS && r2 == CUDA_SUCCESS;
}

// Shape checks shared by the two attention calls.
pkv_status check_attn_shape(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int32_t num_blocks, int32_t max_blocks_per_seq, float scale) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads) return PKV_ERR_SHAPE;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_SHAPE;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_kv_heads > kMaxKvHeads || num_q_heads > kMaxQHeads) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > kMaxGroup) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * kBlockSize >= (int64_t{1} << 31)) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: inconsistent or negative sizes";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: shape outside the supported set";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing or too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA call or kernel launch failed";
    case PKV_ERR_ALIGN: return "PKV_ERR_ALIGN: pointer or stride not 16-byte aligned";
    default: return "unknown pkv status";
  }
}

int pkv_version(void) { return 100; }

pkv_status pkv_kv_cache_write(const pkv_bf16* k, int64_t k_token_stride, const pkv_bf16* v, int64_t v_token_stride,
                       const int32_t* slot_mapping, int32_t num_tokens, pkv_bf16* k_cache, pkv_bf16* v_cache,
                       int32_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                       void* stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_SHAPE;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_token_stride < row || v_token_stride < row) return PKV_ERR_SHAPE;
  if (row % 8 || k_token_stride % 8 || v_token_stride % 8) return PKV_ERR_ALIGN;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  cudaError_t e = launch_kv_cache_write(k, k_token_stride, v, v_token_stride, slot_mapping, num_tokens, k_cache,
                                        v_cache, num_slots, static_cast<int32_t>(row),
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t max_context_len) {
  (void)max_context_len;  // the partials' size does not depend on the lengths
  if (batch < 0 || num_q_heads <= 0) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  return decode_workspace_bytes(batch, num_q_heads, sms);
}

}  // extern "C"

namespace {

// Shared by the plain and the fused-write decode entry points.
pkv_status decode_common(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache, const int32_t* context_lens,
                  const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t batch, int32_t num_q_heads,
                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                  int32_t max_context_len, float scale, pkv_bf16* out, void* workspace, size_t workspace_bytes,
                  void* stream, DecodeArgs& a) {
  if (batch < 0 || max_context_len < 0) return PKV_ERR_SHAPE;
  const pkv_status st = check_attn_shape(num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale);
  if (st != PKV_OK) return st;
  if (max_context_len >= (1 << 26)) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !context_lens || !block_tables || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
  const int sms = sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  if (!workspace || workspace_bytes < decode_workspace_bytes(batch, num_q_heads, sms)) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_ERR_ALIGN;
  CacheMaps maps;
  if (!encode_cache_maps(k_cache, v_cache, num_blocks, num_kv_heads, kDecodeTileTokens, num_kv_heads, &maps))
    return PKV_ERR_CUDA;
  a.q = q;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.out = out;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.num_blocks = num_blocks;
  a.max_context_len = max_context_len;
  a.scale = scale;
  a.workspace = workspace;
  cudaError_t e = launch_paged_attn_decode(a, maps, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Shared by the plain and the fused-write prefill entry points.
pkv_status prefill_common(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                           int32_t max_seqlen_k, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale, pkv_bf16* out, void* stream, PrefillArgs& a) {
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return PKV_ERR_SHAPE;
  const pkv_status st = check_attn_shape(num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale);
  if (st != PKV_OK) return st;
  if (max_seqlen_q > max_seqlen_k) return PKV_ERR_SHAPE;
  if (num_seqs > 65535 || max_seqlen_q > (1 << 22) || max_seqlen_k >= (1 << 26)) return PKV_ERR_UNSUPPORTED;
  if (total_q == 0 || num_seqs == 0 || max_seqlen_q == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !block_tables || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ALIGN;
  auto enc = encode_fn();
  if (!enc) return PKV_ERR_CUDA;
  CUtensorMap qmap;
  {
    // q [total_q, Hq, 128]: boxes of 128 rows x 64 dims of one head, swizzled.
    cuuint64_t dims[3] = {kHeadDim, static_cast<cuuint64_t>(num_q_heads), static_cast<cuuint64_t>(total_q)};
    cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(num_q_heads) * kHeadDim * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<pkv_bf16*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  }
  CUtensorMap omap;
  {
    // out, same layout as q: boxes of 32 rows (one warp's rows) x 64 dims of
    // one head, swizzled, for the bulk tensor stores of the epilogue.
    cuuint64_t dims[3] = {kHeadDim, static_cast<cuuint64_t>(num_q_heads), static_cast<cuuint64_t>(total_q)};
    cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(num_q_heads) * kHeadDim * 2};
    cuuint32_t box[3] = {64, 1, 32};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  }
  CacheMaps maps;
  if (!encode_cache_maps(k_cache, v_cache, num_blocks, num_kv_heads, kPrefillTileTokens, 1, &maps))
    return PKV_ERR_CUDA;
  a.q = q;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.block_tables = block_tables;
  a.out = out;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.num_blocks = num_blocks;
  a.scale = scale;
  cudaError_t e = launch_paged_attn_prefill(a, maps, qmap, omap, sm_count(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attn_decode(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                          const int32_t* context_lens, const int32_t* block_tables, int32_t max_blocks_per_seq,
                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                          pkv_bf16* out, void* workspace, size_t workspace_bytes, void* stream) {
  DecodeArgs a;
  return decode_common(q, k_cache, v_cache, context_lens, block_tables, max_blocks_per_seq, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, out, workspace,
                       workspace_bytes, stream, a);
}

pkv_status pkv_paged_attn_decode_fused_write(const pkv_bf16* q, const pkv_bf16* k_new, int64_t k_token_stride,
                                      const pkv_bf16* v_new, int64_t v_token_stride, const int32_t* slot_mapping,
                                      pkv_bf16* k_cache, pkv_bf16* v_cache, const int32_t* context_lens,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t batch,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                                      pkv_bf16* out, void* workspace, size_t workspace_bytes, void* stream) {
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (batch > 0) {
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_NULL;
    if (k_token_stride < row || v_token_stride < row) return PKV_ERR_SHAPE;
    if (k_token_stride % 8 || v_token_stride % 8 || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGN;
  }
  DecodeArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_stride = k_token_stride;
  a.v_stride = v_token_stride;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  return decode_common(q, k_cache, v_cache, context_lens, block_tables, max_blocks_per_seq, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, out, workspace,
                       workspace_bytes, stream, a);
}

pkv_status pkv_paged_attn_prefill(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
                                  int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  float scale, pkv_bf16* out, void* stream) {
  PrefillArgs a;
  return prefill_common(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, max_blocks_per_seq, num_seqs,
                        total_q, max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, scale, out, stream, a);
}

size_t pkv_prefill_fused_workspace_bytes(void) { return kPrefillFusedWorkspaceBytes; }

pkv_status pkv_paged_attn_prefill_fused_write(
    const pkv_bf16* q, const pkv_bf16* k_new, int64_t k_token_stride, const pkv_bf16* v_new, int64_t v_token_stride,
    const int32_t* slot_mapping, pkv_bf16* k_cache, pkv_bf16* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t num_seqs,
    int32_t total_q, int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale, pkv_bf16* out, void* workspace,
    size_t workspace_bytes, void* stream) {
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (total_q > 0 && num_seqs > 0) {
    if (!k_new || !v_new || !slot_mapping) return PKV_ERR_NULL;
    if (k_token_stride < row || v_token_stride < row) return PKV_ERR_SHAPE;
    if (k_token_stride % 8 || v_token_stride % 8 || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_ALIGN;
    if (!workspace || workspace_bytes < kPrefillFusedWorkspaceBytes) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return PKV_ERR_ALIGN;
  }
  PrefillArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_stride = k_token_stride;
  a.v_stride = v_token_stride;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.barrier_ws = static_cast<unsigned int*>(workspace);
  return prefill_common(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, max_blocks_per_seq, num_seqs,
                        total_q, max_seqlen_q, max_seqlen_k, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, scale, out, stream, a);
}

// ---------------------------------------------------------------------------
// Decode without caller scratch.  For callers that cannot allocate device
// memory (a plugin whose host engine owns all allocations, a C caller holding
// only the pointers it was given): the split-K partials go to one fixed
// library-owned array instead of a caller workspace.  Nothing here allocates.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace pkv {
namespace {

// Fixed scratch of the no-allocation decode call: one copy per GPU that loads
// the library, alive until the process exits.  Its name is only a host-side
// stand-in; kernels get the device address looked up below.
static __device__ __align__(256) uint8_t g_decode_static_scratch[PKV_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevicesCached = 64;
std::mutex g_static_scratch_mutex;
void* g_static_scratch_ptr[kMaxDevicesCached] = {};

// Device address of the fixed scratch on the current device, looked up once
// per device (with that device current) and cached.  nullptr on failure, and
// also when the lookup would have to happen while `stream` is being captured
// into a CUDA graph: the lookup may load the library's device code, which is
// not something to do inside a capture, so the first call on a device must
// come before any capture (the header says so).
void* static_scratch_for_current_device(cudaStream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesCached) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
  if (!g_static_scratch_ptr[dev]) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_static_scratch) != cudaSuccess) return nullptr;
    g_static_scratch_ptr[dev] = ptr;
  }
  return g_static_scratch_ptr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attn_decode_noalloc(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                                  const int32_t* context_lens, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, int32_t batch, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                  int32_t max_context_len, float scale, pkv_bf16* out, void* stream) {
  if (batch < 0 || max_context_len < 0) return PKV_ERR_SHAPE;
  const pkv_status st = check_attn_shape(num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale);
  if (st != PKV_OK) return st;
  if (max_context_len >= (1 << 26)) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  const int sms = sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  // Reject batches whose partials do not fit the fixed array, before launching.
  const size_t need = decode_workspace_bytes(batch, num_q_heads, sms);
  if (need > PKV_DECODE_STATIC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* scratch = static_scratch_for_current_device(static_cast<cudaStream_t>(stream));
  if (!scratch) return PKV_ERR_CUDA;
  // Nothing in the scratch must start at zero: every partial and every
  // per-sequence record the combine step reads is written earlier in the
  // same call.
  return pkv_paged_attn_decode(q, k_cache, v_cache, context_lens, block_tables, max_blocks_per_seq, batch,
                               num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale,
                               out, scratch, PKV_DECODE_STATIC_SCRATCH_BYTES, stream);
}

pkv_status pkv_prepare_metadata(const int32_t* block_ids, const int32_t* table_offsets, const int32_t* num_cached,
                         const int32_t* seq_lens, int32_t num_seqs, int32_t token_capacity,
                         int32_t max_blocks_per_seq, int32_t block_size, int32_t num_blocks, int32_t* cu_seqlens_q,
                         int32_t* cu_seqlens_k, int32_t* context_lens, int32_t* slot_mapping, int32_t* block_tables,
                         void* stream) {
  if (num_seqs < 0 || token_capacity < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
  if (block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * block_size >= (int64_t{1} << 31)) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!block_ids || !table_offsets || !num_cached || !seq_lens || !cu_seqlens_q || !cu_seqlens_k || !context_lens ||
      !block_tables || (token_capacity > 0 && !slot_mapping))
    return PKV_ERR_NULL;
  const int sms = sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  MetaArgs a;
  a.block_ids = block_ids;
  a.table_offsets = table_offsets;
  a.num_cached = num_cached;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.token_capacity = token_capacity;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.context_lens = context_lens;
  a.slot_mapping = slot_mapping;
  a.block_tables = block_tables;
  cudaError_t e = launch_prepare_metadata(a, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_sample_workspace_bytes(int32_t batch, int32_t vocab) {
  if (batch < 0 || vocab <= 0) return 0;
  return sample_workspace_bytes(batch, vocab);
}

pkv_status pkv_sample_exponential_race(const float* logits, int64_t row_stride, const float* temperatures, int32_t batch,
                                int32_t vocab, uint64_t seed, uint64_t offset, int32_t* out_tokens, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (batch < 0 || vocab <= 0 || row_stride < vocab) return PKV_ERR_SHAPE;
  if (batch == 0) return PKV_OK;
  if (static_cast<int64_t>(batch) * ((vocab + 4095) / 4096) >= (int64_t{1} << 31)) return PKV_ERR_UNSUPPORTED;
  if (!logits || !temperatures || !out_tokens) return PKV_ERR_NULL;
  if (!workspace || workspace_bytes < sample_workspace_bytes(batch, vocab)) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_ERR_ALIGN;
  SampleArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.temperatures = temperatures;
  a.batch = batch;
  a.vocab = vocab;
  a.seed = seed;
  a.offset = offset;
  a.out = out_tokens;
  a.workspace = workspace;
  cudaError_t e = launch_sample(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_device_error(uint32_t* out, int clear) {
  if (!out) return PKV_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  uint32_t a = 0, b = 0, c = 0, d = 0;
  if (read_error_kv_write(&a, clear != 0) != cudaSuccess) return PKV_ERR_CUDA;
  if (read_error_decode(&b, clear != 0) != cudaSuccess) return PKV_ERR_CUDA;
  if (read_error_prefill(&c, clear != 0) != cudaSuccess) return PKV_ERR_CUDA;
  if (read_error_metadata(&d, clear != 0) != cudaSuccess) return PKV_ERR_CUDA;
  uint32_t e5 = 0;
  if (read_error_sampler(&e5, clear != 0) != cudaSuccess) return PKV_ERR_CUDA;
  *out = a | b | c | d | e5;
  return PKV_OK;
}

}  // extern "C"
