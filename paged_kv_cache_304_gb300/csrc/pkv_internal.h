// pkv_internal.h -- launchers shared between the C-ABI front end (pkv_api.cu)
// and the kernel translation units.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <utility>

#include "pkv.h"

namespace pkv {

constexpr int kBlockSize = 256;
constexpr int kHeadDim = 128;
constexpr int kMaxKvHeads = 8;
constexpr int kMaxGroup = 16;
constexpr int kMaxQHeads = 64;

// Raise `kernel`'s dynamic shared-memory limit on the current device to at
// least `bytes`, calling the runtime only when the request exceeds what was
// already set on that device (`marks` holds one high-water mark per device,
// zero-initialised static storage of the caller).
constexpr int kMaxDevices = 64;
template <typename... KArgs>
cudaError_t ensure_dyn_smem(void (*kernel)(KArgs...), size_t bytes, std::atomic<int>* marks) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int want = static_cast<int>(bytes);
  if (dev >= 0 && dev < kMaxDevices && want <= marks[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
    int cur = marks[dev].load(std::memory_order_relaxed);
    while (cur < want && !marks[dev].compare_exchange_weak(cur, want, std::memory_order_release)) {
    }
  }
  return e;
}

// Launch `kernel` on `stream` with programmatic stream serialization
// allowed, so it may start while the previous kernel drains (each kernel
// calls griddepcontrol.wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- KV write
cudaError_t launch_kv_cache_write(const uint16_t* k, int64_t k_stride, const uint16_t* v,
                                  int64_t v_stride, const int32_t* slots, int32_t num_tokens,
                                  uint16_t* k_cache, uint16_t* v_cache, int64_t num_slots,
                                  int32_t row_elems, cudaStream_t stream);

// ---- decode
struct DecodeArgs {
  const uint16_t* q;
  const int32_t* context_lens;
  const int32_t* block_tables;
  uint16_t* out;
  int32_t max_blocks_per_seq;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_blocks;
  int32_t max_context_len;
  float scale;
  void* workspace;
  // Fused KV write (optional; all null for plain decode): each sequence's new
  // token row k_new[b] / v_new[b] (token strides in elements) is written to
  // k_cache / v_cache at slot_mapping[b] before it is read.
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
  int64_t k_stride = 0;
  int64_t v_stride = 0;
  const int32_t* slot_mapping = nullptr;
  uint16_t* k_cache = nullptr;
  uint16_t* v_cache = nullptr;
};
// Tensor maps over the caches, built by the front end (see pkv_api.cu).
// `per_head` selects the layout of the copy: one 5-D box per K (or V) tile,
// or 2 * num_kv_heads 3-D boxes with the same shared-memory image.
struct CacheMaps {
  CUtensorMap k;
  CUtensorMap v;
  int per_head;
};
size_t decode_workspace_bytes(int batch, int num_q_heads, int num_sms);
int decode_grid(int num_sms);
cudaError_t launch_paged_attn_decode(const DecodeArgs& a, const CacheMaps& maps, int num_sms,
                                     cudaStream_t stream);

// ---- prefill
struct PrefillArgs {
  const uint16_t* q;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  const int32_t* block_tables;
  uint16_t* out;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t num_blocks;
  float scale;
  // Fused KV write (optional; all null for plain prefill): token i's new row
  // k_new[i] / v_new[i] (token strides in elements) goes to k_cache / v_cache
  // at slot_mapping[i] before any cache read; barrier_ws is the caller's
  // two-word grid-barrier workspace.
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
  int64_t k_stride = 0;
  int64_t v_stride = 0;
  const int32_t* slot_mapping = nullptr;
  uint16_t* k_cache = nullptr;
  uint16_t* v_cache = nullptr;
  unsigned int* barrier_ws = nullptr;
};
// Stated max_seqlen_q up to which the persistent kernel is used (prefill.cu
// dispatches; prefill_persistent.cu holds that kernel).
constexpr int kPersistentMaxSeqlenQ = 2048;
cudaError_t launch_paged_attn_prefill(const PrefillArgs& a, const CacheMaps& kv_maps,
                                      const CUtensorMap& q_map, const CUtensorMap& out_map, int num_sms,
                                      cudaStream_t stream);
cudaError_t launch_prefill_persistent(const PrefillArgs& a, const CacheMaps& kv_maps, const CUtensorMap& q_map,
                                      const CUtensorMap& out_map, int num_sms, cudaStream_t stream);

// ---- step metadata
struct MetaArgs {
  const int32_t* block_ids;
  const int32_t* table_offsets;
  const int32_t* num_cached;
  const int32_t* seq_lens;
  int32_t num_seqs, token_capacity, max_blocks_per_seq, block_size, num_blocks;
  int32_t* cu_seqlens_q;
  int32_t* cu_seqlens_k;
  int32_t* context_lens;
  int32_t* slot_mapping;
  int32_t* block_tables;
};
cudaError_t launch_prepare_metadata(const MetaArgs& a, int num_sms, cudaStream_t stream);

// ---- exponential-race sampler
struct SampleArgs {
  const float* logits;
  int64_t row_stride;
  const float* temperatures;
  int32_t batch, vocab;
  uint64_t seed, offset;
  int32_t* out;
  void* workspace;
};
size_t sample_workspace_bytes(int batch, int vocab);
cudaError_t launch_sample(const SampleArgs& a, cudaStream_t stream);

// ---- device error words (one per translation unit)
cudaError_t read_error_kv_write(uint32_t* out, bool clear);
cudaError_t read_error_decode(uint32_t* out, bool clear);
cudaError_t read_error_prefill(uint32_t* out, bool clear);
cudaError_t read_error_prefill_persistent(uint32_t* out, bool clear);
cudaError_t read_error_metadata(uint32_t* out, bool clear);
cudaError_t read_error_sampler(uint32_t* out, bool clear);

}  // namespace pkv
