// kv_write.cu -- KV-cache write: scatter each scheduled token's K and V row
// into the paged cache at its slot, skipping slot -1 (CUDA-graph padding).
//
// Page "13. 读一个最小推理引擎：nano-vllm", section "第六站：注意力层": before
// attention, in prefill and decode alike, every scheduled token's K and V are
// copied into the paged cache; a slot of -1 is a padding row and is skipped.
//
// The work is a pure copy, bound by HBM: per token, 2 x row_bytes read and
// 2 x row_bytes written (row_bytes = num_kv_heads * head_dim * 2 = 2 KiB for
// 8 kv heads of 128).  One warp moves one token row: 128-bit loads (read-once,
// no L1 allocation) of up to four chunks of K and four of V per lane are all
// issued before the 128-bit stores, so each SM keeps many loads in flight.
// The grid is a multiple of the SM count and strides over the tokens.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_kv_write;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One warp per token row (grid-strided over tokens): the slot is read once
// per warp, then each lane loads its 16-byte chunks of the K row and of the V
// row -- up to four of each, all in flight together -- before storing them.
// Strides are in 16-byte chunks; `row_vecs` chunks make one row.
__global__ void __launch_bounds__(256) kv_write_kernel(const uint4* __restrict__ k, int64_t k_stride,
                                                       const uint4* __restrict__ v, int64_t v_stride,
                                                       const int32_t* __restrict__ slots,
                                                       int32_t num_tokens, uint4* __restrict__ k_cache,
                                                       uint4* __restrict__ v_cache, int64_t num_slots,
                                                       int32_t row_vecs) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < num_tokens;
       t += warps) {
    const int64_t s = __ldg(slots + t);
    if (s == -1) continue;
    if (s < 0 || s >= num_slots) {
      if (lane == 0) atomicOr(&g_err_kv_write, PKV_DEVERR_SLOT_RANGE);
      continue;
    }
    const uint4* ks = k + t * k_stride;
    const uint4* vs = v + t * v_stride;
    uint4* kd = k_cache + s * row_vecs;
    uint4* vd = v_cache + s * row_vecs;
    for (int c0 = 0; c0 < row_vecs; c0 += 128) {
      uint4 kr[4], vr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < row_vecs) {
          kr[u] = ld_stream(ks + c);
          vr[u] = ld_stream(vs + c);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < row_vecs) {
          kd[c] = kr[u];
          vd[c] = vr[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_cache_write(const uint16_t* k, int64_t k_stride, const uint16_t* v,
                                  int64_t v_stride, const int32_t* slots, int32_t num_tokens,
                                  uint16_t* k_cache, uint16_t* v_cache, int64_t num_slots,
                                  int32_t row_elems, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int32_t row_vecs = row_elems / 8;  // 8 bf16 per 16-byte chunk
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int threads = 256;  // 8 warps = 8 token rows per block and iteration
  int64_t blocks = (static_cast<int64_t>(num_tokens) + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  return launch_pdl(kv_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    reinterpret_cast<const uint4*>(k), k_stride / 8, reinterpret_cast<const uint4*>(v),
                    v_stride / 8, slots, num_tokens, reinterpret_cast<uint4*>(k_cache),
                    reinterpret_cast<uint4*>(v_cache), num_slots, row_vecs);
}

cudaError_t read_error_kv_write(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_kv_write, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_kv_write, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
