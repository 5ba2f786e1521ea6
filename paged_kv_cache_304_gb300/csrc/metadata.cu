// metadata.cu -- device-side preparation of the step metadata of the paged-KV
// path: cumulative sequence lengths, context lengths, packed block tables and
// the slot of every new token.
//
// Page "13. 读一个最小推理引擎：nano-vllm": "第二站：一个请求的状态" (every
// step computes from num_cached_tokens onward); "第五站：执行准备与 KV 容量"
// (prepare_prefill / prepare_decode build the slot mapping with
// slot = block_table[p / block_size] * block_size + p % block_size, and a
// prefill feeds only the tokens from num_cached_tokens on); "第六站：注意力层"
// (the varlen calls take cumulative lengths).
//
// Up to 16384 sequences, one kernel does both steps (each CTA scans the
// lengths itself); larger batches use two kernels, chained with
// programmatic dependent launch:
// * scan (one CTA): per sequence n_i = L_i - c_i new tokens; block-wide
//   inclusive scans give cu_seqlens_q and cu_seqlens_k; context_lens = L.
//   A sequence whose table is too short for L_i (the decode rule: a token at
//   position L-1 with L % block_size == 1 needs a fresh block) or whose
//   lengths are inconsistent is flagged and contributes no tokens; one with
//   no tokens at all (num_cached = L = 0) is a CUDA-graph pad row and
//   contributes none without a flag.
// * fill (grid): thread t < token capacity finds its sequence by binary search
//   in cu_seqlens_q and writes its slot (or -1 past the last real token, the
//   CUDA-graph padding value); thread e < S * max_blocks writes one entry of
//   the packed block tables (-1 past the sequence's blocks).
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_metadata;

constexpr int kScanThreads = 1024;

struct MetaParams {
  const int32_t* block_ids;      // concatenated block tables
  const int32_t* table_offsets;  // [S+1]
  const int32_t* num_cached;     // [S]
  const int32_t* seq_lens;       // [S]
  int32_t S, token_capacity, max_blocks, block_size, num_blocks;
  int32_t* cu_q;        // [S+1]
  int32_t* cu_k;        // [S+1]
  int32_t* ctx;         // [S]
  int32_t* slots;       // [token_capacity]
  int32_t* tables;      // [S, max_blocks]
};

// n_i and L_i of sequence i, or (0, 0) (flagged) if its inputs are
// inconsistent.  A sequence with num_cached == seq_len == 0 is a CUDA-graph
// pad row: it contributes no tokens and context length 0, unflagged.
__device__ __forceinline__ void seq_counts(const MetaParams& p, int i, int& n, int& L) {
  const int c = __ldg(p.num_cached + i);
  L = __ldg(p.seq_lens + i);
  const int nb = __ldg(p.table_offsets + i + 1) - __ldg(p.table_offsets + i);
  if (c == 0 && L == 0 && nb >= 0 && nb <= p.max_blocks) {
    n = 0;
    return;
  }
  if (c < 0 || L <= c || nb < 0 || nb > p.max_blocks || static_cast<int64_t>(nb) * p.block_size < L) {
    atomicOr(&g_err_metadata, PKV_DEVERR_LEN_RANGE);
    n = 0;
    L = 0;
    return;
  }
  n = L - c;
}

__global__ void __launch_bounds__(kScanThreads) metadata_scan_kernel(const MetaParams p) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int warp_n[32], warp_l[32];
  __shared__ int carry_n, carry_l;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) {
    carry_n = carry_l = 0;
    p.cu_q[0] = 0;
    p.cu_k[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.S; base += kScanThreads) {
    const int i = base + tid;
    int n = 0, L = 0;
    if (i < p.S) seq_counts(p, i, n, L);
    int sn = n, sl = L;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yn = __shfl_up_sync(0xffffffffu, sn, o), yl = __shfl_up_sync(0xffffffffu, sl, o);
      if (lane >= o) {
        sn += yn;
        sl += yl;
      }
    }
    if (lane == 31) {
      warp_n[wid] = sn;
      warp_l[wid] = sl;
    }
    __syncthreads();
    if (wid == 0) {
      int wn = warp_n[lane], wl = warp_l[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yn = __shfl_up_sync(0xffffffffu, wn, o), yl = __shfl_up_sync(0xffffffffu, wl, o);
        if (lane >= o) {
          wn += yn;
          wl += yl;
        }
      }
      warp_n[lane] = wn;
      warp_l[lane] = wl;
    }
    __syncthreads();
    const int off_n = carry_n + (wid ? warp_n[wid - 1] : 0);
    const int off_l = carry_l + (wid ? warp_l[wid - 1] : 0);
    if (i < p.S) {
      p.cu_q[i + 1] = off_n + sn;
      p.cu_k[i + 1] = off_l + sl;
      p.ctx[i] = L;
    }
    __syncthreads();
    if (tid == kScanThreads - 1) {
      carry_n = off_n + sn;
      carry_l = off_l + sl;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) metadata_fill_kernel(const MetaParams p) {
  griddep_wait();  // needs cu_seqlens_q from the scan kernel
  griddep_launch_dependents();
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int total = p.cu_q[p.S];
  if (t0 == 0 && total > p.token_capacity) atomicOr(&g_err_metadata, PKV_DEVERR_LEN_RANGE);
  for (int64_t t = t0; t < p.token_capacity; t += nthreads) {
    if (t >= total) {
      p.slots[t] = -1;
      continue;
    }
    int lo = 0, hi = p.S;  // find i with cu_q[i] <= t < cu_q[i+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu_q[mid] <= t) lo = mid; else hi = mid;
    }
    const int i = lo;
    const int c = __ldg(p.num_cached + i);
    const int pos = c + static_cast<int>(t - p.cu_q[i]);
    const int off = __ldg(p.table_offsets + i);
    const int blk = __ldg(p.block_ids + off + pos / p.block_size);
    if (blk < 0 || blk >= p.num_blocks) {
      atomicOr(&g_err_metadata, PKV_DEVERR_BLOCK_RANGE);
      p.slots[t] = -1;
      continue;
    }
    p.slots[t] = blk * p.block_size + pos % p.block_size;
  }
  const int64_t entries = static_cast<int64_t>(p.S) * p.max_blocks;
  for (int64_t e = t0; e < entries; e += nthreads) {
    const int i = static_cast<int>(e / p.max_blocks);
    const int k = static_cast<int>(e - static_cast<int64_t>(i) * p.max_blocks);
    const int off = __ldg(p.table_offsets + i);
    const int nb = __ldg(p.table_offsets + i + 1) - off;
    p.tables[e] = k < nb ? __ldg(p.block_ids + off + k) : -1;
  }
}

// One kernel for batches of up to kFusedMaxSeqs sequences: every CTA scans
// the lengths itself (into shared memory) and then fills its share of the
// slots and table entries, so no second launch waits on a first.  CTA 0
// writes the scanned arrays.
constexpr int kFusedThreads = 256;
constexpr int kFusedMaxSeqs = 16384;

__global__ void __launch_bounds__(kFusedThreads) metadata_fused_kernel(const MetaParams p) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int cu_s[];  // [S + 1] cu_seqlens_q
  __shared__ int warp_n[kFusedThreads / 32], warp_l[kFusedThreads / 32];
  __shared__ int carry_n, carry_l;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool writer = blockIdx.x == 0;
  if (tid == 0) {
    carry_n = carry_l = 0;
    cu_s[0] = 0;
    if (writer) {
      p.cu_q[0] = 0;
      p.cu_k[0] = 0;
    }
  }
  __syncthreads();
  for (int base = 0; base < p.S; base += kFusedThreads) {
    const int i = base + tid;
    int n = 0, L = 0;
    if (i < p.S) seq_counts(p, i, n, L);
    int sn = n, sl = L;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yn = __shfl_up_sync(0xffffffffu, sn, o), yl = __shfl_up_sync(0xffffffffu, sl, o);
      if (lane >= o) {
        sn += yn;
        sl += yl;
      }
    }
    if (lane == 31) {
      warp_n[wid] = sn;
      warp_l[wid] = sl;
    }
    __syncthreads();
    if (wid == 0) {
      constexpr int kWarps = kFusedThreads / 32;
      int wn = lane < kWarps ? warp_n[lane] : 0, wl = lane < kWarps ? warp_l[lane] : 0;
#pragma unroll
      for (int o = 1; o < kWarps; o <<= 1) {
        const int yn = __shfl_up_sync(0xffffffffu, wn, o), yl = __shfl_up_sync(0xffffffffu, wl, o);
        if (lane >= o) {
          wn += yn;
          wl += yl;
        }
      }
      if (lane < kWarps) {
        warp_n[lane] = wn;
        warp_l[lane] = wl;
      }
    }
    __syncthreads();
    const int off_n = carry_n + (wid ? warp_n[wid - 1] : 0);
    const int off_l = carry_l + (wid ? warp_l[wid - 1] : 0);
    if (i < p.S) {
      cu_s[i + 1] = off_n + sn;
      if (writer) {
        p.cu_q[i + 1] = off_n + sn;
        p.cu_k[i + 1] = off_l + sl;
        p.ctx[i] = L;
      }
    }
    __syncthreads();
    if (tid == kFusedThreads - 1) {
      carry_n = off_n + sn;
      carry_l = off_l + sl;
    }
    __syncthreads();
  }
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int total = cu_s[p.S];
  if (t0 == 0 && total > p.token_capacity) atomicOr(&g_err_metadata, PKV_DEVERR_LEN_RANGE);
  for (int64_t t = t0; t < p.token_capacity; t += nthreads) {
    if (t >= total) {
      p.slots[t] = -1;
      continue;
    }
    int lo = 0, hi = p.S;  // find i with cu[i] <= t < cu[i+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu_s[mid] <= t) lo = mid; else hi = mid;
    }
    const int i = lo;
    const int c = __ldg(p.num_cached + i);
    const int pos = c + static_cast<int>(t - cu_s[i]);
    const int off = __ldg(p.table_offsets + i);
    const int blk = __ldg(p.block_ids + off + pos / p.block_size);
    if (blk < 0 || blk >= p.num_blocks) {
      atomicOr(&g_err_metadata, PKV_DEVERR_BLOCK_RANGE);
      p.slots[t] = -1;
      continue;
    }
    p.slots[t] = blk * p.block_size + pos % p.block_size;
  }
  const int64_t entries = static_cast<int64_t>(p.S) * p.max_blocks;
  for (int64_t e = t0; e < entries; e += nthreads) {
    const int i = static_cast<int>(e / p.max_blocks);
    const int k = static_cast<int>(e - static_cast<int64_t>(i) * p.max_blocks);
    const int off = __ldg(p.table_offsets + i);
    const int nb = __ldg(p.table_offsets + i + 1) - off;
    p.tables[e] = k < nb ? __ldg(p.block_ids + off + k) : -1;
  }
}

}  // namespace

cudaError_t launch_prepare_metadata(const MetaArgs& a, int num_sms, cudaStream_t stream) {
  MetaParams p;
  p.block_ids = a.block_ids;
  p.table_offsets = a.table_offsets;
  p.num_cached = a.num_cached;
  p.seq_lens = a.seq_lens;
  p.S = a.num_seqs;
  p.token_capacity = a.token_capacity;
  p.max_blocks = a.max_blocks_per_seq;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.cu_q = a.cu_seqlens_q;
  p.cu_k = a.cu_seqlens_k;
  p.ctx = a.context_lens;
  p.slots = a.slot_mapping;
  p.tables = a.block_tables;
  const int64_t work = std::max<int64_t>(a.token_capacity, static_cast<int64_t>(a.num_seqs) * a.max_blocks_per_seq);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (a.num_seqs <= kFusedMaxSeqs) {
    const size_t smem = (static_cast<size_t>(a.num_seqs) + 1) * sizeof(int);
    if (smem > 48 * 1024) {
      static std::atomic<int> smem_set[kMaxDevices];
      cudaError_t e = ensure_dyn_smem(metadata_fused_kernel, smem, smem_set);
      if (e != cudaSuccess) return e;
    }
    return launch_pdl(metadata_fused_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kFusedThreads), smem, stream,
                      p);
  }
  cudaError_t e = launch_pdl(metadata_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(metadata_fill_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
}

cudaError_t read_error_metadata(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_metadata, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_metadata, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
