// prefill.cu -- varlen causal GQA prefill attention reading K/V from the paged
// cache through block tables, on the 5th-generation tensor cores (tcgen05).
//
// Page "13. 读一个最小推理引擎：nano-vllm": section "第二站：一个请求的状态" (each
// step computes from num_cached_tokens onward); "第三站：调度器" (only the
// first sequence of a step may be a split chunk); "第六站：注意力层" (with prefix
// hits or a chunk continuation the block table is passed so the whole context
// is read from the paged cache).  Query row j of sequence i sits at position
// c_i + j, c_i = L_i - n_i, and sees keys 0 .. c_i + j.
//
// Design (one CTA = one 128-row query tile of one query head):
// * warp 0, producer: TMA-loads the Q tile once, then streams the 128-token
//   K and V tiles of the kv head (two per 256-token cache block, looked up in
//   the block table) into 2-stage rings.  Tiles are stored as two 64-dim
//   halves of 128 rows x 128 bytes with the 128-byte swizzle.
// * warp 1, MMA: one thread issues tcgen05.mma (kind::f16, bf16 in, fp32
//   accumulate in tensor memory).  S_j = Q K_j^T goes to one of two TMEM
//   buffers (so S_{j+1} overlaps the softmax of S_j); O += P_j V_j
//   accumulates in a third TMEM region.  tcgen05.commit signals mbarriers.
// * warps 4-7, softmax: thread r owns query row r = TMEM lane r.  It loads its
//   128 scores with tcgen05.ld, applies the causal mask on diagonal tiles,
//   keeps a running row maximum (in log2 units, scale * log2(e) folded in)
//   and row sum, writes P in bf16 to shared memory in the layout the PV MMA
//   reads, and rescales O in TMEM only when its row maximum grew by more than
//   2^8 (otherwise the stale maximum stays the reference; p <= 256 then).
//   At the end it normalises O by the row sum and stores bf16 rows.
// * Tiles are launched heaviest first (the last query tile of a sequence
//   sees the most keys).
// Every wait is bounded (two seconds); on timeout the CTA flags
// PKV_DEVERR_WAIT_TIMEOUT, frees its tensor memory and returns.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_prefill;

constexpr int kTileM = 128;       // query rows per CTA
constexpr int kTileN = 128;       // keys per K/V tile
constexpr int kKvStages = 2;
constexpr int kThreads = 256;     // 8 warps: producer, MMA, 2 idle, 4 softmax
constexpr uint32_t kTileBytes = kTileN * kHeadDim * 2;  // 32 KiB: one Q, K, V or P tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;         // one 64-dim (or 64-key) half
constexpr uint32_t kTmemCols = 512;                     // S0 | S1 | O | unused
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kTileM, kTileN, 0);    // B = K, K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kTileM, kHeadDim, 1);  // B = V, N-major

struct PrefillParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* tables;
  uint16_t* out;
  int32_t maxb, S, Hq, Hkv, G, num_blocks, total_q, per_half;
  float sl2;  // scale * log2(e)
};

struct Smem {
  uint8_t* q;       // kTileBytes
  uint8_t* k0;      // kKvStages K tiles, kTileBytes apart
  uint8_t* v0;      // kKvStages V tiles, kTileBytes apart
  uint8_t* p;       // kTileBytes
  uint64_t* q_full;
  uint64_t* k_full;   // [kKvStages]
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;   // [2]
  uint64_t* s_empty;  // [2]
  uint64_t* p_full;
  uint64_t* o_done;
  uint32_t* tmem_base;
};

__device__ __forceinline__ Smem carve(uint8_t* base) {
  Smem s;
  uint8_t* c = base;
  s.q = c;
  c += kTileBytes;
  s.k0 = c;
  c += kKvStages * kTileBytes;
  s.v0 = c;
  c += kKvStages * kTileBytes;
  s.p = c;
  c += kTileBytes;
  uint64_t* b = reinterpret_cast<uint64_t*>(c);
  s.q_full = b;
  s.k_full = b + 1;
  s.k_empty = b + 1 + kKvStages;
  s.v_full = b + 1 + 2 * kKvStages;
  s.v_empty = b + 1 + 3 * kKvStages;
  s.s_full = b + 1 + 4 * kKvStages;
  s.s_empty = s.s_full + 2;
  s.p_full = s.s_empty + 2;
  s.o_done = s.p_full + 1;
  s.tmem_base = reinterpret_cast<uint32_t*>(s.o_done + 1);
  return s;
}

constexpr size_t kSmemBytes = 1024 + (2 + 2 * kKvStages) * kTileBytes + 32 * sizeof(uint64_t) + 16;

__device__ __forceinline__ int load_block(const PrefillParams& p, int seq, int lb) {
  int phys = __ldg(p.tables + static_cast<int64_t>(seq) * p.maxb + lb);
  if (phys < 0 || phys >= p.num_blocks) {
    atomicOr(&g_err_prefill, PKV_DEVERR_BLOCK_RANGE);
    phys = 0;
  }
  return phys;
}

// Load one 128-token K or V tile (all 128 dims of kv head g) into `dst` as two
// swizzled 64-dim halves.
__device__ __forceinline__ void load_kv_tile(const PrefillParams& p, const CUtensorMap* map, uint8_t* dst,
                                             uint64_t* bar, int phys, int tin, int g) {
  if (!p.per_half) {
    tma_load_5d(dst, map, bar, 0, tin, g, 0, phys);
  } else {
    const int slot = phys * kBlockSize + tin;
    tma_load_3d(dst, map, bar, 0, g, slot);
    tma_load_3d(dst + kHalfBytes, map, bar, 64, g, slot);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int h = blockIdx.x;    // query head
  const int seq = blockIdx.y;  // sequence
  const int q0 = __ldg(p.cu_q + seq), q1 = __ldg(p.cu_q + seq + 1);
  const int k0 = __ldg(p.cu_k + seq), k1 = __ldg(p.cu_k + seq + 1);
  const int n = q1 - q0, L = k1 - k0;
  const int c = L - n;
  if (n <= 0) return;
  if (c < 0 || L > p.maxb * kBlockSize || q1 > p.total_q || q0 < 0) {
    if (threadIdx.x == 0) atomicOr(&g_err_prefill, PKV_DEVERR_LEN_RANGE);
    return;
  }
  const int ntiles = (n + kTileM - 1) / kTileM;
  if (ntiles > static_cast<int>(gridDim.z) && blockIdx.z == 0 && threadIdx.x == 0)
    atomicOr(&g_err_prefill, PKV_DEVERR_LEN_RANGE);  // n exceeds the stated max_seqlen_q
  if (static_cast<int>(blockIdx.z) >= ntiles) return;
  const int m = ntiles - 1 - static_cast<int>(blockIdx.z);  // heaviest tile first
  const int g = h / p.G;
  const int row_end = min(kTileM * (m + 1), n);              // exclusive, tile-local rows < row_end - 128m
  const int kv_end = c + row_end;                            // keys 0 .. kv_end-1 are visible to some row
  const int nkv = (kv_end + kTileN - 1) / kTileN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  const Smem sm = carve(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(sm.q_full, 1);
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_empty[i], 4);
    }
    mbar_init(sm.p_full, 4);
    mbar_init(sm.o_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::alloc(sm.tmem_base, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *sm.tmem_base;
  const uint32_t tmem_s0 = tmem, tmem_s1 = tmem + 128, tmem_o = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      mbar_arrive_expect_tx(sm.q_full, kTileBytes);
      const int row0 = q0 + kTileM * m;
      tma_load_3d(sm.q, &qmap, sm.q_full, 0, h, row0);
      tma_load_3d(sm.q + kHalfBytes, &qmap, sm.q_full, 64, h, row0);
      int phys = load_block(p, seq, 0);
      int nxt = nkv > 2 ? load_block(p, seq, 1) : 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % kKvStages;
        const uint32_t par = ((j / kKvStages) & 1) ^ 1;
        if ((j & 1) == 0 && j > 0) {
          phys = nxt;
          if (2 * (j / 2 + 1) < nkv) nxt = load_block(p, seq, j / 2 + 1);
        }
        const int tin = (j & 1) * kTileN;
        if (!mbar_wait(&sm.k_empty[st], par, &g_err_prefill)) break;
        mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
        load_kv_tile(p, &kmap, (sm.k0 + st * kTileBytes), &sm.k_full[st], phys, tin, g);
        if (!mbar_wait(&sm.v_empty[st], par, &g_err_prefill)) break;
        mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
        load_kv_tile(p, &vmap, (sm.v0 + st * kTileBytes), &sm.v_full[st], phys, tin, g);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t qa = smem_u32(sm.q), pa = smem_u32(sm.p);
      bool ok = mbar_wait(sm.q_full, 0, &g_err_prefill);
      auto issue_s = [&](int j) -> bool {
        const int st = j % kKvStages, sb = j & 1;
        if (!mbar_wait(&sm.k_full[st], (j / kKvStages) & 1, &g_err_prefill)) return false;
        if (!mbar_wait(&sm.s_empty[sb], ((j >> 1) & 1) ^ 1, &g_err_prefill)) return false;
        tc::fence_after();
        const uint32_t ka = smem_u32((sm.k0 + st * kTileBytes));
        const uint32_t d = sb ? tmem_s1 : tmem_s0;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          tc::mma_ss(d, tc::smem_desc_sw128(qa + off, 16, 1024), tc::smem_desc_sw128(ka + off, 16, 1024), kIdescS,
                     kk > 0);
        }
        tc::commit(&sm.s_full[sb]);
        tc::commit(&sm.k_empty[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkv && ok; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) break;
        const int st = j % kKvStages;
        if (!mbar_wait(sm.p_full, j & 1, &g_err_prefill)) break;
        if (!mbar_wait(&sm.v_full[st], (j / kKvStages) & 1, &g_err_prefill)) break;
        tc::fence_after();
        const uint32_t va = smem_u32((sm.v0 + st * kTileBytes));
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          // A = P (rows x keys, keys contiguous); B = V (keys x dims, dims contiguous):
          // 64-dim halves are 16 KiB apart (leading offset), 8-key groups 1 KiB apart.
          const uint32_t aoff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          tc::mma_ss(tmem_o, tc::smem_desc_sw128(pa + aoff, 16, 1024),
                     tc::smem_desc_sw128(va + kk * 2048, kHalfBytes, 1024), kIdescPV, (j > 0 || kk > 0));
        }
        tc::commit(sm.o_done);
        tc::commit(&sm.v_empty[st]);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                 // tile row = TMEM lane
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const int lim_row = c + kTileM * m + r;        // last visible key of this row
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    const uint32_t prow = smem_u32(sm.p) + r * 128;
    for (int j = 0; j < nkv && ok; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&sm.s_full[sb], (j >> 1) & 1, &g_err_prefill)) {
        ok = false;
        break;
      }
      tc::fence_after();
      float s[128];
      const uint32_t sa = (sb ? tmem_s1 : tmem_s0) + lane_bits;
      tc::ld32(sa + 0, s + 0);
      tc::ld32(sa + 32, s + 32);
      tc::ld32(sa + 64, s + 64);
      tc::ld32(sa + 96, s + 96);
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_empty[sb]);
      // causal mask: key 128 j + x visible iff x <= lim
      const int lim = lim_row - kTileN * j;
      if (lim < kTileN - 1) {
#pragma unroll
        for (int x = 0; x < 128; ++x)
          if (x > lim) s[x] = -INFINITY;
      }
      float mt = s[0];
#pragma unroll
      for (int x = 1; x < 128; ++x) mt = fmaxf(mt, s[x]);
      const float m_new = fmaxf(m_ref, mt * p.sl2);
      float alpha = 1.f;
      if (m_new > m_ref + 8.f) {
        alpha = fast_exp2(m_ref - m_new);  // 0 on the first tile (m_ref = -inf)
        m_ref = m_new;
      }
      const float mu = m_ref;  // finite: key 0 is visible to every row
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int x = 0; x < 128; x += 2) {
        const float e0 = fast_exp2(fmaf(s[x], p.sl2, -mu));
        const float e1 = fast_exp2(fmaf(s[x + 1], p.sl2, -mu));
        rs += e0 + e1;
        pk[x >> 1] = pack_bf16x2(e0, e1);
      }
      l = l * alpha + rs;
      // PV_{j-1} must be done before O is rescaled and before P is overwritten.
      if (j > 0) {
        if (!mbar_wait(sm.o_done, (j - 1) & 1, &g_err_prefill)) {
          ok = false;
          break;
        }
        tc::fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t oa = tmem_o + lane_bits;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            float o[32];
            tc::ld32(oa + cc * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            tc::st32(oa + cc * 32, o);
          }
          tc::wait_st();
        }
      }
      // P row r: keys 0-63 in the first half, 64-127 in the second; 16-byte
      // chunk q of a 128-byte row is stored at chunk q ^ (r & 7).
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint32_t addr = prow + (q >> 3) * kHalfBytes + ((((q & 7) ^ (r & 7))) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]), "r"(pk[4 * q + 1]),
                     "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full);
    }
    if (ok && mbar_wait(sm.o_done, (nkv - 1) & 1, &g_err_prefill)) {
      tc::fence_after();
      const float inv = 1.f / l;
      const int row = kTileM * m + r;
      uint16_t* dst = p.out + (static_cast<int64_t>(q0 + row) * p.Hq + h) * kHeadDim;
      const uint32_t oa = tmem_o + lane_bits;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float o[32];
        tc::ld32(oa + cc * 32, o);
        tc::wait_ld();
        if (row < n) {
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 v;
            v.x = pack_bf16x2(o[x] * inv, o[x + 1] * inv);
            v.y = pack_bf16x2(o[x + 2] * inv, o[x + 3] * inv);
            v.z = pack_bf16x2(o[x + 4] * inv, o[x + 5] * inv);
            v.w = pack_bf16x2(o[x + 6] * inv, o[x + 7] * inv);
            *reinterpret_cast<uint4*>(dst + cc * 32 + x) = v;
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_paged_attn_prefill(const PrefillArgs& a, const CacheMaps& kv, const CUtensorMap& qmap,
                                      int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (a.total_q == 0 || a.num_seqs == 0) return cudaSuccess;
  PrefillParams p;
  p.cu_q = a.cu_seqlens_q;
  p.cu_k = a.cu_seqlens_k;
  p.tables = a.block_tables;
  p.out = a.out;
  p.maxb = a.max_blocks_per_seq;
  p.S = a.num_seqs;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.G = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.total_q = a.total_q;
  p.per_half = kv.per_head;
  p.sl2 = a.scale * 1.4426950408889634f;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int max_tiles = (a.max_seqlen_q + kTileM - 1) / kTileM;
  dim3 grid(a.num_q_heads, a.num_seqs, max_tiles);
  return launch_pdl(prefill_kernel, grid, dim3(kThreads), kSmemBytes, stream, qmap, kv.k, kv.v, p);
}

cudaError_t read_error_prefill(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_prefill, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_prefill, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
