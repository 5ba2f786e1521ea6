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
// Design.  One CTA = one 128-row query tile of one sequence for TWO query
// heads of the same kv group ("slots" A and B): both read the same K/V tiles
// under the same causal mask, so every K/V byte brought into shared memory
// feeds twice the tensor work, and the two slots ping-pong so the tensor
// pipe always has one slot's work while the other slot's softmax runs.
// * warp 0, producer: TMA-loads the two Q tiles, then streams the kv head's
//   128-token K and V tiles (two per 256-token cache block, looked up in the
//   block table) into rings of three K and two V stages, as 64-dim halves
//   of 128 rows x 128 bytes with the 128-byte swizzle.
// * warps 1 (slot A) and 10 (slot B), MMA: one thread per slot issues
//   tcgen05.mma (kind::f16, bf16 in, fp32 accumulate); an issuing thread
//   stays blocked while its instructions queue behind the tensor pipe, so
//   one issuer per slot lets one slot's waits overlap the other's MMAs.
//   Tensor memory holds S (128 columns, shared by the slots), P_A | P_B (64
//   columns each, packed bf16) and O_A | O_B (128 each).  The S columns are
//   handed from slot to slot, S_A(0), S_B(0), S_A(1), ..., each S issued as
//   soon as the previous one has been read into registers, so the next
//   tile's S never waits for this tile's P V.  Matrix descriptors are built
//   once; a k-step adds a constant.
// * warps 2-5 (slot A) and 6-9 (slot B), softmax: warp w reads TMEM lanes
//   32 (w % 4) .. +31, so thread r of a group owns query row r (TMEM lane
//   r).  It loads its 128 scores with tcgen05.ld, releases the S columns,
//   applies the causal mask on diagonal tiles, keeps the running row maximum
//   (log2 units, scale * log2(e) folded in), computes the first 64
//   probabilities, waits for the previous P V of its slot, stores them and
//   the other 64, and rescales O in tensor memory only when the maximum grew
//   by more than 2^8.  At the end it normalises O by the row sum
//   and stages the bf16 rows in the Q buffer in the layout of a TMA box; a
//   warp whose 32 rows all belong to the sequence stores them with bulk
//   tensor copies, a warp holding the sequence's end writes its rows with
//   ordinary stores.
// * Q and the first K tile are requested right after the barriers are set
//   up, before the tensor-memory allocation and the block-wide barrier, in
//   the order Q_A, K(0), Q_B with one Q barrier per slot, so slot A's first
//   S waits for two tiles, not three; the first block-table entries are
//   range-checked only after Q has been requested.
// * Tiles are launched heaviest first (the last query tile of a sequence
//   sees the most keys); the hardware block scheduler balances the rest.
// Every wait is bounded (two seconds); on timeout the CTA flags
// PKV_DEVERR_WAIT_TIMEOUT, lets the copies and MMAs it has already issued
// complete (bounded waits on their barriers), frees its tensor memory and
// returns.
//
// This grid form is used for long prompts (stated max_seqlen_q above 2048),
// also after the KV write kernel when the call has the write fused in;
// batches of short query tiles go to the persistent kernel in
// prefill_persistent.cu, which computes the same tiles in the same order.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_prefill;

constexpr int kTileM = 128;    // query rows per slot
constexpr int kTileN = 128;    // keys per K/V tile
constexpr int kKStages = 3;  // K tiles in flight: K(j+3) loads once S(j) of both slots is done
constexpr int kVStages = 2;  // V tiles in flight
constexpr int kThreads = 352;  // 11 warps: producer, MMA A, 4 softmax A, 4 softmax B, MMA B
constexpr uint32_t kTileBytes = kTileN * kHeadDim * 2;  // 32 KiB: one Q, K or V tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;         // one 64-dim half
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kTileM, kTileN, 0);    // B = K tile, K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kTileM, kHeadDim, 1);  // B = V tile, N-major

struct PrefillParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* tables;
  uint16_t* out;
  int32_t maxb, S, Hq, Hkv, G, npairs, num_blocks, total_q, per_half;
  float sl2;  // scale * log2(e)
};

// Shared memory: Q_A | Q_B | K stages | V stages | barriers.
struct Smem {
  uint8_t* q;   // 2 tiles
  uint8_t* k0;  // kKStages tiles
  uint8_t* v0;  // kVStages tiles
  uint64_t* q_full;   // [2 slots]
  uint64_t* k_full;   // [kKStages]
  uint64_t* k_empty;  // [kKStages]
  uint64_t* v_full;   // [kVStages]
  uint64_t* v_empty;  // [kVStages]
  uint64_t* s_full;   // [2 slots]: S of this slot computed
  uint64_t* s_free;   // [2 slots]: the shared S columns may take this slot's next S
  uint64_t* p_full;   // [2 slots]: P of this slot stored
  uint64_t* pv_done;  // [2 slots]: P V of this slot completed (P columns and O reusable)
  uint64_t* o_done;   // [2 slots]
  uint64_t* drain;    // [2 slots]: every MMA of the slot's issuer completed (abort path)
  uint32_t* tmem_base;
};

__device__ __forceinline__ Smem carve(uint8_t* base) {
  Smem s;
  s.q = base;
  s.k0 = base + 2 * kTileBytes;
  s.v0 = s.k0 + kKStages * kTileBytes;
  uint64_t* b = reinterpret_cast<uint64_t*>(s.v0 + kVStages * kTileBytes);
  s.q_full = b;
  s.k_full = b + 2;
  s.k_empty = s.k_full + kKStages;
  s.v_full = s.k_empty + kKStages;
  s.v_empty = s.v_full + kVStages;
  s.s_full = s.v_empty + kVStages;
  s.s_free = s.s_full + 2;
  s.p_full = s.s_free + 2;
  s.pv_done = s.p_full + 2;
  s.o_done = s.pv_done + 2;
  s.drain = s.o_done + 2;
  s.tmem_base = reinterpret_cast<uint32_t*>(s.drain + 2);
  return s;
}

constexpr size_t kSmemBytes = 1024 + (2 + kKStages + kVStages) * kTileBytes + 32 * sizeof(uint64_t) + 16;
static_assert(kSmemBytes <= 232448, "shared memory per block");

// Wait used only after a timeout, to let work this CTA already issued (bulk
// copies, MMAs) finish before its shared and tensor memory are given up:
// bounded (100 ms), reports nothing (the timeout has been reported).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 100000000ull) return;
}

__device__ __forceinline__ int checked_block(const PrefillParams& p, int phys) {
  if (phys < 0 || phys >= p.num_blocks) {
    atomicOr(&g_err_prefill, PKV_DEVERR_BLOCK_RANGE);
    phys = 0;
  }
  return phys;
}

__device__ __forceinline__ int load_block(const PrefillParams& p, int seq, int lb) {
  return checked_block(p, __ldg(p.tables + static_cast<int64_t>(seq) * p.maxb + lb));
}

// One 128-token K or V tile (all 128 dims of kv head g) into `dst` as two
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

// Matrix descriptors are built once per CTA; a k-step only adds a constant to
// the 16-byte address field in the low bits (the addresses stay below
// 256 KiB, so the add never carries out of the field, nor out of the low
// word: one 32-bit add, the high word kept as it is).  Rebuilding the 64-bit
// descriptor for every instruction made the single issuing thread, not the
// tensor pipe, the limit.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) {
  return (d & 0xFFFFFFFF00000000ull) | static_cast<uint32_t>(static_cast<uint32_t>(d) + (bytes >> 4));
}

// Bulk tensor store of one box from shared memory, tracked by the bulk
// async-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// S = Q K^T: A = Q tile, B = K tile, both K-major (dims contiguous) with the
// 128-byte swizzle; k-step kk selects 32 bytes of a 64-dim half.
__device__ __forceinline__ void issue_s(uint32_t d, uint64_t qdesc, uint64_t kdesc) {
#pragma unroll
  for (int kk = 0; kk < kHeadDim / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    tc::mma_ss(d, desc_add(qdesc, off), desc_add(kdesc, off), kIdescS, kk > 0);
  }
}

// O += P V with P (128 x 128 keys, packed bf16) in tensor memory at `p_tmem`
// and V (keys x dims, dims contiguous) in shared memory: 64-dim halves are
// 16 KiB apart (leading offset), 8-key groups 1 KiB apart (stride offset).
__device__ __forceinline__ void issue_pv(uint32_t o, uint32_t p_tmem, uint64_t vdesc, bool acc) {
#pragma unroll
  for (int kk = 0; kk < kTileN / 16; ++kk)
    tc::mma_ts(o, p_tmem + kk * 8, desc_add(vdesc, kk * 2048), kIdescPV, (acc || kk > 0) ? 1u : 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                   const PrefillParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.x / p.npairs;   // kv head
  const int pair = blockIdx.x - g * p.npairs;
  const int hA = g * p.G + 2 * pair;      // query head of slot A
  const bool has_b = 2 * pair + 1 < p.G;  // slot B: query head hA + 1
  const int seq = blockIdx.y;
  const int q0 = __ldg(p.cu_q + seq), q1 = __ldg(p.cu_q + seq + 1);
  const int k0 = __ldg(p.cu_k + seq), k1 = __ldg(p.cu_k + seq + 1);
  const int n = q1 - q0, L = k1 - k0;
  const int c = L - n;
  if (n <= 0) return;
  if (c < 0 || L > p.maxb * kBlockSize || q1 > p.total_q || q0 < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_err_prefill, PKV_DEVERR_LEN_RANGE);
    return;
  }
  const int ntiles = (n + kTileM - 1) / kTileM;
  if (ntiles > static_cast<int>(gridDim.z) && blockIdx.z == 0 && threadIdx.x == 0)
    atomicOr(&g_err_prefill, PKV_DEVERR_LEN_RANGE);  // n exceeds the stated max_seqlen_q
  if (static_cast<int>(blockIdx.z) >= ntiles) return;
  const int m = ntiles - 1 - static_cast<int>(blockIdx.z);  // heaviest tile first
  const int row_end = min(kTileM * (m + 1), n);
  const int kv_end = c + row_end;  // keys 0 .. kv_end-1 are visible to some row
  const int nkv = (kv_end + kTileN - 1) / kTileN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  const Smem sm = carve(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The producer's first block-table entries and the tensor-map prefetches
  // are issued before the barrier set-up so their latency overlaps it.
  int phys = 0, nxt = 0;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    // Range-checked only after Q is requested: the check waits for the load.
    phys = __ldg(p.tables + static_cast<int64_t>(seq) * p.maxb);
    nxt = nkv > 2 ? __ldg(p.tables + static_cast<int64_t>(seq) * p.maxb + 1) : 0;
  }
  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full[0], 1);
    mbar_init(&sm.q_full[1], 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], has_b ? 2 : 1);  // released by each slot's S
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], has_b ? 2 : 1);  // released by each slot's P V
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 4);
      mbar_init(&sm.pv_done[i], 1);
      mbar_init(&sm.o_done[i], 1);
      mbar_init(&sm.drain[i], 1);
    }
    mbar_init(&sm.s_free[0], 4);
    mbar_init(&sm.s_free[1], 4);
    fence_barrier_init();
    // Q and the first K tile go out before the tensor-memory allocation and
    // the block-wide barrier (stage 0 starts empty, so no wait).
    const int row0 = q0 + kTileM * m;
    // Order Q_A, K(0), Q_B: slot A's first S needs only the first two.
    mbar_arrive_expect_tx(&sm.q_full[0], kTileBytes);
    tma_load_3d(sm.q, &qmap, &sm.q_full[0], 0, hA, row0);
    tma_load_3d(sm.q + kHalfBytes, &qmap, &sm.q_full[0], 64, hA, row0);
    phys = checked_block(p, phys);
    mbar_arrive_expect_tx(&sm.k_full[0], kTileBytes);
    load_kv_tile(p, &kmap, sm.k0, &sm.k_full[0], phys, 0, g);
    if (has_b) {
      mbar_arrive_expect_tx(&sm.q_full[1], kTileBytes);
      tma_load_3d(sm.q + kTileBytes, &qmap, &sm.q_full[1], 0, hA + 1, row0);
      tma_load_3d(sm.q + kTileBytes + kHalfBytes, &qmap, &sm.q_full[1], 64, hA + 1, row0);
    }
    nxt = checked_block(p, nxt);
  }
  if (warp == 1) {
    tc::alloc(sm.tmem_base, kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *sm.tmem_base;
  // columns: S 0-127, P_A 128-191, P_B 192-255, O_A 256-383, O_B 384-511

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Order K(0) (already issued with Q), K(1), V(0), K(2), V(1), ...: the
      // MMA warps need K(j+1) (for the next S) before V(j) (for P V of j).
      int phys_v = phys;  // block of the next V tile
      int klast = 0, vlast = -1;  // last K and V tiles issued (K(0) went out with Q)
      bool aborted = false;
      for (int j = 1; j <= nkv && !aborted; ++j) {
        if (j < nkv) {
          if ((j & 1) == 0 && j > 0) {
            phys = nxt;
            if (2 * (j / 2 + 1) < nkv) nxt = load_block(p, seq, j / 2 + 1);
          }
          const int sk = j % kKStages;
          if (!mbar_wait(&sm.k_empty[sk], ((j / kKStages) & 1) ^ 1, &g_err_prefill)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&sm.k_full[sk], kTileBytes);
          load_kv_tile(p, &kmap, sm.k0 + sk * kTileBytes, &sm.k_full[sk], phys, (j & 1) * kTileN, g);
          klast = j;
        }
        if (j > 0) {
          const int jv = j - 1, sv = jv % kVStages;
          if (!mbar_wait(&sm.v_empty[sv], ((jv / kVStages) & 1) ^ 1, &g_err_prefill)) {
            aborted = true;
            break;
          }
          mbar_arrive_expect_tx(&sm.v_full[sv], kTileBytes);
          load_kv_tile(p, &vmap, sm.v0 + sv * kTileBytes, &sm.v_full[sv], phys_v, (jv & 1) * kTileN, g);
          vlast = jv;
          if (jv & 1) phys_v = phys;  // V(jv + 1) starts the block K(j) is in
        }
      }
      if (aborted) {
        // Let every copy already issued land before shared memory is given
        // up: the last load of each stage, and both Q tiles.
        for (int st = 0; st < kKStages; ++st) {
          const int j = klast - (klast - st + kKStages) % kKStages;
          if (j >= 0) drain_wait(&sm.k_full[st], (j / kKStages) & 1);
        }
        for (int st = 0; st < kVStages; ++st) {
          const int j = vlast - (vlast - st + kVStages) % kVStages;
          if (vlast >= 0 && j >= 0) drain_wait(&sm.v_full[st], (j / kVStages) & 1);
        }
        drain_wait(&sm.q_full[0], 0);
        if (has_b) drain_wait(&sm.q_full[1], 0);
      }
    }
  } else if (warp == 1 || (warp == 10 && has_b)) {
    // ------------------------------------------------------------ MMA issue
    // One issuing thread per slot (warp 1: A, warp 10: B).  An issuing thread
    // stays blocked while its MMAs queue behind the tensor pipe, so with one
    // thread per slot one slot's waits overlap the other slot's MMAs.
    if (lane == 0) {
      const int slot = warp == 1 ? 0 : 1;
      const uint32_t qa = smem_u32(sm.q), k0a = smem_u32(sm.k0), v0a = smem_u32(sm.v0);
      const uint64_t qd = desc_add(tc::smem_desc_sw128(qa, 16, 1024), slot * kTileBytes);
      const uint64_t kd0 = tc::smem_desc_sw128(k0a, 16, 1024);
      const uint64_t vd0 = tc::smem_desc_sw128(v0a, kHalfBytes, 1024);
      const uint32_t sT = tmem, pX = tmem + 128 + 64 * slot, oX = tmem + 256 + 128 * slot;
      // The S columns are handed over S_A(0), S_B(0), S_A(1), ...: S_X(j)
      // waits for s_free[X] phase j - 1 (slot A) or j (slot B), completed
      // when the other slot (or, with one slot, this one) has read its S.
      bool ok = mbar_wait(&sm.q_full[slot], 0, &g_err_prefill) && mbar_wait(&sm.k_full[0], 0, &g_err_prefill);
      if (ok && slot == 1) ok = mbar_wait(&sm.s_free[1], 0, &g_err_prefill);
      if (ok) {
        tc::fence_after();
        issue_s(sT, qd, kd0);
        tc::commit(&sm.s_full[slot]);
        tc::commit(&sm.k_empty[0]);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int sv = j % kVStages;
        const bool more = j + 1 < nkv;
        const int st1 = (j + 1) % kKStages;
        if (more) {
          if (!mbar_wait(&sm.s_free[slot], (slot == 0 ? j : j + 1) & 1, &g_err_prefill) ||
              !mbar_wait(&sm.k_full[st1], ((j + 1) / kKStages) & 1, &g_err_prefill)) {
            ok = false;
            break;
          }
          tc::fence_after();
          issue_s(sT, qd, desc_add(kd0, st1 * kTileBytes));
          tc::commit(&sm.s_full[slot]);
          tc::commit(&sm.k_empty[st1]);
        }
        if (!mbar_wait(&sm.p_full[slot], j & 1, &g_err_prefill) ||
            !mbar_wait(&sm.v_full[sv], (j / kVStages) & 1, &g_err_prefill)) {
          ok = false;
          break;
        }
        tc::fence_after();
        issue_pv(oX, pX, desc_add(vd0, sv * kTileBytes), j > 0);
        tc::commit(&sm.pv_done[slot]);
        if (!more) tc::commit(&sm.o_done[slot]);
        tc::commit(&sm.v_empty[sv]);
      }
      if (!ok) {
        // A wait gave up: every MMA this thread issued has completed once
        // this commit arrives, so tensor memory can be freed after it.
        tc::commit(&sm.drain[slot]);
        drain_wait(&sm.drain[slot], 0);
      }
    }
  } else if (warp >= 2 && warp < 10 && (warp < 6 || has_b)) {
    // ------------------------------------------------------------ softmax + epilogue
    const int slot = warp >= 6 ? 1 : 0;
    const int h = hA + slot;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_bits;                   // shared S columns
    const uint32_t p_addr = tmem + 128 + slot * 64 + lane_bits;  // this slot's P
    const uint32_t o_addr = tmem + 256 + slot * 128 + lane_bits;
    const int lim_row = c + kTileM * m + r;  // last visible key of this row
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      if (!mbar_wait(&sm.s_full[slot], j & 1, &g_err_prefill)) {
        ok = false;
        break;
      }
      tc::fence_after();
      // causal mask: key 128 j + x is visible iff x <= lim.  Only warps that
      // hold a diagonal row take the masked path; the mask of a 32-key
      // chunk is a 32-bit word (bit x set iff key x of the chunk is visible).
      const int lim = lim_row - kTileN * j;
      const bool wdiag = __any_sync(0xffffffffu, lim < kTileN - 1);
      // All 128 scores of the row in one tensor-memory round trip.
      float s[128];
      tc::ld32(s_addr + 0, s + 0);
      tc::ld32(s_addr + 32, s + 32);
      tc::ld32(s_addr + 64, s + 64);
      tc::ld32(s_addr + 96, s + 96);
      tc::wait_ld();
      // S is in registers: let the MMA warp reuse the S columns.
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[(slot == 0 && has_b) ? 1 : 0]);
      if (wdiag) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int nv = lim - 32 * q + 1;  // visible keys in chunk q
          const uint32_t vm = nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : ((1u << nv) - 1u));
#pragma unroll
          for (int x = 0; x < 32; ++x)
            if (!((vm >> x) & 1u)) s[32 * q + x] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = s[u];
#pragma unroll
      for (int x = 8; x < 128; x += 2) mx[(x >> 1) & 7] = fmax3(mx[(x >> 1) & 7], s[x], s[x + 1]);
      const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      const float m_new = fmaxf(m_ref, mt * p.sl2);
      float alpha = 1.f;
      if (m_new > m_ref + 8.f) {
        alpha = fast_exp2(m_ref - m_new);  // 0 on the first tile (m_ref = -inf)
        m_ref = m_new;
      }
      const float mu = m_ref;  // finite: key 0 is visible to every row
      // p = 2^(s * scale * log2e - m), packed to bf16 pairs; the first
      // 64 keys before the wait below (their exponentials overlap PV_X(j-1)),
      // the rest after it (keys 32q..32q+31 go to columns 16q..16q+15).
      float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 sl2 = make_float2(p.sl2, p.sl2), nmu = make_float2(-mu, -mu);
      uint32_t pk[64];
#pragma unroll
      for (int x = 0; x < 64; x += 2) {
        const float2 a = ffma2(make_float2(s[x], s[x + 1]), sl2, nmu);
        const float2 e = make_float2(fast_exp2(a.x), fast_exp2(a.y));
        rs[(x >> 1) & 3] = fadd2(rs[(x >> 1) & 3], e);
        pk[x >> 1] = pack_bf16x2(e.x, e.y);
      }
      // P_X(j-1) must be consumed (and O_X stable) before P_X(j) is stored.
      if (j > 0) {
        if (!mbar_wait(&sm.pv_done[slot], (j - 1) & 1, &g_err_prefill)) {
          ok = false;
          break;
        }
        tc::fence_after();
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) tc::st16u(p_addr + 16 * q, pk + 16 * q);
#pragma unroll
      for (int q = 2; q < 4; ++q) {
#pragma unroll
        for (int x = 32 * q; x < 32 * q + 32; x += 2) {
          const float2 a = ffma2(make_float2(s[x], s[x + 1]), sl2, nmu);
          const float2 e = make_float2(fast_exp2(a.x), fast_exp2(a.y));
          rs[(x >> 1) & 3] = fadd2(rs[(x >> 1) & 3], e);
          pk[x >> 1] = pack_bf16x2(e.x, e.y);
        }
        tc::st16u(p_addr + 16 * q, pk + 16 * q);
      }
      // O_X is stable here: PV_X(j-1) has completed (pv_done above).
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float o[32];
          tc::ld32(o_addr + cc * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] *= alpha;
          tc::st32(o_addr + cc * 32, o);
        }
      }
      const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
      const float2 rt = fadd2(r01, r23);
      l = l * alpha + (rt.x + rt.y);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[slot]);
    }
    if (ok && mbar_wait(&sm.o_done[slot], 0, &g_err_prefill)) {
      tc::fence_after();
      const float inv = fast_rcp(l);
      // Stage the bf16 row in this slot's Q buffer (free: o_done implies
      // every MMA of the CTA that reads Q has completed) in the layout of a
      // TMA box: 64-dim halves 16 KiB apart, 128-byte rows, 16-byte chunk c
      // of row r at chunk c ^ (r % 8).  A warp whose 32 rows all belong to
      // the sequence stores each 64-dim half with a bulk tensor copy as soon
      // as it is staged; otherwise it writes its rows that exist with
      // ordinary stores.
      fence_proxy_async_smem();
      uint8_t* stage = sm.q + slot * kTileBytes;
      const int rows_left = n - kTileM * m;  // rows of this tile inside the sequence
      const bool whole = 32 * wq + 32 <= rows_left;
      const int row0 = q0 + kTileM * m + 32 * wq;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float o[64];
        tc::ld32(o_addr + 64 * hh, o);
        tc::ld32(o_addr + 64 * hh + 32, o + 32);
        tc::wait_ld();
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const float* v = o + 8 * c8;
          uint4 w;
          w.x = pack_bf16x2(v[0] * inv, v[1] * inv);
          w.y = pack_bf16x2(v[2] * inv, v[3] * inv);
          w.z = pack_bf16x2(v[4] * inv, v[5] * inv);
          w.w = pack_bf16x2(v[6] * inv, v[7] * inv);
          *reinterpret_cast<uint4*>(stage + hh * kHalfBytes + r * 128 + ((c8 ^ (r & 7)) << 4)) = w;
        }
        if (whole) {  // this half goes out while the next one is staged
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tma_store_3d(&omap, stage + hh * kHalfBytes + wq * 32 * 128, 64 * hh, h, row0);
        }
      }
      if (whole) {
        if (lane == 0) bulk_commit_and_wait_read();
        __syncwarp();
      } else {
        __syncwarp();
        const int ch = lane & 15;
        const int64_t row_stride = static_cast<int64_t>(p.Hq) * kHeadDim;  // elements between token rows
        uint16_t* dst0 = p.out + static_cast<int64_t>(q0 + kTileM * m) * row_stride + h * kHeadDim + ch * 8;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int tr = 32 * wq + 2 * i + (lane >> 4);  // tile row written by this lane
          const uint4 w = *reinterpret_cast<const uint4*>(stage + (ch >> 3) * kHalfBytes + tr * 128 +
                                                          (((ch & 7) ^ (tr & 7)) << 4));
          if (tr < rows_left) {
            uint16_t* dst = dst0 + tr * row_stride;
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(w.x), "r"(w.y), "r"(w.z),
                         "r"(w.w)
                         : "memory");
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
                                      const CUtensorMap& omap, int num_sms, cudaStream_t stream) {
  if (a.total_q == 0 || a.num_seqs == 0) return cudaSuccess;
  // Short query tiles: a CTA launch per 128-row tile costs about as much as
  // the tile's tensor work, so they go to the persistent kernel.
  // The fused KV write needs every CTA resident at once (a grid barrier
  // separates the write from the first cache read): also the persistent kernel.
  if (a.max_seqlen_q <= kPersistentMaxSeqlenQ) return launch_prefill_persistent(a, kv, qmap, omap, num_sms, stream);
  if (a.k_new) {
    // Long prompts: the write costs the same as its own kernel, and this
    // kernel is faster than the persistent one there.  The attention kernel's
    // dependent-launch wait orders its cache reads after the write.
    cudaError_t e = launch_kv_cache_write(a.k_new, a.k_stride, a.v_new, a.v_stride, a.slot_mapping, a.total_q,
                                          a.k_cache, a.v_cache, static_cast<int64_t>(a.num_blocks) * kBlockSize,
                                          a.num_kv_heads * kHeadDim, stream);
    if (e != cudaSuccess) return e;
    PrefillArgs b = a;
    b.k_new = b.v_new = nullptr;
    b.slot_mapping = nullptr;
    b.k_cache = b.v_cache = nullptr;
    b.barrier_ws = nullptr;
    return launch_paged_attn_prefill(b, kv, qmap, omap, num_sms, stream);
  }
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
  p.npairs = (p.G + 1) / 2;
  p.num_blocks = a.num_blocks;
  p.total_q = a.total_q;
  p.per_half = kv.per_head;
  p.sl2 = a.scale * 1.4426950408889634f;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = ensure_dyn_smem(prefill_kernel, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int max_tiles = (a.max_seqlen_q + kTileM - 1) / kTileM;
  dim3 grid(a.num_kv_heads * p.npairs, a.num_seqs, max_tiles);
  return launch_pdl(prefill_kernel, grid, dim3(kThreads), kSmemBytes, stream, qmap, kv.k, kv.v, omap, p);
}

cudaError_t read_error_prefill(uint32_t* out, bool clear) {
  unsigned int v = 0;
  uint32_t vp = 0;
  cudaError_t e = read_error_prefill_persistent(&vp, clear);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(&v, g_err_prefill, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v | vp;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_prefill, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
