// prefill_persistent.cu -- varlen causal GQA prefill attention for batches of
// short query tiles: one persistent CTA per SM walks a list of work items, so
// an item's start and end overlap its neighbours' tensor work instead of each
// costing a CTA launch.  The per-tile arithmetic is the grid kernel's
// (prefill.cu) step for step, in the same order, so both give bit-identical
// outputs; the library runs this kernel when the stated max_seqlen_q is at
// most 2048 and the grid kernel above that.
//
// Page "13. 读一个最小推理引擎：nano-vllm": section "第二站：一个请求的状态" (each
// step computes from num_cached_tokens onward); "第三站：调度器" (only the
// first sequence of a step may be a split chunk, so a step is mostly whole
// short prompts); "第六站：注意力层" (with prefix hits or a chunk continuation
// the block table is passed so the whole context is read from the paged
// cache).  Query row j of sequence i sits at position c_i + j, c_i = L_i - n_i,
// and sees keys 0 .. c_i + j.
//
// A work item is one 128-row query tile of one sequence for TWO query heads of
// the same kv group ("slots" A and B), which share every K/V tile and the
// causal mask.  Warpgroups (16 warps):
// * WG0 (64 registers a thread): warp 0 producer, warps 1-2 MMA issue (slot A,
//   slot B), warp 3 scheduler.
//   - Item order.  Every CTA derives the same list on the device from
//     cu_seqlens: query tiles sorted by the number of K/V tiles they read,
//     most first (ties: sequence order), each tile expanded into its (kv head,
//     head pair) items; CTA c takes list positions c, 2G-1-c, c+2G, ... (G =
//     CTAs), a snake deal of a longest-first list.  Very long level ranges
//     fall back to "each sequence's last query tile, then the one before".
//     The scheduler hands this CTA's items (with the first two block-table
//     entries) to the other warps through an 8-deep queue in shared memory
//     (an entry is refilled only after every reader, the epilogue last, has
//     released it: 4 deep held the item hand-over back by ~9% on short
//     prompts).
//   - The producer TMA-loads each item's two Q tiles and streams the kv head's
//     128-token K and V tiles (two per 256-token block) into rings of three K
//     and two V stages, as 64-dim halves of 128 rows x 128 bytes with the
//     128-byte swizzle.  The next item's first K tile is loaded while the
//     current item's last tiles are in use and its Q tile for a slot as soon
//     as that slot's last S of the current item has completed; after the next
//     item's first K tile one K-ring entry is handed to the epilogue as the
//     output staging buffer of the item just finished.
//   - One thread per slot issues tcgen05.mma (kind::f16, bf16 in, fp32
//     accumulate), S(j+1) before P V(j).  Tensor memory holds S (128 columns,
//     shared by the slots and handed over S_A(0), S_B(0), S_A(1), ...),
//     P_A | P_B (64 columns each, packed bf16) and O_A | O_B (128 each).
// * WG1 / WG2 (176 registers): softmax of slot A / B; thread r owns query row
//   r (TMEM lane r): scores read with tcgen05.ld, S columns released, causal
//   mask on diagonal tiles, running maximum in log2 units, all 128
//   probabilities packed in registers before the wait for the slot's
//   previous P V, then P stored and O rescaled in tensor memory only when the
//   maximum grew by more than 2^8; the row sum goes to the epilogue through
//   shared memory.
// * WG3 (96 registers): epilogue; per item and slot it reads O (after which the
//   slot's next P V may overwrite it), normalises by the row sum and writes
//   the bf16 rows through the staging entry (bulk tensor stores for warps
//   whose 32 rows all exist, ordinary stores at a sequence's end).
// Every wait is bounded (two seconds); a wait that gives up flags
// PKV_DEVERR_WAIT_TIMEOUT and raises a CTA-wide abort flag that ends every
// role's loop.  Before the tensor memory is freed the MMA threads wait for
// their issued MMAs, the producer for its issued loads and the storing
// threads for their bulk stores.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_prefill_persistent;

constexpr int kTileM = 128;    // query rows per slot
constexpr int kTileN = 128;    // keys per K/V tile
constexpr int kKStages = 3;    // K ring (also carries the epilogue staging entries)
constexpr int kVStages = 2;    // V ring
constexpr int kQueue = 8;      // work-item queue depth
constexpr int kThreads = 512;  // 16 warps = 4 warpgroups
constexpr int kWarpProducer = 0, kWarpMmaA = 1, kWarpSched = 3, kWarpSoftmax = 4, kWarpEpi = 12;
constexpr int kItemReaders = 15;  // warps that take items off the queue: all but the scheduler
// Registers per thread after the warpgroups rebalance them (setmaxnreg).  The
// launch gives every thread 128 (512 threads, 64K registers); the four
// shares below add up to exactly that total: 64 + 176 + 176 + 96 = 4 x 128.
constexpr int kRegsLaunch = 128, kRegsCtl = 64, kRegsSoftmax = 176, kRegsEpi = 96;
static_assert(kRegsCtl + 2 * kRegsSoftmax + kRegsEpi == 4 * kRegsLaunch, "register split must match the launch");
constexpr int kSortLimit = 8192;  // level x sequence-chunk steps allowed for the sorted order
constexpr uint32_t kTileBytes = kTileN * kHeadDim * 2;  // 32 KiB: one Q, K or V tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;         // one 64-dim half
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kTileM, kTileN, 0);    // B = K tile, K-major
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kTileM, kHeadDim, 1);  // B = V tile, N-major
constexpr uint64_t kDrainNs = 100000000ull;  // bound of the waits that drain in-flight work

// The KV write fused in front of the attention (optional): every new token's
// K and V row goes to its cache slot before any CTA reads the cache.
struct FusedWrite {
  const uint16_t* k_new;  // null: no fused write
  const uint16_t* v_new;
  int64_t k_stride, v_stride;  // elements between token rows
  const int32_t* slots;        // [num_tokens]
  uint16_t* k_cache;
  uint16_t* v_cache;
  int64_t num_slots;
  int32_t num_tokens, row_elems;  // row_elems = num_kv_heads * 128
  unsigned int* barrier;          // caller workspace: [0] arrivals, [1] epoch
};

struct PrefillParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* tables;
  uint16_t* out;
  int32_t maxb, S, Hq, Hkv, G, npairs, num_blocks, total_q, per_half, max_tiles;
  float sl2;  // scale * log2(e)
  FusedWrite fw;
};

// One work item: a 128-row query tile of one sequence for one head pair.
struct Item {
  int seq;   // < 0: no more items
  int m;     // query tile within the sequence
  int g;     // kv head
  int hA;    // query head of slot A (slot B: hA + 1)
  int has_b;
  int q0;    // first packed query row of the sequence
  int n, c;  // new and cached tokens of the sequence
  int nkv;   // K/V tiles visible to some row of the tile
  int phys0, phys1;  // block-table entries 0 and 1 (unchecked; phys1 only if nkv > 2)
  int pad[5];
};
static_assert(sizeof(Item) == 64, "queue entry size");

// Shared memory: Q_A | Q_B | K stages | V stages | barriers | queue | flags,
// addressed as constant offsets from one 1024-byte aligned base so that no
// pointer per buffer or barrier occupies registers.
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
// barrier indices
constexpr int kBQFull = 0;                   // [2 slots]
constexpr int kBQEmpty = 2;                  // [2 slots]: the slot's last S of the item has completed
constexpr int kBKFull = 4;                   // [kKStages]
constexpr int kBKEmpty = kBKFull + kKStages;  // [kKStages]
constexpr int kBVFull = kBKEmpty + kKStages;  // [kVStages]
constexpr int kBVEmpty = kBVFull + kVStages;  // [kVStages]
constexpr int kBSFull = kBVEmpty + kVStages;  // [2 slots]: S of this slot computed
constexpr int kBSFree = kBSFull + 2;          // [2]: the shared S columns may take this slot's next S
constexpr int kBPFull = kBSFree + 2;          // [2 slots]: P of this slot stored
constexpr int kBPvDone = kBPFull + 2;         // [2 slots]: P V of this slot completed
constexpr int kBODone = kBPvDone + 2;         // [2 slots]: the item's last P V of this slot completed
constexpr int kBOFree = kBODone + 2;          // [2 slots]: O of this slot has been read by the epilogue
constexpr int kBDrain = kBOFree + 2;          // [2 slots]: every MMA of this slot's issuer completed
constexpr int kBEDone = kBDrain + 2;          // [1]: the epilogue warps left the staging entry
constexpr int kBLReady = kBEDone + 2;         // [2 slots]: the item's row sums are in shared memory
constexpr int kBLFree = kBLReady + 2;         // [2 slots]: the epilogue has read them
constexpr int kBItFull = kBLFree + 2;         // [kQueue]
constexpr int kBItEmpty = kBItFull + kQueue;  // [kQueue]
constexpr int kNumBarriers = kBItEmpty + kQueue;
constexpr uint32_t kOffItems = kOffBar + kNumBarriers * 8;
constexpr uint32_t kOffLsum = kOffItems + kQueue * sizeof(Item);  // float [2 slots][128 rows]
constexpr uint32_t kOffTmem = kOffLsum + 2 * kTileM * 4;
constexpr uint32_t kOffAbort = kOffTmem + 4;
constexpr size_t kSmemBytes = 1024 + kOffAbort + 4;
static_assert(kOffItems % 16 == 0, "queue entries are copied as 16-byte words");
static_assert(kSmemBytes <= 232448, "shared memory per block");

struct Smem {
  uint8_t* gen;  // generic address of the aligned base
  uint32_t sa;   // shared-window address of the aligned base
  __device__ __forceinline__ uint32_t bar(int i) const { return sa + kOffBar + 8u * i; }
  __device__ __forceinline__ Item* item(int i) const { return reinterpret_cast<Item*>(gen + kOffItems) + i; }
  __device__ __forceinline__ int* abort() const { return reinterpret_cast<int*>(gen + kOffAbort); }
  __device__ __forceinline__ float* lsum(int slot) const {
    return reinterpret_cast<float*>(gen + kOffLsum) + slot * kTileM;
  }
};

// ---------------------------------------------------------------- mbarrier ops on shared-window addresses
__device__ __forceinline__ void bar_init(uint32_t b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(b) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t b, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(b),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bar_try_wait(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}
// Arrive on `b` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void tma3(uint32_t dst, const CUtensorMap* map, uint32_t b, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(b), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma5(uint32_t dst, const CUtensorMap* map, uint32_t b, int c0, int c1, int c2,
                                     int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(b), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// Bounded wait that also gives up when another role has raised the CTA's
// abort flag.  A wait that times out flags PKV_DEVERR_WAIT_TIMEOUT and raises
// the flag itself.  Every role polls without sleeping: a sleep of even 200 ns
// in the epilogue and scheduler warps delayed the hand-over of items and of
// O by more than their polling costs the softmax warps.
__device__ __forceinline__ bool wait(const Smem& sm, uint32_t b, uint32_t parity) {
  if (bar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (bar_try_wait(b, parity)) return true;
    if ((i & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(sm.abort())) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
        atomicOr(&g_err_prefill_persistent, PKV_DEVERR_WAIT_TIMEOUT);
        *reinterpret_cast<volatile int*>(sm.abort()) = 1;
        return false;
      }
    }
  }
}

// The same wait by every lane of a warp, with one warp-wide answer, so that
// the warp stays converged for the tcgen05 loads that follow.
__device__ __forceinline__ bool wait_warp(const Smem& sm, uint32_t b, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(sm, b, parity));
}

// Wait used only to drain work already in flight after an abort: bounded,
// ignores the abort flag, reports nothing (the abort has been reported).
__device__ __forceinline__ void drain_wait(uint32_t b, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!bar_try_wait(b, parity))
    if (globaltimer_ns() - t0 > kDrainNs) return;
}

__device__ __forceinline__ int checked_block(const PrefillParams& p, int phys) {
  if (phys < 0 || phys >= p.num_blocks) {
    atomicOr(&g_err_prefill_persistent, PKV_DEVERR_BLOCK_RANGE);
    phys = 0;
  }
  return phys;
}

__device__ __forceinline__ int table_entry(const PrefillParams& p, int seq, int lb) {
  return __ldg(p.tables + static_cast<int64_t>(seq) * p.maxb + lb);
}

// One 128-token K or V tile (all 128 dims of kv head g) into shared address
// `dst` as two swizzled 64-dim halves.
__device__ __forceinline__ void load_kv_tile(const PrefillParams& p, const CUtensorMap* map, uint32_t dst,
                                             uint32_t b, int phys, int tin, int g) {
  if (!p.per_half) {
    tma5(dst, map, b, 0, tin, g, 0, phys);
  } else {
    const int slot = phys * kBlockSize + tin;
    tma3(dst, map, b, 0, g, slot);
    tma3(dst + kHalfBytes, map, b, 64, g, slot);
  }
}

// Matrix descriptors are built once per CTA; a k-step only adds a constant to
// the 16-byte address field in the low bits (the addresses stay below
// 256 KiB, so the add never carries out of the field).  Rebuilding the 64-bit
// descriptor for every instruction made the single issuing thread, not the
// tensor pipe, the limit.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Bulk tensor store of one box from shared memory, tracked by the bulk
// async-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// tcgen05.mma with the k-step's constant descriptor offsets added inside the
// instruction sequence, so the issuing thread keeps only the base
// descriptors in registers (a precomputed descriptor per k-step would hold
// 32 registers in a warp that runs with 64).  The offset lands in the 14-bit
// start-address field (bits 0-13: shared-memory address / 16, below 2^14 for
// any operand inside the CTA's shared memory), so it never carries out of the
// low word and a 32-bit add is exact.
template <uint32_t AOFF, uint32_t BOFF>
__device__ __forceinline__ void mma_ss_at(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 t, u;\n\t.reg .b64 a, b;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "add.u32 t, %1, %7;\n\tadd.u32 u, %3, %8;\n\t"
      "mov.b64 a, {t, %2};\n\tmov.b64 b, {u, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t}" ::"r"(d),
      "r"(static_cast<uint32_t>(adesc)), "r"(static_cast<uint32_t>(adesc >> 32)),
      "r"(static_cast<uint32_t>(bdesc)), "r"(static_cast<uint32_t>(bdesc >> 32)), "r"(idesc), "r"(acc),
      "n"(AOFF >> 4), "n"(BOFF >> 4)
      : "memory");
}
template <uint32_t BOFF>
__device__ __forceinline__ void mma_ts_at(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 u;\n\t.reg .b64 b;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "add.u32 u, %2, %6;\n\tmov.b64 b, {u, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(static_cast<uint32_t>(bdesc)), "r"(static_cast<uint32_t>(bdesc >> 32)), "r"(idesc),
      "r"(acc), "n"(BOFF >> 4)
      : "memory");
}

// S = Q K^T: A = Q tile, B = K tile, both K-major (dims contiguous) with the
// 128-byte swizzle; k-step kk selects 32 bytes of a 64-dim half.
template <int KK = 0>
__device__ __forceinline__ void issue_s(uint32_t d, uint64_t qdesc, uint64_t kdesc) {
  if constexpr (KK < kHeadDim / 16) {
    constexpr uint32_t off = (KK >> 2) * kHalfBytes + (KK & 3) * 32;
    mma_ss_at<off, off>(d, qdesc, kdesc, kIdescS, KK > 0 ? 1u : 0u);
    issue_s<KK + 1>(d, qdesc, kdesc);
  }
}

// O += P V with P (128 x 128 keys, packed bf16) in tensor memory at `p_tmem`
// and V (keys x dims, dims contiguous) in shared memory: 64-dim halves are
// 16 KiB apart (leading offset), 8-key groups 1 KiB apart (stride offset).
template <int KK = 0>
__device__ __forceinline__ void issue_pv(uint32_t o, uint32_t p_tmem, uint64_t vdesc, bool acc) {
  if constexpr (KK < kTileN / 16) {
    mma_ts_at<KK * 2048>(o, p_tmem + KK * 8, vdesc, kIdescPV, (acc || KK > 0) ? 1u : 0u);
    issue_pv<KK + 1>(o, p_tmem, vdesc, acc);
  }
}

// ---------------------------------------------------------------- item queue
// Entry k lives in queue slot k % kQueue; its phase parity is (k / kQueue) & 1.
__device__ __forceinline__ bool queue_get(const Smem& sm, int k, Item& it) {
  if (!wait(sm, sm.bar(kBItFull + k % kQueue), (k / kQueue) & 1)) return false;
  const int4* src = reinterpret_cast<const int4*>(sm.item(k % kQueue));
  int4* dst = reinterpret_cast<int4*>(&it);
#pragma unroll
  for (int i = 0; i < 3; ++i) dst[i] = src[i];
  return true;
}
__device__ __forceinline__ void queue_release(const Smem& sm, int k) { bar_arrive(sm.bar(kBItEmpty + k % kQueue)); }

// Per-sequence view used to enumerate query tiles.  A tile m of a sequence
// with n new and c cached tokens reads nkv(m) = ceil((c + min(128 (m+1), n)) / 128)
// K/V tiles: b + m + 1 for every tile but the last (b = ceil(c / 128)) and
// vlast = ceil((c + n) / 128) for the last.  Tiles below tmin (leading tiles
// beyond the stated max_seqlen_q) are not computed.
struct SeqTiles {
  int q0, n, c, T, tmin, b, vlast;
  bool bad;
};

__device__ __forceinline__ SeqTiles seq_tiles(const PrefillParams& p, int i) {
  SeqTiles t;
  const int q0 = __ldg(p.cu_q + i), q1 = __ldg(p.cu_q + i + 1);
  const int k0 = __ldg(p.cu_k + i), k1 = __ldg(p.cu_k + i + 1);
  const int n = q1 - q0, L = k1 - k0, c = L - n;
  const bool valid = n > 0 && c >= 0 && q0 >= 0 && q1 <= p.total_q && L <= p.maxb * kBlockSize;
  t.q0 = q0;
  t.n = n;
  t.c = c;
  t.T = valid ? (n + kTileM - 1) / kTileM : 0;
  t.tmin = t.T > p.max_tiles ? t.T - p.max_tiles : 0;
  t.b = valid ? (c + kTileN - 1) / kTileN : 0;
  t.vlast = valid ? (c + n + kTileN - 1) / kTileN : 0;
  t.bad = (n != 0 && !valid) || t.tmin > 0;
  return t;
}

__device__ __forceinline__ int nkv_of(const SeqTiles& t, int m) { return m == t.T - 1 ? t.vlast : t.b + m + 1; }

// Tiles of a sequence at one level of the enumeration: (sorted) the tiles
// reading exactly `lev` K/V tiles, the last tile first; (otherwise) the tile
// `lev` places before the sequence's last.
__device__ __forceinline__ int tiles_at(const SeqTiles& t, bool sorted, int lev, int& mA, int& mB) {
  int cnt = 0;
  if (sorted) {
    if (t.T > t.tmin && t.vlast == lev) mA = t.T - 1, cnt = 1;
    const int mm = lev - 1 - t.b;
    if (mm >= t.tmin && mm <= t.T - 2) {
      if (cnt) mB = mm;
      else mA = mm;
      ++cnt;
    }
  } else {
    const int mm = t.T - 1 - lev;
    if (mm >= t.tmin) mA = mm, cnt = 1;
  }
  return cnt;
}

// Largest level below `lev` at which the sequence has a tile (sorted order), or 0.
__device__ __forceinline__ int level_below(const SeqTiles& t, int lev) {
  if (t.T <= t.tmin) return 0;
  int best = t.vlast < lev ? t.vlast : 0;
  const int lo = t.b + 1 + t.tmin, hi = t.b + t.T - 1;  // levels of the tiles before the last
  if (lo <= hi && lo < lev) best = max(best, min(hi, lev - 1));
  return best;
}

// ------------------------------------------------------------------ scheduler
// Position p of the list belongs to CTA p mod 2G when that is below G, else
// to CTA 2G-1 - p mod 2G.  This CTA's positions, in order, are therefore
// c, 2G-1-c, c+2G, 2G-1-c+2G, ...
__device__ void run_scheduler(const PrefillParams& p, const Smem& sm, int lane) {
  const int nch = (p.S + 31) / 32;
  int vmax = 0, zmax = 0;
  bool bad = false;
  for (int ch = 0; ch < nch; ++ch) {
    const int i = 32 * ch + lane;
    if (i < p.S) {
      const SeqTiles t = seq_tiles(p, i);
      if (t.T > t.tmin) {
        vmax = max(vmax, t.vlast);
        zmax = max(zmax, t.T - t.tmin);
      }
      bad |= t.bad;
    }
  }
#pragma unroll
  for (int d = 16; d; d >>= 1) {
    vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, d));
    zmax = max(zmax, __shfl_xor_sync(0xffffffffu, zmax, d));
  }
  if (__any_sync(0xffffffffu, bad) && blockIdx.x == 0 && lane == 0) atomicOr(&g_err_prefill_persistent, PKV_DEVERR_LEN_RANGE);
  const bool sorted = static_cast<long long>(vmax) * nch <= kSortLimit;
  // Positions stay below 2^31: there are at most total_q / 128 + S tiles and
  // at most 64 items per tile.
  const int G2 = 2 * static_cast<int>(gridDim.x);
  const int step_a = G2 - 1 - 2 * static_cast<int>(blockIdx.x);  // c -> 2G-1-c
  const int HG = p.Hkv * p.npairs;
  int target = blockIdx.x;  // next position of this CTA
  bool second = false;      // target is of the form 2G-1-c + 2G l
  int rbase = 0;            // tiles enumerated so far
  int kq = 0;               // items pushed
  bool ok = true;
  int lev = sorted ? vmax : 0;
  while (ok && (sorted ? lev > 0 : lev < zmax)) {
    int next = 0;  // sorted: the next lower level with a tile
    for (int ch = 0; ch < nch && ok; ++ch) {
      const int i = 32 * ch + lane;
      SeqTiles t{};
      int cnt = 0, mA = 0, mB = 0;
      if (i < p.S) {
        t = seq_tiles(p, i);
        cnt = tiles_at(t, sorted, lev, mA, mB);
        if (sorted) next = max(next, level_below(t, lev));
      }
      int inc = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += y;
      }
      const int tot = __shfl_sync(0xffffffffu, inc, 31);
      const int A = (rbase + inc - cnt) * HG, B = (rbase + inc) * HG;  // this lane's positions
      for (;;) {
        const unsigned mask = __ballot_sync(0xffffffffu, cnt > 0 && A <= target && target < B);
        if (!mask || !ok) break;
        const int src = __ffs(mask) - 1;
        const int off = target - __shfl_sync(0xffffffffu, A, src);
        const int u = off >= HG ? 1 : 0;  // which of the lane's (at most two) tiles
        const int hg = off - u * HG;
        const int s_seq = __shfl_sync(0xffffffffu, i, src);
        const int m = __shfl_sync(0xffffffffu, u ? mB : mA, src);
        SeqTiles st;
        st.q0 = __shfl_sync(0xffffffffu, t.q0, src);
        st.n = __shfl_sync(0xffffffffu, t.n, src);
        st.c = __shfl_sync(0xffffffffu, t.c, src);
        st.T = __shfl_sync(0xffffffffu, t.T, src);
        st.b = __shfl_sync(0xffffffffu, t.b, src);
        st.vlast = __shfl_sync(0xffffffffu, t.vlast, src);
        if (lane == 0) {
          const int slot = kq % kQueue;
          ok = wait(sm, sm.bar(kBItEmpty + slot), ((kq / kQueue) & 1) ^ 1);
          if (ok) {
            Item it;
            it.seq = s_seq;
            it.m = m;
            it.g = hg / p.npairs;
            const int pair = hg - it.g * p.npairs;
            it.hA = it.g * p.G + 2 * pair;
            it.has_b = 2 * pair + 1 < p.G;
            it.q0 = st.q0;
            it.n = st.n;
            it.c = st.c;
            it.nkv = nkv_of(st, m);
            it.phys0 = table_entry(p, s_seq, 0);
            it.phys1 = it.nkv > 2 ? table_entry(p, s_seq, 1) : 0;
            int4* dst = reinterpret_cast<int4*>(sm.item(slot));
            const int4* srcp = reinterpret_cast<const int4*>(&it);
#pragma unroll
            for (int w = 0; w < 3; ++w) dst[w] = srcp[w];
            bar_arrive(sm.bar(kBItFull + slot));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++kq;
        target += second ? G2 - step_a : step_a;
        second = !second;
      }
      rbase += tot;
    }
    if (sorted) {
#pragma unroll
      for (int d = 16; d; d >>= 1) next = max(next, __shfl_xor_sync(0xffffffffu, next, d));
      lev = next;
    } else {
      ++lev;
    }
  }
  if (ok && lane == 0) {
    const int slot = kq % kQueue;
    if (wait(sm, sm.bar(kBItEmpty + slot), ((kq / kQueue) & 1) ^ 1)) {
      sm.item(slot)->seq = -1;
      bar_arrive(sm.bar(kBItFull + slot));
    }
  }
}

// ------------------------------------------------------------------ producer
// Parity of the last load issued into stage `st` of a ring of `n` stages
// whose highest position issued so far is `last` (-1: none into that stage).
__device__ __forceinline__ int last_parity(int last, int st, int n) {
  if (last < 0) return -1;
  const int pos = last - (last - st + n) % n;
  return pos < 0 ? -1 : (pos / n) & 1;
}

__device__ void run_producer(const PrefillParams& p, const Smem& sm, const CUtensorMap* qmap,
                             const CUtensorMap* kmap, const CUtensorMap* vmap) {
  int klast = -1, vlast = -1;  // highest K-ring / V-ring position issued
  int nqa = 0, nqb = 0;        // Q loads issued per slot

  auto load_q = [&](int slot, const Item& it) -> bool {
    const int nq = slot ? nqb : nqa;
    if (nq > 0 && !wait(sm, sm.bar(kBQEmpty + slot), (nq - 1) & 1)) return false;
    const int row0 = it.q0 + kTileM * it.m;
    const uint32_t dst = sm.sa + kOffQ + slot * kTileBytes, b = sm.bar(kBQFull + slot);
    bar_expect_tx(b, kTileBytes);
    tma3(dst, qmap, b, 0, it.hA + slot, row0);
    tma3(dst + kHalfBytes, qmap, b, 64, it.hA + slot, row0);
    if (slot) ++nqb;
    else ++nqa;
    return true;
  };
  auto load_k = [&](int pos, int phys, int tile, int g) -> bool {
    const int st = pos % kKStages;
    if (!wait(sm, sm.bar(kBKEmpty + st), ((pos / kKStages) & 1) ^ 1)) return false;
    const uint32_t b = sm.bar(kBKFull + st);
    bar_expect_tx(b, kTileBytes);
    load_kv_tile(p, kmap, sm.sa + kOffK + st * kTileBytes, b, phys, (tile & 1) * kTileN, g);
    klast = pos;
    return true;
  };
  auto load_v = [&](int pos, int phys, int tile, int g) -> bool {
    const int st = pos % kVStages;
    if (!wait(sm, sm.bar(kBVEmpty + st), ((pos / kVStages) & 1) ^ 1)) return false;
    const uint32_t b = sm.bar(kBVFull + st);
    bar_expect_tx(b, kTileBytes);
    load_kv_tile(p, vmap, sm.sa + kOffV + st * kTileBytes, b, phys, (tile & 1) * kTileN, g);
    vlast = pos;
    return true;
  };
  // Hand a K-ring entry to the softmax warps as output staging.
  auto staging = [&](int pos) -> bool {
    const int st = pos % kKStages;
    if (!wait(sm, sm.bar(kBKEmpty + st), ((pos / kKStages) & 1) ^ 1)) return false;
    bar_arrive(sm.bar(kBKFull + st));
    klast = pos;
    return true;
  };

  bool ok = false;
  Item cur;
  if (queue_get(sm, 0, cur)) {
    queue_release(sm, 0);
    ok = true;
    if (cur.seq >= 0) {
      // Q_A, K(0), Q_B: slot A's first S needs only the first two.
      ok = load_q(0, cur) && load_k(0, checked_block(p, cur.phys0), 0, cur.g) && (!cur.has_b || load_q(1, cur));
      int kpos = 0, vpos = 0;
      for (int k = 0; ok; ++k) {
        const int off = k > 0 ? 1 : 0;
        const int base = kpos;  // position of K(0) of this item
        // Block ids: tiles 2b and 2b+1 read block b.
        int bcur = checked_block(p, cur.phys0), bprev = bcur;
        int bnext = cur.nkv > 2 ? cur.phys1 : 0;
        for (int j = 1; j < cur.nkv && ok; ++j) {
          if ((j & 1) == 0) {
            bprev = bcur;
            bcur = checked_block(p, bnext);
            if (j + 2 < cur.nkv) bnext = table_entry(p, cur.seq, j / 2 + 1);
          }
          ok = load_k(base + j + off, bcur, j, cur.g);
          // V(j-1) reads block (j-1)/2: the previous block when j starts one.
          if (ok) ok = load_v(vpos + j - 1, (j & 1) == 0 ? bprev : bcur, j - 1, cur.g);
        }
        if (!ok) break;
        Item nxt;
        if (!queue_get(sm, k + 1, nxt)) {
          ok = false;
          break;
        }
        queue_release(sm, k + 1);
        const int kend = base + cur.nkv + off;  // position after this item's K tiles
        const int last = cur.nkv - 1;
        if (nxt.seq < 0) {
          ok = load_v(vpos + last, bcur, last, cur.g) && staging(kend);
          break;
        }
        ok = load_k(kend, checked_block(p, nxt.phys0), 0, nxt.g) && staging(kend + 1) &&
             load_v(vpos + last, bcur, last, cur.g) && load_q(0, nxt) && (!nxt.has_b || load_q(1, nxt));
        kpos = kend;
        vpos += cur.nkv;
        cur = nxt;
      }
    }
  }
  if (!ok) {
    // Aborted: let every load already issued land before shared memory is
    // given up.
    for (int st = 0; st < kKStages; ++st) {
      const int par = last_parity(klast, st, kKStages);
      if (par >= 0) drain_wait(sm.bar(kBKFull + st), par);
    }
    for (int st = 0; st < kVStages; ++st) {
      const int par = last_parity(vlast, st, kVStages);
      if (par >= 0) drain_wait(sm.bar(kBVFull + st), par);
    }
    if (nqa > 0) drain_wait(sm.bar(kBQFull + 0), (nqa - 1) & 1);
    if (nqb > 0) drain_wait(sm.bar(kBQFull + 1), (nqb - 1) & 1);
  }
}

// ------------------------------------------------------------------ MMA issue
// One issuing thread per slot (warp 1: A, warp 2: B).  An issuing thread
// stays blocked while its MMAs queue behind the tensor pipe, so with one
// thread per slot one slot's waits overlap the other slot's MMAs.
__device__ void run_issuer(const Smem& sm, int slot, uint32_t tmem) {
  const uint64_t qd = desc_add(tc::smem_desc_sw128(sm.sa + kOffQ, 16, 1024), slot * kTileBytes);
  const uint64_t kd0 = tc::smem_desc_sw128(sm.sa + kOffK, 16, 1024);
  const uint64_t vd0 = tc::smem_desc_sw128(sm.sa + kOffV, kHalfBytes, 1024);
  const uint32_t sT = tmem, pX = tmem + 128 + 64 * slot, oX = tmem + 256 + 128 * slot;
  int kpos = 0, vpos = 0;
  int ns = 0, npv = 0, nq = 0;  // S and P V issued, items done by this slot
  bool ok = true;
  for (int k = 0; ok; ++k) {
    Item it;
    if (!queue_get(sm, k, it)) break;
    queue_release(sm, k);
    if (it.seq < 0) break;
    const int off = k > 0 ? 1 : 0;
    const int base = kpos, vbase = vpos, nkv = it.nkv;
    kpos = base + nkv + off;
    vpos = vbase + nkv;
    if (slot == 1 && !it.has_b) continue;
    // Stages shared with slot B are released by both slots; without slot B,
    // slot A releases them twice.
    const int reps = (slot == 0 && !it.has_b) ? 2 : 1;
    if (!wait(sm, sm.bar(kBQFull + slot), nq & 1)) break;
    // S_X(j).  The S columns are handed over S_A(0), S_B(0), S_A(1), ...:
    // S_A waits for the read of the S before it in that chain (s_free[0]);
    // S_B for slot A's read of S_A of the same tile (s_free[1]).
    auto issue_s_tile = [&](int j) -> bool {
      const int kp = j == 0 ? base : base + j + off;
      const int st = kp % kKStages;
      if (slot == 0) {
        if (ns > 0 && !wait(sm, sm.bar(kBSFree + 0), (ns - 1) & 1)) return false;
      } else {
        if (!wait(sm, sm.bar(kBSFree + 1), ns & 1)) return false;
      }
      if (!wait(sm, sm.bar(kBKFull + st), (kp / kKStages) & 1)) return false;
      tc::fence_after();
      issue_s(sT, qd, desc_add(kd0, st * kTileBytes));
      mma_commit(sm.bar(kBSFull + slot));
      for (int r = 0; r < reps; ++r) mma_commit(sm.bar(kBKEmpty + st));
      if (j == nkv - 1) mma_commit(sm.bar(kBQEmpty + slot));
      ++ns;
      return true;
    };
    if (!issue_s_tile(0)) break;
    for (int j = 0; j < nkv && ok; ++j) {
      if (j + 1 < nkv && !issue_s_tile(j + 1)) {
        ok = false;
        break;
      }
      const int vp = vbase + j, sv = vp % kVStages;
      if (!wait(sm, sm.bar(kBPFull + slot), npv & 1) || !wait(sm, sm.bar(kBVFull + sv), (vp / kVStages) & 1) ||
          (j == 0 && nq > 0 && !wait(sm, sm.bar(kBOFree + slot), (nq - 1) & 1))) {
        ok = false;
        break;
      }
      tc::fence_after();
      issue_pv(oX, pX, desc_add(vd0, sv * kTileBytes), j > 0);
      mma_commit(sm.bar(kBPvDone + slot));
      if (j == nkv - 1) mma_commit(sm.bar(kBODone + slot));
      for (int r = 0; r < reps; ++r) mma_commit(sm.bar(kBVEmpty + sv));
      ++npv;
    }
    ++nq;
  }
  // Every MMA this thread issued has completed (and its barrier arrivals
  // have landed) once this last commit arrives.
  mma_commit(sm.bar(kBDrain + slot));
  drain_wait(sm.bar(kBDrain + slot), 0);
}

// ------------------------------------------------------------ softmax
__device__ void run_softmax(const PrefillParams& p, const Smem& sm, int slot, int wq, int lane, uint32_t tmem) {
  const int r = wq * 32 + lane;  // tile row = TMEM lane
  const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t s_addr = tmem + lane_bits;                   // shared S columns
  const uint32_t p_addr = tmem + 128 + slot * 64 + lane_bits;  // this slot's P
  const uint32_t o_addr = tmem + 256 + slot * 128 + lane_bits;
  int gt = 0, ni = 0;  // tiles and items done by this slot
  bool ok = true;
  for (int k = 0; ok; ++k) {
    if (!__all_sync(0xffffffffu, wait(sm, sm.bar(kBItFull + k % kQueue), (k / kQueue) & 1))) break;
    const Item* e = sm.item(k % kQueue);
    const int seq = e->seq, nkv = e->nkv, has_b = e->has_b;
    const int lim_row = e->c + kTileM * e->m + r;  // last visible key of this row
    __syncwarp();
    if (lane == 0) queue_release(sm, k);
    if (seq < 0) break;
    if (slot == 1 && !has_b) continue;
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nkv; ++j, ++gt) {
      if (!wait_warp(sm, sm.bar(kBSFull + slot), gt & 1)) {
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
      if (lane == 0) bar_arrive(sm.bar(kBSFree + ((slot == 0 && has_b) ? 1 : 0)));
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
      // p = 2^(s * scale * log2e - m), packed to bf16 pairs in registers
      // before the wait below, so that the exponentials overlap the previous
      // tile's P V (keys 32q..32q+31 go to columns 16q..16q+15).
      float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 sl2 = make_float2(p.sl2, p.sl2), nmu = make_float2(-mu, -mu);
      uint32_t pk[64];
#pragma unroll
      for (int x = 0; x < 128; x += 2) {
        const float2 a = ffma2(make_float2(s[x], s[x + 1]), sl2, nmu);
        const float2 ex = make_float2(fast_exp2(a.x), fast_exp2(a.y));
        rs[(x >> 1) & 3] = fadd2(rs[(x >> 1) & 3], ex);
        pk[x >> 1] = pack_bf16x2(ex.x, ex.y);
      }
      // P_X of the previous tile must be consumed (and O_X stable) before
      // this tile's P_X is stored.
      if (gt > 0) {
        if (!wait_warp(sm, sm.bar(kBPvDone + slot), (gt - 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after();
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::st16u(p_addr + 16 * q, pk + 16 * q);
      // O_X is stable here: P V_X of the previous tile has completed.
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
      if (lane == 0) bar_arrive(sm.bar(kBPFull + slot));
    }
    if (!ok) break;
    // The row sum goes to the epilogue warps through shared memory (once
    // they have read the previous item's).
    if (ni > 0 && !wait(sm, sm.bar(kBLFree + slot), (ni - 1) & 1)) break;
    sm.lsum(slot)[r] = l;
    bar_arrive(sm.bar(kBLReady + slot));
    ++ni;
  }
  if (!ok) *reinterpret_cast<volatile int*>(sm.abort()) = 1;
}

// ------------------------------------------------------------ epilogue
// Warps 12-15 (thread r = TMEM lane r).  For each item, and each of its
// slots in turn: wait for the slot's last P V, read O into registers (after
// which the slot's next P V may overwrite it), normalise by the row sum and
// write the bf16 rows through the item's staging entry of the K ring (one
// 32 KiB entry, both 64-dim halves, in the layout of a TMA box: 128-byte rows,
// 16-byte chunk c of row r at chunk c ^ (r % 8)).  A warp whose 32 rows all
// belong to the sequence stores them with bulk tensor copies; a warp holding
// the sequence's end writes its rows that exist with ordinary stores.
__device__ void run_epilogue(const PrefillParams& p, const Smem& sm, const CUtensorMap* omap, int wq, int lane,
                             uint32_t tmem) {
  const int r = wq * 32 + lane;
  const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
  int kpos = 0;
  int nx[2] = {0, 0};  // items epilogued per slot
  int ne = 0;          // staging entries used
  bool pending = false;  // this warp's bulk stores may still be reading the staging rows
  for (int k = 0;; ++k) {
    if (!__all_sync(0xffffffffu, wait(sm, sm.bar(kBItFull + k % kQueue), (k / kQueue) & 1))) break;
    const Item* e = sm.item(k % kQueue);
    const int seq = e->seq, nkv = e->nkv, has_b = e->has_b;
    const int q0 = e->q0, m = e->m, n = e->n, hA = e->hA;
    if (seq < 0) break;
    kpos += nkv + (k > 0 ? 1 : 0);  // position after this item's K tiles
    // The staging entry follows the next item's first K tile in the K ring,
    // or ends the ring after the last item.
    if (!__all_sync(0xffffffffu, wait(sm, sm.bar(kBItFull + (k + 1) % kQueue), ((k + 1) / kQueue) & 1))) break;
    const int epos = sm.item((k + 1) % kQueue)->seq >= 0 ? kpos + 1 : kpos;
    __syncwarp();
    if (lane == 0) queue_release(sm, k);
    const int est = epos % kKStages;
    if (!wait_warp(sm, sm.bar(kBKFull + est), (epos / kKStages) & 1)) break;
    const uint32_t stage_off = kOffK + est * kTileBytes;
    uint8_t* stage = sm.gen + stage_off;
    const int rows_left = n - kTileM * m;  // rows of this tile inside the sequence
    const bool whole = 32 * wq + 32 <= rows_left;
    const int row0 = q0 + kTileM * m + 32 * wq;
    bool ok = true;
    for (int slot = 0; slot <= has_b && ok; ++slot) {
      if (!wait_warp(sm, sm.bar(kBODone + slot), nx[slot] & 1) ||
          !wait_warp(sm, sm.bar(kBLReady + slot), nx[slot] & 1)) {
        ok = false;
        break;
      }
      const float inv = fast_rcp(sm.lsum(slot)[r]);
      bar_arrive(sm.bar(kBLFree + slot));
      // The previous bulk stores of this warp must have read its staging rows.
      if (pending && lane == 0) bulk_wait_read();
      __syncwarp();
      tc::fence_after();
      const uint32_t o_addr = tmem + 256 + slot * 128 + lane_bits;
      // 32 columns at a time: load, normalise, pack, stage (columns 32cc..
      // 32cc+31 are 16-byte chunks 4(cc % 2) .. +3 of 64-dim half cc / 2).
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float o[32];
        tc::ld32(o_addr + 32 * cc, o);
        tc::wait_ld();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const float* v = o + 8 * c4;
          const int c8 = 4 * (cc & 1) + c4;
          *reinterpret_cast<uint4*>(stage + (cc >> 1) * kHalfBytes + r * 128 + ((c8 ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv), pack_bf16x2(v[2] * inv, v[3] * inv),
                         pack_bf16x2(v[4] * inv, v[5] * inv), pack_bf16x2(v[6] * inv, v[7] * inv));
        }
      }
      // O is in registers: the slot's next P V may overwrite it.
      tc::fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(sm.bar(kBOFree + slot));
      const int h = hA + slot;
      if (whole) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(omap, sm.sa + stage_off + wq * 32 * 128, 0, h, row0);
          tma_store_3d(omap, sm.sa + stage_off + kHalfBytes + wq * 32 * 128, 64, h, row0);
          bulk_commit();
        }
        pending = true;
      } else {
        __syncwarp();
        const int ch = lane & 15;  // 16-byte chunk of the 256-byte row
        const int64_t row_stride = static_cast<int64_t>(p.Hq) * kHeadDim;  // elements between token rows
        uint16_t* dst0 = p.out + static_cast<int64_t>(q0 + kTileM * m) * row_stride + h * kHeadDim + ch * 8;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int tr = 32 * wq + 2 * i + (lane >> 4);  // tile row written by this lane
          const uint4 v = *reinterpret_cast<const uint4*>(stage + (ch >> 3) * kHalfBytes + tr * 128 +
                                                          (((ch & 7) ^ (tr & 7)) << 4));
          if (tr < rows_left) {
            uint16_t* dst = dst0 + tr * row_stride;
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                         "r"(v.w)
                         : "memory");
          }
        }
        __syncwarp();
      }
      ++nx[slot];
    }
    if (!ok) break;
    // The staging entry goes back to the K ring once every warp's stores
    // have read it.
    if (pending && lane == 0) bulk_wait_read();
    pending = false;
    __syncwarp();
    if (lane == 0) bar_arrive(sm.bar(kBEDone));
    if (wq == 0 && lane == 0 && wait(sm, sm.bar(kBEDone), ne & 1)) {
      bar_arrive(sm.bar(kBKEmpty + est));
      bar_arrive(sm.bar(kBKEmpty + est));
    }
    __syncwarp();
    ++ne;
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

// ------------------------------------------------------------ fused KV write
// One warp per token row (like the standalone write kernel): 16-byte loads
// of the new K and V rows, 16-byte stores into the cache slot; slot -1 is
// skipped, an out-of-range slot flagged and skipped.  The stores are then
// made visible to the bulk-copy (async) proxy that the attention's loads use.
__device__ void write_new_rows(const PrefillParams& p) {
  const int warps = kThreads / 32;
  const int lane = threadIdx.x & 31;
  const int nvec = p.fw.row_elems / 8;  // 16-byte vectors per row
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < p.fw.num_tokens; t += gridDim.x * warps) {
    const int slot = __ldg(p.fw.slots + t);
    if (slot == -1) continue;
    if (slot < 0 || slot >= p.fw.num_slots) {
      if (lane == 0) atomicOr(&g_err_prefill_persistent, PKV_DEVERR_SLOT_RANGE);
      continue;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(p.fw.k_new + static_cast<int64_t>(t) * p.fw.k_stride);
    const uint4* vs = reinterpret_cast<const uint4*>(p.fw.v_new + static_cast<int64_t>(t) * p.fw.v_stride);
    uint4* kd = reinterpret_cast<uint4*>(p.fw.k_cache + static_cast<int64_t>(slot) * p.fw.row_elems);
    uint4* vd = reinterpret_cast<uint4*>(p.fw.v_cache + static_cast<int64_t>(slot) * p.fw.row_elems);
    for (int i = lane; i < nvec; i += 32) {
      const uint4 kv = __ldg(ks + i), vv = __ldg(vs + i);
      kd[i] = kv;
      vd[i] = vv;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Grid-wide barrier on the caller's two-word workspace (arrival count, epoch;
// both zero before the first call).  The last CTA to arrive resets the count
// and advances the epoch; the others wait (bounded, two seconds) for the
// epoch to move.  The launch is cooperative, so every CTA is resident.
// Returns false (flagging PKV_DEVERR_WAIT_TIMEOUT) if the wait gave up.
__device__ bool grid_barrier(unsigned int* bar, int* ok_smem) {
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned int* vb = bar;
    const unsigned int e = vb[1];
    __threadfence();
    bool ok = true;
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (vb[1] == e) {
        __nanosleep(64);
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
          atomicOr(&g_err_prefill_persistent, PKV_DEVERR_WAIT_TIMEOUT);
          ok = false;
          break;
        }
      }
    }
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    *ok_smem = ok;
  }
  __syncthreads();
  return *reinterpret_cast<volatile int*>(ok_smem) != 0;
}

__device__ __forceinline__ void regs_dec_ctl() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl)); }
__device__ __forceinline__ void regs_dec_epi() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsEpi)); }
__device__ __forceinline__ void regs_inc_softmax() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_persistent_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                   const PrefillParams p) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  sm.gen = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  sm.sa = smem_u32(sm.gen);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&omap);
    for (int i = 0; i < 2; ++i) {
      bar_init(sm.bar(kBQFull + i), 1);
      bar_init(sm.bar(kBQEmpty + i), 1);
      bar_init(sm.bar(kBSFull + i), 1);
      bar_init(sm.bar(kBSFree + i), 4);
      bar_init(sm.bar(kBPFull + i), 4);
      bar_init(sm.bar(kBPvDone + i), 1);
      bar_init(sm.bar(kBODone + i), 1);
      bar_init(sm.bar(kBOFree + i), 4);
      bar_init(sm.bar(kBDrain + i), 1);
      bar_init(sm.bar(kBEDone + i), 4);
      bar_init(sm.bar(kBLReady + i), kTileM);
      bar_init(sm.bar(kBLFree + i), kTileM);
    }
    for (int i = 0; i < kKStages; ++i) {
      bar_init(sm.bar(kBKFull + i), 1);
      bar_init(sm.bar(kBKEmpty + i), 2);  // released by each slot's S (or epilogue)
    }
    for (int i = 0; i < kVStages; ++i) {
      bar_init(sm.bar(kBVFull + i), 1);
      bar_init(sm.bar(kBVEmpty + i), 2);  // released by each slot's P V
    }
    for (int i = 0; i < kQueue; ++i) {
      bar_init(sm.bar(kBItFull + i), 1);
      bar_init(sm.bar(kBItEmpty + i), kItemReaders);
    }
    *sm.abort() = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMmaA) {
    tc::alloc(reinterpret_cast<uint32_t*>(sm.gen + kOffTmem), kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.gen + kOffTmem);
  // columns: S 0-127, P_A 128-191, P_B 192-255, O_A 256-383, O_B 384-511

  // With the write fused in: every CTA writes its share of the new rows,
  // then all wait for each other before the first cache read.
  bool run = true;
  if (p.fw.k_new) {
    write_new_rows(p);
    run = grid_barrier(p.fw.barrier, sm.abort());
    if (threadIdx.x == 0) *sm.abort() = 0;
    __syncthreads();
  }

  // Warpgroup 0 (producer, MMA issuers, scheduler) and 3 (epilogue) give
  // registers to warpgroups 1 and 2 (softmax).
  if (!run) {
    // the barrier gave up: no attention (flagged)
  } else if (warp < kWarpSoftmax) {
    regs_dec_ctl();
    if (warp == kWarpSched) {
      run_scheduler(p, sm, lane);
    } else if (warp == kWarpProducer) {
      if (lane == 0) run_producer(p, sm, &qmap, &kmap, &vmap);
    } else {
      if (lane == 0) run_issuer(sm, warp == kWarpMmaA ? 0 : 1, tmem);
    }
  } else if (warp < kWarpEpi) {
    regs_inc_softmax();
    run_softmax(p, sm, warp >= kWarpSoftmax + 4 ? 1 : 0, warp & 3, lane, tmem);
  } else {
    regs_dec_epi();
    run_epilogue(p, sm, &omap, warp & 3, lane, tmem);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kWarpMmaA) tc::dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_prefill_persistent(const PrefillArgs& a, const CacheMaps& kv, const CUtensorMap& qmap,
                                      const CUtensorMap& omap, int num_sms, cudaStream_t stream) {
  if (a.total_q == 0 || a.num_seqs == 0 || num_sms <= 0) return cudaSuccess;
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
  p.max_tiles = (a.max_seqlen_q + kTileM - 1) / kTileM;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.fw = FusedWrite{};
  if (a.k_new) {
    p.fw.k_new = a.k_new;
    p.fw.v_new = a.v_new;
    p.fw.k_stride = a.k_stride;
    p.fw.v_stride = a.v_stride;
    p.fw.slots = a.slot_mapping;
    p.fw.k_cache = a.k_cache;
    p.fw.v_cache = a.v_cache;
    p.fw.num_slots = static_cast<int64_t>(a.num_blocks) * kBlockSize;
    p.fw.num_tokens = a.total_q;
    p.fw.row_elems = a.num_kv_heads * kHeadDim;
    p.fw.barrier = a.barrier_ws;
  }
  // The warpgroups' register shares (setmaxnreg) add up to the launch's
  // total only if the kernel was built with exactly kRegsLaunch registers per
  // thread; with fewer, the softmax warpgroups' request could never be met.
  static std::atomic<int> regs_checked{0};
  if (!regs_checked.load(std::memory_order_acquire)) {
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_persistent_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidKernelImage;
    regs_checked.store(1, std::memory_order_release);
  }
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = ensure_dyn_smem(prefill_persistent_kernel, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  if (a.k_new) {
    // Fused write: one CTA per SM (the write wants every SM's bandwidth), all
    // resident at once -- a cooperative launch guarantees that or fails --
    // since every CTA waits for every other at the grid barrier.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_persistent_kernel, qmap, kv.k, kv.v, omap, p);
  }
  // One CTA per SM, or fewer when the launch bounds allow fewer items.
  const long long items = static_cast<long long>(a.num_seqs) * p.max_tiles * a.num_kv_heads * p.npairs;
  const int grid = static_cast<int>(std::min<long long>(num_sms, items));
  return launch_pdl(prefill_persistent_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, qmap, kv.k, kv.v, omap, p);
}

cudaError_t read_error_prefill_persistent(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_prefill_persistent, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_prefill_persistent, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
