// decode.cu -- paged decode attention: one query token per sequence attends
// to the sequence's cached K/V, read through its block table.
//
// Page "13. 读一个最小推理引擎：nano-vllm": section "第六站：注意力层" (decode reads
// the history K/V from the paged cache through the block table, after the new
// token's K/V has been written); section "第五站：执行准备与 KV 容量" (the cache
// layout, the slot formula, CUDA-graph pad rows).
//
// Design (GB300, sm_103a).  The step is bound by HBM: every context token
// costs 2 x num_kv_heads x head_dim x 2 bytes of K/V (4 KiB for 8 kv heads of
// 128) and only 4 x group x head_dim flops per kv head.
//
// * Work split.  All sequences' tokens are laid end to end; CTA c (one per
//   SM, persistent) takes the c-th equal share of that stream, so every SM
//   moves the same number of bytes whatever the length mix.  A sequence that
//   straddles CTAs is finished by a small combine kernel that merges the
//   per-CTA partial (max, sum, unnormalised output) triples.
// * Pipeline.  One producer warp walks its share in 16-token tiles.  A tile
//   holds the K rows (or V rows) of all kv heads of 16 consecutive tokens of
//   one 256-token cache block; it is fetched by one TMA tensor copy into a
//   3-stage shared-memory ring (64 KiB per stage with 8 kv heads), completion
//   tracked by mbarriers.  The tensor map walks (dim, token, head, dim-half,
//   block), so the 128-byte swizzled rows of one head are consecutive tokens
//   and the ldmatrix reads below are free of bank conflicts.
// * Math.  Consumer warp g handles kv head g and its group of query heads.
//   QK^T and PV use the m16n8k16 bf16 warp MMA with fp32 accumulation: the
//   group's query heads are the 16 MMA rows (rows >= group are zero), the 16
//   tokens of a tile are the columns.  The online softmax works on the MMA
//   accumulator fragments in the log2 domain (scale * log2(e) folded in),
//   with quad shuffles for the row max, and rescales the output only when
//   some row maximum moved.  Probabilities are rounded to bf16 for the PV
//   product.  The tensor work keeps the issue rate well below the HBM rate;
//   it is not what bounds the kernel.
// * Waits are bounded: a wait that exceeds two seconds sets
//   PKV_DEVERR_WAIT_TIMEOUT in the device error word and the CTA returns.
#include <cuda_runtime.h>

#include <cfloat>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_decode;

constexpr int kT = 16;          // tokens per tile (pipeline stage)
constexpr int kStages = 3;      // depth of the shared-memory ring
constexpr int kQSlots = 2;      // query staging slots (one per unit in flight)
constexpr int kMinPer = 64;     // smallest token share of one CTA
constexpr int kThreads = 32 * (kMaxKvHeads + 1);

enum : int32_t { kFirst = 1, kLast = 2, kWhole = 4 };

struct alignas(16) TileHeader {
  int32_t b;      // sequence, or -1 for "no more work"
  int32_t lo;     // unit = tokens [lo, hi) of sequence b
  int32_t hi;
  int32_t t0;     // first token of this tile (multiple of kT)
  int32_t flags;  // kFirst / kLast tile of the unit; kWhole: unit == sequence
  int32_t slot;   // partial-result slot of the unit (b + CTA index)
  int32_t pad0, pad1;
};

struct DecodeParams {
  const uint16_t* q;
  const int32_t* ctx;
  const int32_t* tables;
  uint16_t* out;
  float* ws_o;     // [slots, Hq, 128] unnormalised partial outputs
  float2* ws_ml;   // [slots, Hq] (row max in log2 units, row sum)
  int2* ws_meta;   // [B] first and last CTA holding sequence b
  int32_t maxb, B, Hq, Hkv, G, num_blocks, lmax, per_head;
  float sl2;       // scale * log2(e)
  uint32_t kv_tile_bytes;  // kT * Hkv * 256
  uint32_t stage_bytes;    // 2 * kv_tile_bytes
  uint32_t q_slot_bytes;   // Hq * 256 rounded up to 1 KiB
  // fused KV write (fuse_write != 0): new token rows and their slots
  const uint4* k_new;
  const uint4* v_new;
  int64_t k_stride_vec, v_stride_vec;  // token strides in 16-byte chunks
  const int32_t* slots;
  uint4* k_cache_w;
  uint4* v_cache_w;
  int32_t fuse_write;
};

__device__ __forceinline__ int clamp_len(int L, int lmax) {
  if (L < 0 || L > lmax) {
    atomicOr(&g_err_decode, PKV_DEVERR_LEN_RANGE);
    L = L < 0 ? 0 : lmax;
  }
  return L;
}

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

struct Smem {
  uint8_t* stages;
  uint8_t* qbuf;
  TileHeader* hdr;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* qfull;
  uint64_t* qempty;
};

__device__ __forceinline__ Smem carve(uint8_t* base, const DecodeParams& p) {
  Smem s;
  s.stages = base;
  s.qbuf = base + kStages * p.stage_bytes;
  s.hdr = reinterpret_cast<TileHeader*>(s.qbuf + kQSlots * p.q_slot_bytes);
  s.full = reinterpret_cast<uint64_t*>(s.hdr + kStages);
  s.empty = s.full + kStages;
  s.qfull = s.empty + kStages;
  s.qempty = s.qfull + kQSlots;
  return s;
}

// ------------------------------------------------------------------ producer
// Wait used only after a timeout, to let copies this CTA already issued land
// before its shared memory is given up: bounded (100 ms), reports nothing
// (the timeout has been reported).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 100000000ull) return;
}

struct ProducerState {
  uint32_t it = 0;     // tiles issued
  uint32_t units = 0;  // units started
  bool ok = true;
};

__device__ __forceinline__ int load_block(const DecodeParams& p, int b, int lb) {
  int phys = __ldg(p.tables + static_cast<int64_t>(b) * p.maxb + lb);
  if (phys < 0 || phys >= p.num_blocks) {
    atomicOr(&g_err_decode, PKV_DEVERR_BLOCK_RANGE);
    phys = 0;
  }
  return phys;
}

// Fused KV write, by the whole producer warp of the one CTA whose share holds
// position L-1 of sequence b: copy the new token's K and V rows (all kv heads)
// to its slot, then make the writes visible to this thread's later TMA reads.
// The slot must be the slot of position L-1 (the decode invariant); -1 means
// a padding row (nothing written); any other value is flagged and skipped,
// since writing elsewhere could race with other CTAs' reads.
__device__ void write_new_token(const DecodeParams& p, int b, int L, int lane) {
  // The slot, its table entry and the new rows are loaded together (one
  // round of latency on the producer's path), then checked and stored.
  constexpr int kVecsPerLane = kMaxKvHeads * kHeadDim / 8 / 32;  // 16-byte chunks of a row per lane
  const int pos = L - 1;
  const int row_vecs = p.Hkv * kHeadDim / 8;
  const int s = __ldg(p.slots + b);
  const int phys = __ldg(p.tables + static_cast<int64_t>(b) * p.maxb + pos / kBlockSize);
  const uint4* ks = p.k_new + static_cast<int64_t>(b) * p.k_stride_vec;
  const uint4* vs = p.v_new + static_cast<int64_t>(b) * p.v_stride_vec;
  uint4 kr[kVecsPerLane], vr[kVecsPerLane];
#pragma unroll
  for (int i = 0; i < kVecsPerLane; ++i) {
    const int c = lane + 32 * i;
    if (c < row_vecs) {
      kr[i] = __ldg(ks + c);
      vr[i] = __ldg(vs + c);
    }
  }
  if (s == -1) return;
  if (phys < 0 || phys >= p.num_blocks || s != phys * kBlockSize + pos % kBlockSize) {
    if (lane == 0) atomicOr(&g_err_decode, PKV_DEVERR_SLOT_RANGE);
    return;
  }
  uint4* kd = p.k_cache_w + static_cast<int64_t>(s) * row_vecs;
  uint4* vd = p.v_cache_w + static_cast<int64_t>(s) * row_vecs;
#pragma unroll
  for (int i = 0; i < kVecsPerLane; ++i) {
    const int c = lane + 32 * i;
    if (c < row_vecs) {
      kd[c] = kr[i];
      vd[c] = vr[i];
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Issue every tile of unit (b, [lo, hi)).  Lane 0 of the producer warp only.
__device__ void emit_unit(const DecodeParams& p, const Smem& sm, const CUtensorMap* kmap,
                          const CUtensorMap* vmap, ProducerState& ps, int b, int lo, int hi, int L,
                          int slot, int first_phys) {
  const int t_begin = lo & ~(kT - 1);
  int lb_cur = -1, phys = 0;
  int nxt = first_phys;  // block of token t_begin, looked up ahead by the warp
  for (int t = t_begin; t < hi && ps.ok; t += kT) {
    const int lb = t >> 8;
    if (lb != lb_cur) {
      phys = nxt;
      lb_cur = lb;
      if ((lb + 1) * kBlockSize < hi) nxt = load_block(p, b, lb + 1);  // used 16 tiles later
    }
    const uint32_t stage = ps.it % kStages;
    const uint32_t par = (ps.it / kStages) & 1u;
    if (!mbar_wait(&sm.empty[stage], par ^ 1u, &g_err_decode)) {
      ps.ok = false;
      return;
    }
    int32_t flags = 0;
    if (t == t_begin) flags |= kFirst;
    if (t + kT >= hi) flags |= kLast;
    if (lo == 0 && hi == L) flags |= kWhole;
    TileHeader h;
    h.b = b;
    h.lo = lo;
    h.hi = hi;
    h.t0 = t;
    h.flags = flags;
    h.slot = slot;
    h.pad0 = h.pad1 = 0;
    sm.hdr[stage] = h;
    if (flags & kFirst) {
      const uint32_t qs = ps.units % kQSlots;
      if (!mbar_wait(&sm.qempty[qs], ((ps.units / kQSlots) & 1u) ^ 1u, &g_err_decode)) {
        ps.ok = false;
        return;
      }
      const uint32_t qbytes = static_cast<uint32_t>(p.Hq) * kHeadDim * 2;
      mbar_arrive_expect_tx(&sm.qfull[qs], qbytes);
      bulk_g2s(sm.qbuf + qs * p.q_slot_bytes, p.q + static_cast<int64_t>(b) * p.Hq * kHeadDim, qbytes,
               &sm.qfull[qs]);
      ++ps.units;
    }
    uint8_t* kdst = sm.stages + stage * p.stage_bytes;
    uint8_t* vdst = kdst + p.kv_tile_bytes;
    mbar_arrive_expect_tx(&sm.full[stage], 2 * p.kv_tile_bytes);
    const int tin = t & (kBlockSize - 1);
    if (!p.per_head) {
      tma_load_5d(kdst, kmap, &sm.full[stage], 0, tin, 0, 0, phys);
      tma_load_5d(vdst, vmap, &sm.full[stage], 0, tin, 0, 0, phys);
    } else {
      const int slot0 = phys * kBlockSize + tin;
      for (int half = 0; half < 2; ++half)
        for (int g = 0; g < p.Hkv; ++g) {
          const uint32_t off = static_cast<uint32_t>((half * p.Hkv + g) * kT) * 128u;
          tma_load_3d(kdst + off, kmap, &sm.full[stage], half * 64, g, slot0);
          tma_load_3d(vdst + off, vmap, &sm.full[stage], half * 64, g, slot0);
        }
    }
    ++ps.it;
  }
}

__device__ void producer(const DecodeParams& p, const Smem& sm, const CUtensorMap* kmap,
                         const CUtensorMap* vmap) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    prefetch_tensormap(kmap);
    prefetch_tensormap(vmap);
  }
  // Pass 1: total tokens of the batch.
  long long total = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    int L = b < p.B ? clamp_len(__ldg(p.ctx + b), p.lmax) : 0;
    total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(L));
  }
  ProducerState ps;
  if (total > 0) {
    long long per = (total + gridDim.x - 1) / gridDim.x;
    if (per < kMinPer) per = kMinPer;
    const long long my_lo = static_cast<long long>(blockIdx.x) * per;
    const long long my_hi = my_lo + per < total ? my_lo + per : total;
    // Pass 2: the sequences overlapping [my_lo, my_hi), in order.
    long long S = 0;
    for (int base = 0; base < p.B && S < my_hi && ps.ok; base += 32) {
      const int b = base + lane;
      const int L = b < p.B ? clamp_len(__ldg(p.ctx + b), p.lmax) : 0;
      const int incl = warp_incl_scan(L, lane);
      const long long Sb = S + incl - L;
      if (L > 0 && Sb / per == blockIdx.x)
        p.ws_meta[b] = make_int2(static_cast<int>(Sb / per), static_cast<int>((Sb + L - 1) / per));
      const long long lo = my_lo > Sb ? my_lo : Sb;
      const long long hi = my_hi < Sb + L ? my_hi : Sb + L;
      const bool has = L > 0 && lo < hi;
      unsigned mask = __ballot_sync(0xffffffffu, has);
      const int lo_rel = has ? static_cast<int>(lo - Sb) : 0;
      const int hi_rel = has ? static_cast<int>(hi - Sb) : 0;
      // the first block of every piece of this batch, looked up together
      const int first_phys = has ? load_block(p, b, lo_rel >> 8) : 0;
      while (mask) {
        const int j = __ffs(mask) - 1;
        mask &= mask - 1;
        const int bj = __shfl_sync(0xffffffffu, b, j);
        const int loj = __shfl_sync(0xffffffffu, lo_rel, j);
        const int hij = __shfl_sync(0xffffffffu, hi_rel, j);
        const int Lj = __shfl_sync(0xffffffffu, L, j);
        const int physj = __shfl_sync(0xffffffffu, first_phys, j);
        if (p.fuse_write && hij == Lj) write_new_token(p, bj, Lj, lane);
        __syncwarp();
        if (lane == 0 && ps.ok) emit_unit(p, sm, kmap, vmap, ps, bj, loj, hij, Lj, bj + blockIdx.x, physj);
        ps.ok = __shfl_sync(0xffffffffu, ps.ok, 0);
        ps.it = __shfl_sync(0xffffffffu, ps.it, 0);
        ps.units = __shfl_sync(0xffffffffu, ps.units, 0);
      }
      S += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (lane == 0 && ps.ok) {
    const uint32_t stage = ps.it % kStages;
    if (mbar_wait(&sm.empty[stage], ((ps.it / kStages) & 1u) ^ 1u, &g_err_decode)) {
      sm.hdr[stage].b = -1;
      mbar_arrive(&sm.full[stage]);
    }
  }
  if (lane == 0 && !ps.ok) {
    // A wait gave up: let the copies already issued into the ring and the
    // query slots land (bounded waits on their barriers) before the CTA
    // exits and its shared memory is handed to another CTA.
    for (uint32_t i = ps.it > kStages ? ps.it - kStages : 0; i < ps.it; ++i)
      drain_wait(&sm.full[i % kStages], (i / kStages) & 1u);
    for (uint32_t u = ps.units > kQSlots ? ps.units - kQSlots : 0; u < ps.units; ++u)
      drain_wait(&sm.qfull[u % kQSlots], (u / kQSlots) & 1u);
  }
}

// ------------------------------------------------------------------ consumer
__device__ void consumer(const DecodeParams& p, const Smem& sm) {
  const int w = threadIdx.x >> 5;  // kv head
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;        // MMA row (query head within the group)
  const int cq = lane & 3;
  const int mi = lane >> 3;        // ldmatrix sub-matrix served by this lane
  const int r8 = lane & 7;
  const bool rows_hi = p.G > 8;    // MMA rows 8..15 hold real query heads

  // Per-lane byte offsets inside a K (or V) tile.  Row R of the tile is token
  // t of head g in dim-half h, R = (h * Hkv + g) * kT + t, 128 bytes per row,
  // 16-byte chunk c stored at chunk c ^ (R & 7) (TMA 128-byte swizzle).
  uint32_t koff[8];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int t = (mi >> 1) * 8 + r8;
    const int chunk = ((ks & 3) << 1) | (mi & 1);
    const int R = ((ks >> 2) * p.Hkv + w) * kT + t;
    koff[ks] = static_cast<uint32_t>(R * 128 + ((chunk ^ (R & 7)) << 4));
  }
  uint32_t voff[8];
#pragma unroll
  for (int np = 0; np < 8; ++np) {
    const int t = (mi & 1) * 8 + r8;
    const int gc = 2 * np + (mi >> 1);
    const int R = ((gc >> 3) * p.Hkv + w) * kT + t;
    voff[np] = static_cast<uint32_t>(R * 128 + (((gc & 7) ^ (R & 7)) << 4));
  }

  float acc[16][4];
  uint32_t qa[8][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float NEG_INF = -INFINITY;
  uint32_t it = 0, units = 0;
  const int hq0 = w * p.G + gq;
  const bool v0ok = gq < p.G;
  const bool v1ok = gq + 8 < p.G;

  for (;;) {
    const uint32_t stage = it % kStages;
    if (!mbar_wait(&sm.full[stage], (it / kStages) & 1u, &g_err_decode)) return;
    const TileHeader h = sm.hdr[stage];
    if (h.b < 0) return;
    if (h.flags & kFirst) {
      const uint32_t qs = units % kQSlots;
      if (!mbar_wait(&sm.qfull[qs], (units / kQSlots) & 1u, &g_err_decode)) return;
      const uint16_t* qs_ptr = reinterpret_cast<const uint16_t*>(sm.qbuf + qs * p.q_slot_bytes);
      const uint32_t* r0 = reinterpret_cast<const uint32_t*>(qs_ptr + hq0 * kHeadDim);
      const uint32_t* r1 = reinterpret_cast<const uint32_t*>(qs_ptr + (hq0 + 8) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = v0ok ? r0[ks * 8 + cq] : 0u;
        qa[ks][1] = v1ok ? r1[ks * 8 + cq] : 0u;
        qa[ks][2] = v0ok ? r0[ks * 8 + 4 + cq] : 0u;
        qa[ks][3] = v1ok ? r1[ks * 8 + 4 + cq] : 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.qempty[qs]);
      ++units;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) acc[nd][0] = acc[nd][1] = acc[nd][2] = acc[nd][3] = 0.f;
      m0 = m1 = NEG_INF;
      l0 = l1 = 0.f;
    }
    const uint32_t kb = smem_u32(sm.stages + stage * p.stage_bytes);
    const uint32_t vb = kb + p.kv_tile_bytes;

    // S = Q K^T for 16 tokens: two n-tiles of 8 tokens.
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + koff[ks], b0, b1, b2, b3);
      mma_bf16_16816(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_bf16_16816(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
    }

    // Online softmax in log2 units.  Fragment element j of n-tile n is token
    // t0 + 8n + 2cq + (j & 1) of row gq (j < 2) or gq + 8 (j >= 2).
    const int tok = h.t0 + 2 * cq;
    const bool ok00 = tok >= h.lo && tok < h.hi;
    const bool ok01 = tok + 1 >= h.lo && tok + 1 < h.hi;
    const bool ok10 = tok + 8 >= h.lo && tok + 8 < h.hi;
    const bool ok11 = tok + 9 >= h.lo && tok + 9 < h.hi;
    float x00 = ok00 ? s0[0] * p.sl2 : NEG_INF;
    float x01 = ok01 ? s0[1] * p.sl2 : NEG_INF;
    float x10 = ok10 ? s1[0] * p.sl2 : NEG_INF;
    float x11 = ok11 ? s1[1] * p.sl2 : NEG_INF;
    float mx = fmaxf(fmaxf(x00, x01), fmaxf(x10, x11));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn0 = fmaxf(m0, mx);
    const float mu0 = mn0 == NEG_INF ? 0.f : mn0;
    const float alpha0 = fast_exp2(m0 - mu0);
    const float p00 = fast_exp2(x00 - mu0), p01 = fast_exp2(x01 - mu0);
    const float p10 = fast_exp2(x10 - mu0), p11 = fast_exp2(x11 - mu0);
    l0 = l0 * alpha0 + ((p00 + p01) + (p10 + p11));
    m0 = mn0;
    uint32_t a0 = pack_bf16x2(p00, p01), a2 = pack_bf16x2(p10, p11), a1 = 0u, a3 = 0u;
    float alpha1 = 1.f;
    if (rows_hi) {
      float y00 = ok00 ? s0[2] * p.sl2 : NEG_INF;
      float y01 = ok01 ? s0[3] * p.sl2 : NEG_INF;
      float y10 = ok10 ? s1[2] * p.sl2 : NEG_INF;
      float y11 = ok11 ? s1[3] * p.sl2 : NEG_INF;
      float my = fmaxf(fmaxf(y00, y01), fmaxf(y10, y11));
      my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
      my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
      const float mn1 = fmaxf(m1, my);
      const float mu1 = mn1 == NEG_INF ? 0.f : mn1;
      alpha1 = fast_exp2(m1 - mu1);
      const float q00 = fast_exp2(y00 - mu1), q01 = fast_exp2(y01 - mu1);
      const float q10 = fast_exp2(y10 - mu1), q11 = fast_exp2(y11 - mu1);
      l1 = l1 * alpha1 + ((q00 + q01) + (q10 + q11));
      m1 = mn1;
      a1 = pack_bf16x2(q00, q01);
      a3 = pack_bf16x2(q10, q11);
    }
    if (__any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f)) {
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        acc[nd][0] *= alpha0;
        acc[nd][1] *= alpha0;
        acc[nd][2] *= alpha1;
        acc[nd][3] *= alpha1;
      }
    }

    // O += P V: 16 n-tiles of 8 dims, one k-step of 16 tokens.
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t v0, v1, v2, v3;
      ldsm_x4_trans(vb + voff[np], v0, v1, v2, v3);
      mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, v0, v1);
      mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, v2, v3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);

    if (h.flags & kLast) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      if (h.flags & kWhole) {
        const float inv0 = 1.f / l0, inv1 = 1.f / l1;
        uint16_t* o0 = p.out + (static_cast<int64_t>(h.b) * p.Hq + hq0) * kHeadDim + 2 * cq;
        uint16_t* o1 = o0 + 8 * kHeadDim;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
          if (v0ok) *reinterpret_cast<uint32_t*>(o0 + 8 * nd) = pack_bf16x2(acc[nd][0] * inv0, acc[nd][1] * inv0);
          if (v1ok) *reinterpret_cast<uint32_t*>(o1 + 8 * nd) = pack_bf16x2(acc[nd][2] * inv1, acc[nd][3] * inv1);
        }
      } else {
        float* o0 = p.ws_o + (static_cast<int64_t>(h.slot) * p.Hq + hq0) * kHeadDim + 2 * cq;
        float* o1 = o0 + 8 * kHeadDim;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
          if (v0ok) *reinterpret_cast<float2*>(o0 + 8 * nd) = make_float2(acc[nd][0], acc[nd][1]);
          if (v1ok) *reinterpret_cast<float2*>(o1 + 8 * nd) = make_float2(acc[nd][2], acc[nd][3]);
        }
        if (cq == 0) {
          float2* ml = p.ws_ml + static_cast<int64_t>(h.slot) * p.Hq + hq0;
          if (v0ok) ml[0] = make_float2(m0, l0);
          if (v1ok) ml[8] = make_float2(m1, l1);
        }
      }
    }
    ++it;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  const Smem sm = carve(base, p);
  const int warp = threadIdx.x >> 5;
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], p.Hkv);
    }
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(&sm.qfull[s], 1);
      mbar_init(&sm.qempty[s], p.Hkv);
    }
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == p.Hkv)
    producer(p, sm, &kmap, &vmap);
  else if (warp < p.Hkv)
    consumer(p, sm);
}

// Merge the per-CTA partials of sequences that straddle CTAs; zero pad rows.
// One warp per (sequence, query head); lane i handles dims 4i .. 4i+3.
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(32 * kCombineWarps) decode_combine_kernel(const DecodeParams p, int grid) {
  griddep_wait();
  griddep_launch_dependents();
  const int pair = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (pair >= p.B * p.Hq) return;
  const int b = pair / p.Hq, hq = pair - b * p.Hq;
  const int lane = threadIdx.x & 31;
  // The length and the CTA range are requested together (the range is only
  // read when the length is positive, i.e. when the decode kernel wrote it).
  const int L_in = __ldg(p.ctx + b);
  const int2 meta = p.ws_meta[b];
  const int L = clamp_len(L_in, p.lmax);
  uint16_t* o = p.out + static_cast<int64_t>(pair) * kHeadDim + 4 * lane;
  if (L == 0) {
    *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
    return;
  }
  const int c0 = max(0, meta.x), c1 = min(grid - 1, meta.y);
  if (c1 <= c0) return;  // finished inside one CTA
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c) M = fmaxf(M, p.ws_ml[static_cast<int64_t>(b + c) * p.Hq + hq].x);
  float lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = c0; c <= c1; ++c) {
    const int64_t row = static_cast<int64_t>(b + c) * p.Hq + hq;
    const float2 ml = p.ws_ml[row];
    const float wgt = fast_exp2(ml.x - M);
    const float4 v = *reinterpret_cast<const float4*>(p.ws_o + row * kHeadDim + 4 * lane);
    lsum += wgt * ml.y;
    acc.x += wgt * v.x;
    acc.y += wgt * v.y;
    acc.z += wgt * v.z;
    acc.w += wgt * v.w;
  }
  const float inv = 1.f / lsum;
  *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

size_t align256(size_t x) { return (x + 255) & ~size_t{255}; }

struct WsLayout {
  size_t o, ml, meta, total;
};

WsLayout ws_layout(int batch, int num_q_heads, int grid) {
  const size_t slots = static_cast<size_t>(batch) + grid;
  WsLayout l;
  l.o = 0;
  l.ml = align256(slots * num_q_heads * kHeadDim * sizeof(float));
  l.meta = l.ml + align256(slots * num_q_heads * sizeof(float2));
  l.total = l.meta + align256(static_cast<size_t>(batch) * sizeof(int2));
  return l;
}

}  // namespace

int decode_grid(int num_sms) { return num_sms; }

size_t decode_workspace_bytes(int batch, int num_q_heads, int num_sms) {
  return ws_layout(batch, num_q_heads, decode_grid(num_sms)).total;
}

cudaError_t launch_paged_attn_decode(const DecodeArgs& a, const CacheMaps& maps, int num_sms,
                                     cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  const int grid = decode_grid(num_sms);
  const WsLayout wl = ws_layout(a.batch, a.num_q_heads, grid);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  DecodeParams p;
  p.q = a.q;
  p.ctx = a.context_lens;
  p.tables = a.block_tables;
  p.out = a.out;
  p.ws_o = reinterpret_cast<float*>(ws + wl.o);
  p.ws_ml = reinterpret_cast<float2*>(ws + wl.ml);
  p.ws_meta = reinterpret_cast<int2*>(ws + wl.meta);
  p.maxb = a.max_blocks_per_seq;
  p.B = a.batch;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.G = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  const long long cap = static_cast<long long>(a.max_blocks_per_seq) * kBlockSize;
  p.lmax = static_cast<int>(a.max_context_len < cap ? a.max_context_len : cap);
  p.per_head = maps.per_head;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.kv_tile_bytes = static_cast<uint32_t>(kT * a.num_kv_heads * kHeadDim * 2);
  p.stage_bytes = 2 * p.kv_tile_bytes;
  p.q_slot_bytes = static_cast<uint32_t>((a.num_q_heads * kHeadDim * 2 + 1023) & ~1023);
  p.fuse_write = a.k_new != nullptr;
  p.k_new = reinterpret_cast<const uint4*>(a.k_new);
  p.v_new = reinterpret_cast<const uint4*>(a.v_new);
  p.k_stride_vec = a.k_stride / 8;
  p.v_stride_vec = a.v_stride / 8;
  p.slots = a.slot_mapping;
  p.k_cache_w = reinterpret_cast<uint4*>(a.k_cache);
  p.v_cache_w = reinterpret_cast<uint4*>(a.v_cache);
  const size_t smem = 1024 + kStages * p.stage_bytes + kQSlots * p.q_slot_bytes +
                      kStages * sizeof(TileHeader) + (2 * kStages + 2 * kQSlots) * sizeof(uint64_t);
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = ensure_dyn_smem(decode_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_kernel, dim3(grid), dim3(32 * (a.num_kv_heads + 1)), smem, stream, maps.k, maps.v, p);
  if (e != cudaSuccess) return e;
  const int pairs = a.batch * a.num_q_heads;
  return launch_pdl(decode_combine_kernel, dim3((pairs + kCombineWarps - 1) / kCombineWarps),
                    dim3(32 * kCombineWarps), 0, stream, p, grid);
}

cudaError_t read_error_decode(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_decode, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_decode, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
