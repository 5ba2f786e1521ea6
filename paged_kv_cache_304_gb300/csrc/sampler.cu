// sampler.cu -- exponential-race (temperature) sampling of the next token.
//
// Page "13. 读一个最小推理引擎：nano-vllm", section "其余部分": the sampler
// supports temperature only (temperature 0 is not allowed); instead of a
// multinomial draw it divides the probabilities by exponentially distributed
// random numbers and takes the largest quotient, which samples each token
// with its probability.
//
// With p = softmax(l / T) and E_i = -ln(U_i), argmax_i p_i / E_i is the argmax
// of the monotone transform  key_i = l_i * log2(e) / T - log2(-log2 U_i)
// (the softmax normaliser and the constant log2(ln 2) drop out), so no
// softmax pass is needed: one streaming pass over the logits.
//
// Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC 2011).  Token i of row b uses output word
// i % 4 of Philox(counter = {i / 4, b, offset_lo, offset_hi},
// key = {seed_lo, seed_hi}); U = ((word >> 9) + 0.5) / 2^23 in (0, 1).
//
// Kernels: a grid of (8192-token chunk, row) CTAs streams the logits with
// 16-byte loads (all of a thread's loads issued first), generates the noise
// in registers and reduces (key, index) to one partial per chunk (ties go to
// the smaller index); a second kernel (one warp per row) reduces the
// partials.  The pass moves 4 bytes of logits per token; at a Qwen3-sized
// vocabulary it is bound by instruction issue (a quarter Philox block and
// two logarithms per token) rather than by HBM.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ unsigned int g_err_sampler;

constexpr int kChunk = 8192;
constexpr int kThreads = 256;  // 32 tokens per thread

struct SampleParams {
  const float* logits;
  int64_t row_stride;
  const float* temps;
  int32_t B, V, nchunks, vec4;
  uint32_t seed_lo, seed_hi, off_lo, off_hi;
  float2* ws;  // [B, nchunks]: (key, index bits)
  int32_t* out;
};

__device__ __forceinline__ uint32_t mulhi(uint32_t a, uint32_t b) { return __umulhi(a, b); }

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = mulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = mulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Race key of one token: l * log2(e) / T - log2(-log2(U)), with
// U = ((word >> 9) + 0.5) / 2^23 built from the float with exponent 0 and the
// top 23 bits of the word as mantissa ([1, 2)), minus 1 - 2^-24 (exact).
__device__ __forceinline__ float race_key(float l, float scale, uint32_t word) {
  const float u = __uint_as_float(0x3F800000u | (word >> 9)) - 0.99999994039535522f;
  return l * scale - fast_log2(-fast_log2(u));
}

// Within one thread tokens arrive in increasing index order, so a later token
// replaces the current best only if its key is strictly larger.
__device__ __forceinline__ void better_in_order(float& bk, int& bi, float k, int i) {
  if (k > bk) {
    bk = k;
    bi = i;
  }
}

__device__ __forceinline__ void better(float& bk, int& bi, float k, int i) {
  if (k > bk || (k == bk && i < bi)) {
    bk = k;
    bi = i;
  }
}

// 64 registers per thread (4 CTAs per SM) hold the eight logit quads in flight.
__global__ void __launch_bounds__(kThreads, 4) sample_chunk_kernel(const SampleParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x / p.nchunks;
  const int chunk = blockIdx.x - b * p.nchunks;
  const float T = __ldg(p.temps + b);
  float bk = -INFINITY;
  int bi = 0x7fffffff;
  if (T > 0.f && T < INFINITY) {
    const float scale = 1.4426950408889634f / T;
    const float* row = p.logits + static_cast<int64_t>(b) * p.row_stride;
    const int base = chunk * kChunk;
    // All of this thread's logits are requested before any noise is drawn,
    // so the loads overlap each other and the Philox arithmetic.
    constexpr int kQuads = kChunk / (4 * kThreads);
    float4 lv[kQuads];
    if (p.vec4) {
#pragma unroll
      for (int j = 0; j < kQuads; ++j) {
        const int i = base + 4 * (threadIdx.x + j * kThreads);
        lv[j] = i + 3 < p.V ? __ldg(reinterpret_cast<const float4*>(row + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int j = 0; j < kChunk / (4 * kThreads); ++j) {
      const int i = base + 4 * (threadIdx.x + j * kThreads);  // first token of this quad
      if (i >= p.V) break;
      const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(i >> 2), static_cast<uint32_t>(b), p.off_lo,
                                               p.off_hi),
                                    p.seed_lo, p.seed_hi);
      if (p.vec4 && i + 3 < p.V) {
        const float4 l = lv[j];
        better_in_order(bk, bi, race_key(l.x, scale, w.x), i);
        better_in_order(bk, bi, race_key(l.y, scale, w.y), i + 1);
        better_in_order(bk, bi, race_key(l.z, scale, w.z), i + 2);
        better_in_order(bk, bi, race_key(l.w, scale, w.w), i + 3);
      } else {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (i + q < p.V) better_in_order(bk, bi, race_key(__ldg(row + i + q), scale, ws[q]), i + q);
      }
    }
  }
  // CTA reduction of (key, index)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float k = __shfl_xor_sync(0xffffffffu, bk, o);
    const int i = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bk, bi, k, i);
  }
  __shared__ float sk[kThreads / 32];
  __shared__ int si[kThreads / 32];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sk[wid] = bk;
    si[wid] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kThreads / 32; ++k) better(bk, bi, sk[k], si[k]);
    p.ws[static_cast<int64_t>(b) * p.nchunks + chunk] = make_float2(bk, __int_as_float(bi));
  }
}

__global__ void __launch_bounds__(256) sample_reduce_kernel(const SampleParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= p.B) return;
  float bk = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = lane; c < p.nchunks; c += 32) {
    const float2 v = p.ws[static_cast<int64_t>(b) * p.nchunks + c];
    better(bk, bi, v.x, __float_as_int(v.y));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float k = __shfl_xor_sync(0xffffffffu, bk, o);
    const int i = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bk, bi, k, i);
  }
  if (lane == 0) {
    const float T = __ldg(p.temps + b);
    const bool ok = T > 0.f && T < INFINITY && bi != 0x7fffffff;
    if (!ok) atomicOr(&g_err_sampler, PKV_DEVERR_LEN_RANGE);
    p.out[b] = ok ? bi : -1;
  }
}

}  // namespace

size_t sample_workspace_bytes(int batch, int vocab) {
  const size_t nchunks = (static_cast<size_t>(vocab) + kChunk - 1) / kChunk;
  return ((static_cast<size_t>(batch) * nchunks * sizeof(float2)) + 255) & ~size_t{255};
}

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t stream) {
  SampleParams p;
  p.logits = a.logits;
  p.row_stride = a.row_stride;
  p.temps = a.temperatures;
  p.B = a.batch;
  p.V = a.vocab;
  p.nchunks = (a.vocab + kChunk - 1) / kChunk;
  p.vec4 = (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) && (a.row_stride % 4 == 0);
  p.seed_lo = static_cast<uint32_t>(a.seed);
  p.seed_hi = static_cast<uint32_t>(a.seed >> 32);
  p.off_lo = static_cast<uint32_t>(a.offset);
  p.off_hi = static_cast<uint32_t>(a.offset >> 32);
  p.ws = static_cast<float2*>(a.workspace);
  p.out = a.out;
  const int64_t ctas = static_cast<int64_t>(p.nchunks) * a.batch;  // (row, chunk), chunk fastest
  if (ctas >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(sample_chunk_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_reduce_kernel, dim3((a.batch + 7) / 8), dim3(256), 0, stream, p);
}

cudaError_t read_error_sampler(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_err_sampler, sizeof v);
  if (e != cudaSuccess) return e;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_sampler, &zero, sizeof zero);
  }
  return e;
}

}  // namespace pkv
