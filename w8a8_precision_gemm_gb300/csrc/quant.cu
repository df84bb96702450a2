// quant.cu -- the memory-bound kernels of the W8A8 path:
//   * per-token activation quantization (optionally with a UAQ pre-scale),
//   * RMSNorm with the UAQ-folded gain -> per-token quantization,
//   * SiLU(gate) * up -> per-token quantization,
//   * UAQ weight fold W' = W/s + per-output-channel weight quantization,
//   * gain fold gamma' = gamma * s,
//   * code-flip count of two code buffers.
//
// Method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
// Quantized Rollout", sections "更新感知量化 (UAQ)" (W X = (W/s)(sX), s folded
// into the norm gain) and "损失函数 / 训练策略" (per-channel weight and
// per-token activation INT8/FP8 quantization, s = 1.5).
//
// Every row (token or output channel) is one CTA: 16-byte vector loads, the
// row cached in registers between the absmax pass and the code pass, a
// warp-shuffle + shared-memory block reduction.  Arithmetic that decides a
// code is IEEE fp32 with explicit rounding intrinsics (no contraction):
//   scale = absmax / qmax (absmax == 0 -> 1);  code = RNE(v / scale)
//   clamped to +-127 (INT8), or e4m3 RNE with saturation (FP8).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace qurl {
namespace {

constexpr int kVPT = 8;           // 16-byte vectors cached per thread
constexpr int kRowThreads = 512;  // most threads of a row CTA (register budget of the row kernels)

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Block-wide reduction (max or sum); every thread gets the result.
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = kMax ? warp_max(v) : warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < nw ? red[lane] : 0.0f;
    t = kMax ? warp_max(t) : warp_sum(t);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  const float r = red[32];
  __syncthreads();
  return r;
}

// s + c += y without rounding error in the pair (two-sum of s and y; the
// rounding error goes to c).
__device__ __forceinline__ void two_sum_acc(float& s, float& c, float y) {
  const float t = __fadd_rn(s, y);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(y, bp));
  s = t;
  c = __fadd_rn(c, err);
}

// The row's mean of squares ms = (s + c) / K (the compensated block sum of
// x^2, divided in fp64 and rounded to fp32) and r = 1 / sqrt(ms + eps)
// (correctly rounded fp32 square root and division), computed by one thread
// and handed to every thread of the block.
__device__ __forceinline__ void block_mean_sq(float s, float c, float* red, int K, float eps, float& ms, float& r) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float oc = __shfl_xor_sync(0xFFFFFFFFu, c, o);
    two_sum_acc(s, c, os);
    c = __fadd_rn(c, oc);
  }
  if (lane == 0) {
    red[2 * warp] = s;
    red[2 * warp + 1] = c;
  }
  __syncthreads();
  if (warp == 0) {
    float ts = lane < nw ? red[2 * lane] : 0.0f;
    float tc = lane < nw ? red[2 * lane + 1] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xFFFFFFFFu, ts, o);
      const float oc = __shfl_xor_sync(0xFFFFFFFFu, tc, o);
      two_sum_acc(ts, tc, os);
      tc = __fadd_rn(tc, oc);
    }
    if (lane == 0) {
      const float m = static_cast<float>((static_cast<double>(ts) + static_cast<double>(tc)) / static_cast<double>(K));
      red[64] = m;
      red[65] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(m, eps)));
    }
  }
  __syncthreads();
  ms = red[64];
  r = red[65];
  __syncthreads();
}

__device__ __forceinline__ float row_scale(float amax, int qt) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, qt == kQInt8 ? 127.0f : 448.0f);
}

// A row's quantization step: the scale and, for INT8, its reciprocal.
struct Enc {
  float scale;
  float inv;
  int qt;
};

__device__ __forceinline__ Enc make_enc(float amax, int qt) {
  const float scale = row_scale(amax, qt);
  return {scale, __frcp_rn(scale), qt};
}

// Code of v / scale.  Both types are decided on the IEEE quotient fl(v /
// scale), but most codes come from the product r = v * fl(1 / scale) instead:
// r carries two roundings of relative size 2^-24 on top of the exact quotient,
// so it lies within 2.5 units in the last place of fl(v / scale).
//  * INT8: fl(v / scale) rounded to the nearest integer, ties to even, clamped
//    to +-127.  For |r| < 256 r is within 5e-5 of the quotient, so wherever r
//    is more than 1e-4 away from a half-integer both round to the same integer
//    and r is used; otherwise (one code in ~5000, and NaN or out-of-range
//    inputs) the quotient itself is computed.
//  * FP8-E4M3: round to nearest even with saturation to +-448.  For magnitudes
//    of at least 2^-6 (e4m3's normal range) the code keeps 3 of fp32's 23
//    fraction bits, so r and the quotient give the same code unless the 20
//    dropped bits of r lie within 8 units of the halfway pattern 0x80000; then,
//    and below 2^-6 (e4m3 subnormals round at another bit) or for non-finite
//    r, the quotient itself is computed.
// The codes are therefore those of the plain division.
__device__ __forceinline__ uint8_t encode(float v, const Enc& e) {
  const float r = __fmul_rn(v, e.inv);
  if (e.qt == kQInt8) {
    const float f = r - floorf(r);
    const bool fast = fabsf(r) < 256.0f && fabsf(f - 0.5f) > 1e-4f;
    int q = __float2int_rn(fast ? r : __fdiv_rn(v, e.scale));
    q = max(-127, min(127, q));
    return static_cast<uint8_t>(static_cast<int8_t>(q));
  }
  const uint32_t b = __float_as_uint(r) & 0x7FFFFFFFu;
  const bool fast = b >= 0x3C800000u && b < 0x7F800000u && ((b & 0xFFFFFu) - 0x7FFF8u) > 16u;
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(fast ? r : __fdiv_rn(v, e.scale), __NV_SATFINITE, __NV_E4M3));
}

// 8 values -> 8 code bytes packed in a uint2 (little-endian byte order = k order).
__device__ __forceinline__ uint2 encode8(const float (&v)[8], const Enc& en) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) lo |= static_cast<uint32_t>(encode(v[e], en)) << (8 * e);
#pragma unroll
  for (int e = 0; e < 4; ++e) hi |= static_cast<uint32_t>(encode(v[4 + e], en)) << (8 * e);
  return make_uint2(lo, hi);
}

// Saturation of the sums of |code| (any value above 2^24 / 128 means
// "accumulate in chunks" to the GEMM that reads them).
constexpr int kAbsSumCap = 1 << 24;

// Store 8 codes (and, for INT8 when x16 is given, the same 8 codes as fp16 --
// exact, integers of magnitude <= 127 -- for the tensor-core GEMM to read).
// Returns the sum of |code| and the sum of code^2 of the 8 INT8 codes when x16
// is given, else zeros.
__device__ __forceinline__ int2 store8(uint8_t* __restrict__ q, uint8_t* __restrict__ x16, size_t idx,
                                       const float (&v)[8], const Enc& en) {
  const uint2 c = encode8(v, en);
  reinterpret_cast<uint2*>(q)[idx] = c;
  if (x16 == nullptr) return make_int2(0, 0);
  {
    // the same 8 codes as fp16, exactly: with u = c + 128 in [0, 255], the
    // fp16 with bits 0x6400 | u is 1024 + u, and subtracting 1152 leaves c
    const uint32_t w[2] = {c.x ^ 0x80808080u, c.y ^ 0x80808080u};
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t p = __byte_perm(w[e >> 1], 0x64646464u, (e & 1) ? 0x4342 : 0x4140);
      const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&p), bias);
      h[e] = *reinterpret_cast<const uint32_t*>(&d);
    }
    reinterpret_cast<uint4*>(x16)[idx] = make_uint4(h[0], h[1], h[2], h[3]);
  }
  const int a = static_cast<int>(__dp4a(__vabs4(c.y), 0x01010101u, __dp4a(__vabs4(c.x), 0x01010101u, 0u)));
  const int sq = __dp4a(static_cast<int>(c.y), static_cast<int>(c.y), __dp4a(static_cast<int>(c.x),
                                                                              static_cast<int>(c.x), 0));
  return make_int2(a, sq);
}

// Per-row sums of |code| (and of code^2) over the ranges of a CodeSums, in
// shared-memory counters cnt[0, kMaxSums) and cnt[kMaxSums, 2 kMaxSums): one
// atomic per warp, step and sum (the 32 vectors of 8 codes a warp visits in
// one step lie in one range, as ranges are multiples of 256 codes).
// sums_begin zeroes the counters; the block reductions that follow in every
// kernel order it before the first sums_add_warp.
__device__ __forceinline__ void sums_begin(unsigned long long* cnt, const CodeSums& cs) {
  if (cs.asum != nullptr)
    for (int j = threadIdx.x; j < cs.nsum; j += blockDim.x) cnt[j] = cnt[kMaxSums + j] = 0;
}

// Called by all 32 lanes of the warp; idx: this lane's vector; v: its sums (0 if none).
__device__ __forceinline__ void sums_add_warp(unsigned long long* cnt, const CodeSums& cs, int idx, int2 v) {
  if (cs.asum == nullptr) return;
  const unsigned s = __reduce_add_sync(0xFFFFFFFFu, static_cast<unsigned>(v.x));
  const unsigned q = cs.qsum ? __reduce_add_sync(0xFFFFFFFFu, static_cast<unsigned>(v.y)) : 0u;
  if ((threadIdx.x & 31) == 0) {
    const int r = (idx * 8) / cs.sum_len;
    if (s != 0) atomicAdd(&cnt[r], static_cast<unsigned long long>(s));
    if (q != 0) atomicAdd(&cnt[kMaxSums + r], static_cast<unsigned long long>(q));
  }
}

__device__ __forceinline__ void sums_end(unsigned long long* cnt, const CodeSums& cs, int m) {
  if (cs.asum == nullptr) return;
  __syncthreads();
  for (int j = threadIdx.x; j < cs.nsum; j += blockDim.x) {
    cs.asum[static_cast<size_t>(m) * cs.nsum + j] =
        static_cast<int>(cnt[j] < static_cast<unsigned long long>(kAbsSumCap) ? cnt[j] : kAbsSumCap);
    if (cs.qsum)
      cs.qsum[static_cast<size_t>(m) * cs.nsum + j] =
          static_cast<unsigned>(cnt[kMaxSums + j] < 0xFFFFFFFFull ? cnt[kMaxSums + j] : 0xFFFFFFFFull);
  }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// Visit the 16-byte vectors idx = threadIdx.x + c * blockDim.x of a row: the
// first kVPT from the register cache (fully unrolled, so the cache stays in
// registers), the rest (rows longer than kVPT * blockDim vectors) from memory.
template <int NC, typename F>
__device__ __forceinline__ void for_vectors(const uint4* row, int nvec, const uint4 (&cache)[NC], F&& f) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    if (idx < nvec) f(cache[c], idx);
  }
  for (int idx = threadIdx.x + NC * blockDim.x; idx < nvec; idx += blockDim.x) f(__ldg(row + idx), idx);
}

// The same vectors, visited warp-uniformly: every lane calls f(u, idx, valid)
// in every step of its warp (u is undefined where !valid), so f may use warp
// collectives.  blockDim.x is a multiple of 32.
template <int NC, typename F>
__device__ __forceinline__ void for_vectors_warp(const uint4* row, int nvec, const uint4 (&cache)[NC], F&& f) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    f(cache[c], idx, idx < nvec);
  }
  for (int i0 = NC * blockDim.x + (threadIdx.x & ~31); i0 < nvec; i0 += blockDim.x) {
    const int idx = i0 + (threadIdx.x & 31);
    const bool valid = idx < nvec;
    f(valid ? __ldg(row + idx) : make_uint4(0, 0, 0, 0), idx, valid);
  }
}

template <int NC>
__device__ __forceinline__ void fill_cache(const uint4* row, int nvec, uint4 (&cache)[NC]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    if (idx < nvec) cache[c] = __ldg(row + idx);
  }
}

// ------------------------------------------------------------------ activation quant

__global__ void __launch_bounds__(kRowThreads) quant_act_kernel(const __nv_bfloat16* __restrict__ X, int K, long long ldx, float pre, int qt,
                                 uint8_t* __restrict__ Xq, float* __restrict__ sx, uint8_t* __restrict__ x16,
                                 const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[33];
  __shared__ unsigned long long cnt[2 * kMaxSums];
  sums_begin(cnt, sums);
  const int m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * ldx);
  const int nvec = K >> 3;
  uint4 cache[kVPT];
  fill_cache(row, nvec, cache);
  float amax = 0.0f;
  for_vectors(row, nvec, cache, [&](const uint4 u, int) {
    float x[8];
    bf16x8_to_f32(u, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(__fmul_rn(x[e], pre)));
  });
  amax = block_reduce<true>(amax, red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sx[m] = en.scale;
  uint8_t* out = Xq + static_cast<size_t>(m) * K;
  uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * K * 2 : nullptr;
  for_vectors_warp(row, nvec, cache, [&](const uint4 u, int idx, bool valid) {
    int2 v = make_int2(0, 0);
    if (valid) {
      float x[8];
      bf16x8_to_f32(u, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(x[e], pre);
      v = store8(out, out16, idx, x, en);
    }
    sums_add_warp(cnt, sums, idx, v);
  });
  sums_end(cnt, sums, m);
}

// ------------------------------------------------------------------ RMSNorm -> quant

__global__ void __launch_bounds__(kRowThreads) rmsnorm_quant_kernel(const __nv_bfloat16* __restrict__ X, int K, long long ldx,
                                     const float* __restrict__ gamma, float eps, int qt, uint8_t* __restrict__ Xq,
                                     float* __restrict__ sx, float* __restrict__ ms_out, uint8_t* __restrict__ x16,
                                     const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[66];
  __shared__ unsigned long long cnt[2 * kMaxSums];
  sums_begin(cnt, sums);
  const int m = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * ldx);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  const int nvec = K >> 3;
  uint4 cache[kVPT];
  fill_cache(row, nvec, cache);
  // mean of squares.  Each x^2 is exact in fp32 (a bf16 has an 8-bit
  // significand); the sum is carried as an unevaluated pair s + c (error-free
  // two-sum per term, Knuth) and divided by K in fp64, so ms is the fp32
  // rounding of the mean to within ~2^-44 relative -- the same fp32 value a
  // plain fp64 sum gives, except when the mean lies that close to a rounding
  // midpoint.
  float ss = 0.0f, sc = 0.0f;
  for_vectors(row, nvec, cache, [&](const uint4 u, int) {
    float x[8];
    bf16x8_to_f32(u, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) two_sum_acc(ss, sc, __fmul_rn(x[e], x[e]));
  });
  // the gain of the vectors this thread normalises is read while the sums are reduced
#pragma unroll
  for (int c = 0; c < kVPT; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    if (idx < nvec) asm volatile("prefetch.global.L1 [%0];" ::"l"(g4 + 2 * idx));
  }
  float ms, r;
  block_mean_sq(ss, sc, red, K, eps, ms, r);
  if (threadIdx.x == 0 && ms_out) ms_out[m] = ms;
  // v = (x * r) * gamma'
  auto normed = [&](const uint4 u, int idx, float (&x)[8]) {
    bf16x8_to_f32(u, x);
    const float4 ga = __ldg(g4 + 2 * idx), gb = __ldg(g4 + 2 * idx + 1);
    const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(__fmul_rn(x[e], r), g[e]);
  };
  float amax = 0.0f;
  for_vectors(row, nvec, cache, [&](const uint4 u, int idx) {
    float x[8];
    normed(u, idx, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
  });
  amax = block_reduce<true>(amax, red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sx[m] = en.scale;
  uint8_t* out = Xq + static_cast<size_t>(m) * K;
  uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * K * 2 : nullptr;
  for_vectors_warp(row, nvec, cache, [&](const uint4 u, int idx, bool valid) {
    int2 v = make_int2(0, 0);
    if (valid) {
      float x[8];
      normed(u, idx, x);
      v = store8(out, out16, idx, x, en);
    }
    sums_add_warp(cnt, sums, idx, v);
  });
  sums_end(cnt, sums, m);
}

// ------------------------------------------------------------------ SiLU * up -> quant

__device__ __forceinline__ void silu_mul8(const uint4 gu, const uint4 uu, float (&h)[8]) {
  float g[8], u[8];
  bf16x8_to_f32(gu, g);
  bf16x8_to_f32(uu, u);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    // g / (1 + exp(-g)) to within ~2 units in the last place (h is held to a
    // relative 2e-6 of the exact value; the codes are decided on this h).  A
    // denominator beyond 2^126 (g < -87.3) makes |h| < 2e-36: 0.
    const float den = __fadd_rn(1.0f, expf(-g[e]));
    const float sg = den < 0x1p126f ? __fdividef(g[e], den) : 0.0f;
    h[e] = __fmul_rn(sg, u[e]);
  }
}

// MINB = 2: two blocks per SM (at most 64 registers a thread) when there are
// more rows than SMs, so a batch of up to two rows per SM runs as one wave.
template <int MINB>
__global__ void __launch_bounds__(kRowThreads, MINB) silu_mul_quant_kernel(const __nv_bfloat16* __restrict__ GU, int I, long long ldgu, float pre,
                                      int qt, uint8_t* __restrict__ Xq, float* __restrict__ sx,
                                      float* __restrict__ h_out, uint8_t* __restrict__ x16,
                                      const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[33];
  __shared__ unsigned long long cnt[2 * kMaxSums];
  sums_begin(cnt, sums);
  const int m = blockIdx.x;
  const uint4* grow = reinterpret_cast<const uint4*>(GU + static_cast<size_t>(m) * ldgu);
  const uint4* urow = reinterpret_cast<const uint4*>(GU + static_cast<size_t>(m) * ldgu + I);
  const int nvec = I >> 3;
  uint4 cg[kVPT / 2], cu[kVPT / 2];
  fill_cache(grow, nvec, cg);
  fill_cache(urow, nvec, cu);
  // pass 1: h = silu(g) * u, kept in registers for the cached positions
  float hc[kVPT / 2][8];
  float amax = 0.0f;
  auto take = [&](const float (&h)[8], int idx) {
    if (h_out) {
      float4* ho = reinterpret_cast<float4*>(h_out + static_cast<size_t>(m) * I) + 2 * idx;
      ho[0] = make_float4(h[0], h[1], h[2], h[3]);
      ho[1] = make_float4(h[4], h[5], h[6], h[7]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(__fmul_rn(h[e], pre)));
  };
#pragma unroll
  for (int c = 0; c < kVPT / 2; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    if (idx < nvec) {
      silu_mul8(cg[c], cu[c], hc[c]);
      take(hc[c], idx);
    }
  }
  for (int idx = threadIdx.x + (kVPT / 2) * blockDim.x; idx < nvec; idx += blockDim.x) {
    float h[8];
    silu_mul8(__ldg(grow + idx), __ldg(urow + idx), h);
    take(h, idx);
  }
  amax = block_reduce<true>(amax, red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sx[m] = en.scale;
  uint8_t* out = Xq + static_cast<size_t>(m) * I;
  uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * I * 2 : nullptr;
  // pass 2: codes (warp-uniform steps, see for_vectors_warp)
  auto put = [&](float (&h)[8], int idx, bool valid) {
    int2 v = make_int2(0, 0);
    if (valid) {
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = __fmul_rn(h[e], pre);
      v = store8(out, out16, idx, h, en);
    }
    sums_add_warp(cnt, sums, idx, v);
  };
#pragma unroll
  for (int c = 0; c < kVPT / 2; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    put(hc[c], idx, idx < nvec);
  }
  for (int i0 = (kVPT / 2) * blockDim.x + (threadIdx.x & ~31); i0 < nvec; i0 += blockDim.x) {
    const int idx = i0 + (threadIdx.x & 31);
    float h[8] = {};
    if (idx < nvec) silu_mul8(__ldg(grow + idx), __ldg(urow + idx), h);
    put(h, idx, idx < nvec);
  }
  sums_end(cnt, sums, m);
}

// ------------------------------------------------------------------ weight fold + quant

// Loads 8 consecutive weights of a row as fp32 (bf16 or fp32 storage).
template <bool kF32>
__device__ __forceinline__ void load_w8(const void* row, int idx, float (&w)[8]) {
  if (kF32) {
    const float4* p = reinterpret_cast<const float4*>(row) + 2 * idx;
    const float4 a = __ldg(p), b = __ldg(p + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else {
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(row) + idx), w);
  }
}

template <bool kF32>
__global__ void __launch_bounds__(kRowThreads) prepare_weights_kernel(const void* __restrict__ W, int K, long long ldw, float s, int qt,
                                       uint8_t* __restrict__ Wq, float* __restrict__ sw, float* W_scaled) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[33];
  const int n = blockIdx.x;
  const char* row = reinterpret_cast<const char*>(W) + static_cast<size_t>(n) * ldw * (kF32 ? 4 : 2);
  const int nvec = K >> 3;
  // pass 1: absmax of W' = W / s (reads only)
  float amax = 0.0f;
  for (int idx = threadIdx.x; idx < nvec; idx += blockDim.x) {
    float w[8];
    load_w8<kF32>(row, idx, w);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(__fdiv_rn(w[e], s)));
  }
  amax = block_reduce<true>(amax, red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sw[n] = en.scale;
  // pass 2: codes; W' is written here, after the row has been read (each
  // thread rewrites only the vectors it has just read, so W_scaled may alias W)
  uint2* out = reinterpret_cast<uint2*>(Wq + static_cast<size_t>(n) * K);
  for (int idx = threadIdx.x; idx < nvec; idx += blockDim.x) {
    float w[8];
    load_w8<kF32>(row, idx, w);
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = __fdiv_rn(w[e], s);
    if (W_scaled) {
      float4* o = reinterpret_cast<float4*>(W_scaled + static_cast<size_t>(n) * K) + 2 * idx;
      o[0] = make_float4(w[0], w[1], w[2], w[3]);
      o[1] = make_float4(w[4], w[5], w[6], w[7]);
    }
    out[idx] = encode8(w, en);
  }
}

__global__ void fold_gamma_kernel(const float* __restrict__ gamma, int K, float s, float* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k < K) out[k] = __fmul_rn(gamma[k], s);
}

// ------------------------------------------------------------------ code-flip count

__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t x) {
  x |= x >> 4;
  x |= x >> 2;
  x |= x >> 1;
  return __popc(x & 0x01010101u);
}

__global__ void count_diff_kernel(const uint8_t* __restrict__ a, const uint8_t* __restrict__ b, size_t n,
                                  unsigned long long* __restrict__ count) {
  griddep_wait();
  griddep_launch_dependents();
  const size_t nv = n >> 4;
  const uint4* a4 = reinterpret_cast<const uint4*>(a);
  const uint4* b4 = reinterpret_cast<const uint4*>(b);
  unsigned long long c = 0;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nv;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 x = __ldg(a4 + i), y = __ldg(b4 + i);
    c += nonzero_bytes(x.x ^ y.x) + nonzero_bytes(x.y ^ y.y) + nonzero_bytes(x.z ^ y.z) +
         nonzero_bytes(x.w ^ y.w);
  }
  if (blockIdx.x == 0 && threadIdx.x < (n & 15)) {
    const size_t i = (nv << 4) + threadIdx.x;
    c += (a[i] != b[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(count, c);
}

// ------------------------------------------------------------------ FP8 key/value cache

// One warp per (token, KV head, key or value): the head's head_dim values
// (16-byte vectors of 8 bf16, one per lane; head_dim <= 256) are quantized as
// one row with the FP8 rule -- the per-token rule applied to each attention
// head -- and the codes and the scale are written to the token's cache slot.
// A negative slot (padding) writes nothing; a slot >= num_slots writes
// nothing and latches kDevBadIndex.
__global__ void __launch_bounds__(256) kv_cache_quant_kernel(const __nv_bfloat16* __restrict__ QKV, int M,
                                                             long long ldq, int q_dim, int kv_heads, int head_dim,
                                                             const long long* __restrict__ slots,
                                                             long long num_slots, uint8_t* __restrict__ kc,
                                                             float* __restrict__ ks, uint8_t* __restrict__ vc,
                                                             float* __restrict__ vs, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const long long item = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= static_cast<long long>(M) * kv_heads * 2) return;
  const int part = static_cast<int>(item & 1);  // 0: key, 1: value
  const long long th = item >> 1;
  const int h = static_cast<int>(th % kv_heads);
  const long long m = th / kv_heads;
  const long long slot = __ldg(slots + m);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) atomicCAS(status, kDevOk, kDevBadIndex);
    return;
  }
  const int nvec = head_dim >> 3;
  const uint4* src = reinterpret_cast<const uint4*>(QKV + m * ldq + q_dim + static_cast<long long>(part) * kv_heads * head_dim +
                                                    static_cast<long long>(h) * head_dim);
  float x[8] = {};
  if (lane < nvec) bf16x8_to_f32(__ldg(src + lane), x);
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
  amax = warp_max(amax);
  const Enc en = make_enc(amax, kQFp8);
  const long long at = slot * kv_heads + h;
  uint8_t* dst = (part ? vc : kc) + at * head_dim;
  if (lane < nvec) reinterpret_cast<uint2*>(dst)[lane] = encode8(x, en);
  if (lane == 0) (part ? vs : ks)[at] = en.scale;
}

// The values a cache holds for the slots a reader gathers: out[n][h hd + d] =
// bf16_RNE(fp32(e4m3 value) * scale); one thread per 8 values.
__global__ void __launch_bounds__(256) kv_cache_dequant_kernel(const uint8_t* __restrict__ cache,
                                                               const float* __restrict__ scale,
                                                               const long long* __restrict__ slots, int n,
                                                               int kv_heads, int head_dim, long long num_slots,
                                                               __nv_bfloat16* __restrict__ out, int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int per_row = kv_heads * head_dim / 8;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n) * per_row) return;
  const long long i = idx / per_row;
  const int j = static_cast<int>(idx - i * per_row);
  const long long slot = __ldg(slots + i);
  if (slot < 0 || slot >= num_slots) {
    atomicCAS(status, kDevOk, kDevBadIndex);
    return;
  }
  const int h = (j * 8) / head_dim;
  const float sc = __ldg(scale + slot * kv_heads + h);
  const uint2 c = __ldg(reinterpret_cast<const uint2*>(cache + slot * kv_heads * head_dim) + j);
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t w = e < 2 ? c.x : c.y;
    const int sh = 16 * (e & 1);
    const __nv_fp8_e4m3 a = *reinterpret_cast<const __nv_fp8_e4m3*>(reinterpret_cast<const uint8_t*>(&w) + sh / 8);
    const __nv_fp8_e4m3 b = *reinterpret_cast<const __nv_fp8_e4m3*>(reinterpret_cast<const uint8_t*>(&w) + sh / 8 + 1);
    const __nv_bfloat162 p = __floats2bfloat162_rn(__fmul_rn(static_cast<float>(a), sc), __fmul_rn(static_cast<float>(b), sc));
    o[e] = *reinterpret_cast<const uint32_t*>(&p);
  }
  reinterpret_cast<uint4*>(out + i * kv_heads * head_dim)[j] = make_uint4(o[0], o[1], o[2], o[3]);
}

// Threads per row-CTA: enough that `per` vectors per thread cover the row, at
// most kRowThreads (longer rows stream their tail from L1/L2 in the code pass).
// With few rows (decode batches: fewer rows than ~2 per SM) a row gets about 2
// vectors per thread instead of kVPT, so each thread's serial chain (loads,
// divisions, block reductions) is short: such kernels are latency-bound.
int row_threads(int nvec, int rows, int per = kVPT) {
  const int want = rows < 304 ? 2 : per;
  int t = 32;
  while (t < kRowThreads && t * want < nvec) t *= 2;
  return t;
}

}  // namespace

cudaError_t launch_quant_act(const void* X, int M, int K, long long ldx, float pre, int qt, void* Xq, float* sx,
                             void* x16, CodeSums sums, cudaStream_t st) {
  if (x16 == nullptr) sums.asum = nullptr;
  return launch_pdl(quant_act_kernel, dim3(M), dim3(row_threads(K / 8, M)), 0, st,
                    reinterpret_cast<const __nv_bfloat16*>(X), K, ldx, pre, qt, reinterpret_cast<uint8_t*>(Xq), sx,
                    reinterpret_cast<uint8_t*>(x16), sums);
}

cudaError_t launch_rmsnorm_quant(const void* X, int M, int K, long long ldx, const float* gamma, float eps,
                                 int qt, void* Xq, float* sx, float* ms_out, void* x16, CodeSums sums,
                                 cudaStream_t st) {
  if (x16 == nullptr) sums.asum = nullptr;
  return launch_pdl(rmsnorm_quant_kernel, dim3(M), dim3(row_threads(K / 8, M)), 0, st,
                    reinterpret_cast<const __nv_bfloat16*>(X), K, ldx, gamma, eps, qt, reinterpret_cast<uint8_t*>(Xq),
                    sx, ms_out, reinterpret_cast<uint8_t*>(x16), sums);
}

cudaError_t launch_silu_mul_quant(const void* GU, int M, int I, long long ldgu, float pre, int qt, void* Xq,
                                  float* sx, float* h_out, void* x16, CodeSums sums, cudaStream_t st) {
  if (x16 == nullptr) sums.asum = nullptr;
  // two vectors (gate, up) are cached per position: half as many per thread
  const int t = row_threads(I / 8, M, kVPT / 2);
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  auto* kern = (sms > 0 && M > sms) ? silu_mul_quant_kernel<2> : silu_mul_quant_kernel<1>;
  return launch_pdl(kern, dim3(M), dim3(t), 0, st, reinterpret_cast<const __nv_bfloat16*>(GU), I, ldgu, pre, qt,
                    reinterpret_cast<uint8_t*>(Xq), sx, h_out, reinterpret_cast<uint8_t*>(x16), sums);
}

cudaError_t launch_prepare_weights(const void* W, bool w_f32, int N, int K, long long ldw, const float* gamma,
                                   float s, int qt, void* Wq, float* sw, float* gamma_folded, float* W_scaled,
                                   cudaStream_t st) {
  const int t = row_threads(K / 8, N);
  cudaError_t e = w_f32 ? launch_pdl(prepare_weights_kernel<true>, dim3(N), dim3(t), 0, st, W, K, ldw, s, qt,
                                     reinterpret_cast<uint8_t*>(Wq), sw, W_scaled)
                        : launch_pdl(prepare_weights_kernel<false>, dim3(N), dim3(t), 0, st, W, K, ldw, s, qt,
                                     reinterpret_cast<uint8_t*>(Wq), sw, W_scaled);
  if (e != cudaSuccess) return e;
  if (gamma) e = launch_pdl(fold_gamma_kernel, dim3((K + 255) / 256), dim3(256), 0, st, gamma, K, s, gamma_folded);
  return e;
}

cudaError_t launch_count_diff(const void* a, const void* b, size_t n, unsigned long long* count, int num_sms,
                              cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(unsigned long long), st);
  if (e != cudaSuccess) return e;
  const size_t nv = n >> 4;
  size_t blocks = (nv + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms > 0 ? num_sms : 152) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(count_diff_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                    reinterpret_cast<const uint8_t*>(a), reinterpret_cast<const uint8_t*>(b), n, count);
}

cudaError_t launch_kv_cache_quant(const void* QKV, int M, long long ldq, int q_dim, int kv_heads, int head_dim,
                                  const long long* slots, long long num_slots, void* kc, float* ks, void* vc,
                                  float* vs, int* status, cudaStream_t st) {
  const long long items = static_cast<long long>(M) * kv_heads * 2;
  const unsigned blocks = static_cast<unsigned>((items + 7) / 8);
  return launch_pdl(kv_cache_quant_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const __nv_bfloat16*>(QKV),
                    M, ldq, q_dim, kv_heads, head_dim, slots, num_slots, reinterpret_cast<uint8_t*>(kc), ks,
                    reinterpret_cast<uint8_t*>(vc), vs, status);
}

cudaError_t launch_kv_cache_dequant(const void* cache, const float* scale, const long long* slots, int n,
                                    int kv_heads, int head_dim, long long num_slots, void* out, int* status,
                                    cudaStream_t st) {
  const long long items = static_cast<long long>(n) * kv_heads * head_dim / 8;
  const unsigned blocks = static_cast<unsigned>((items + 255) / 256);
  return launch_pdl(kv_cache_dequant_kernel, dim3(blocks), dim3(256), 0, st, reinterpret_cast<const uint8_t*>(cache),
                    scale, slots, n, kv_heads, head_dim, num_slots, reinterpret_cast<__nv_bfloat16*>(out), status);
}

}  // namespace qurl
