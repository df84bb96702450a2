// rowquant.cuh -- per-row quantization of activations, shared by the
// quantizer kernels (one row per CTA) and the decode GEMMs that quantize their
// own input rows (fused entry points):
//   * per-token activation quantization (optionally with a UAQ pre-scale),
//   * RMSNorm with the UAQ-folded gain -> per-token quantization,
//   * SiLU(gate) * up -> per-token quantization.
//
// Method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
// Quantized Rollout", sections "更新感知量化 (UAQ)" (W X = (W/s)(sX), s folded
// into the norm gain) and "损失函数 / 训练策略" (per-token activation INT8/FP8
// quantization, s = 1.5).
//
// A row is processed by every thread of the calling block: 16-byte vector
// loads, up to NC vectors per thread cached in registers between the absmax
// pass and the code pass, warp-shuffle + shared-memory block reductions.
// Arithmetic that decides a code is IEEE fp32 with explicit rounding
// intrinsics (no contraction):
//   scale = absmax / qmax (absmax == 0 -> 1);  code = RNE(v / scale)
//   clamped to +-127 (INT8), or e4m3 RNE with saturation (FP8).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "internal.h"

namespace qurl {
namespace rq {

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

// The same for two independent accumulator pairs at once (lanes x and y).
__device__ __forceinline__ void two_sum_acc2(float2& s, float2& c, float2 y) {
  const float2 t = __fadd2_rn(s, y);
  const float2 bp = __fadd2_rn(t, make_float2(-s.x, -s.y));
  const float2 tb = __fadd2_rn(t, make_float2(-bp.x, -bp.y));
  const float2 err = __fadd2_rn(__fadd2_rn(s, make_float2(-tb.x, -tb.y)), __fadd2_rn(y, make_float2(-bp.x, -bp.y)));
  s = t;
  c = __fadd2_rn(c, err);
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
  bool fma_quotient;  // FP8: the scale admits the FMA-corrected quotient (below)
};

__device__ __forceinline__ Enc make_enc(float amax, int qt) {
  const float scale = row_scale(amax, qt);
  return {scale, __frcp_rn(scale), qt, scale >= 0x1p-80f && scale <= 0x1p100f};
}

// ---- paired fp32 arithmetic: sm_100's two-lane fp32 instructions, each lane
// rounded exactly like its scalar counterpart (no contraction).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

// Codes of v / scale.  Both types are decided on the IEEE quotient fl(v /
// scale), but most codes come from the product r = v * fl(1 / scale) instead:
// r carries two roundings of relative size 2^-24 on top of the exact quotient,
// so it lies within 2.5 units in the last place of fl(v / scale).
//  * INT8: fl(v / scale) rounded to the nearest integer, ties to even, clamped
//    to +-127.  |v| <= absmax makes |r| <= 127 (1 + 2^-22), so r is within
//    5e-5 of the quotient: wherever r is more than 1e-4 away from a
//    half-integer both round to the same integer, which r + 1.5 * 2^23 gives
//    (the sum's unit in the last place is 1, so the addition itself rounds r
//    to an integer, ties to even; its low byte is the two's-complement code)
//    and which needs no clamp.  Otherwise (one code in ~5000, and NaN inputs,
//    whose distance to the integer is NaN) the quotient itself is computed.
//  * FP8-E4M3: round to nearest even with saturation to +-448, applied to
//    fl(v / scale) itself, which one correction step gives without a
//    division: with inv = fl(1 / scale) (correctly rounded) and r = fl(v *
//    inv) within an ulp of the quotient, the residual v - r * scale is exact
//    in one FMA and fl(r + residual * inv) is the correctly rounded quotient
//    (Markstein's theorem for FMA division, valid while the residual does not
//    underflow, i.e. for |v| >= 2^-102: with the scale in [2^-80, 2^100] and
//    |quotient| <= 448 every quotient of 2^-11 or more -- all that can give a
//    nonzero code -- qualifies, and smaller ones, exact or not, encode to a
//    signed zero).  The sign is copied from v, so that -0 keeps its sign.
//    Rows with a scale outside that range divide.  Two codes per conversion.
// The codes are therefore those of the plain division.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ int i8_quotient_code(float v, const Enc& e) {
  const int q = __float2int_rn(__fdiv_rn(v, e.scale));
  return max(-127, min(127, q));
}

// Low bytes of four words -> one word (byte i from word i).
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// 8 INT8 codes of v (pairs in k order) packed in k order; q receives the
// same codes as floats.
__device__ __forceinline__ uint2 encode8_i8(const float2 (&v)[4], const Enc& e, float2 (&q)[4]) {
  const float2 inv = splat2(e.inv), mg = splat2(kRoundMagic);
  uint32_t b[8];
  bool fast = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 r = mul2(v[i], inv);
    const float2 t = add2(r, mg);
    q[i] = sub2(t, mg);
    const float2 d = sub2(r, q[i]);
    fast = fast & (fabsf(d.x) < 0.4999f) & (fabsf(d.y) < 0.4999f);
    b[2 * i] = __float_as_uint(t.x);
    b[2 * i + 1] = __float_as_uint(t.y);
  }
  if (!fast) {
    float qs[8], vs[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qs[2 * i] = q[i].x;
      qs[2 * i + 1] = q[i].y;
      vs[2 * i] = v[i].x;
      vs[2 * i + 1] = v[i].y;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!(fabsf(__fsub_rn(__fmul_rn(vs[j], e.inv), qs[j])) < 0.4999f)) {
        const int c = i8_quotient_code(vs[j], e);
        b[j] = static_cast<uint32_t>(c);
        qs[j] = static_cast<float>(c);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = make_float2(qs[2 * i], qs[2 * i + 1]);
  }
  return make_uint2(pack_low_bytes(b[0], b[1], b[2], b[3]), pack_low_bytes(b[4], b[5], b[6], b[7]));
}

// 8 FP8-E4M3 codes of v (pairs in k order) packed in k order.
__device__ __forceinline__ uint2 encode8_f8(const float2 (&v)[4], const Enc& e) {
  uint32_t h[4];
  if (e.fma_quotient) {
    const float2 inv = splat2(e.inv), nscale = splat2(-e.scale);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 r = mul2(v[i], inv);
      const float2 res = __ffma2_rn(r, nscale, v[i]);  // v - r * scale, exact
      float2 q = __ffma2_rn(res, inv, r);
      q.x = copysignf(q.x, v[i].x);
      q.y = copysignf(q.y, v[i].y);
      h[i] = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);  // .x in the low byte
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      h[i] = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(v[i].x, e.scale), __fdiv_rn(v[i].y, e.scale)),
                                      __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

__device__ __forceinline__ uint2 encode8(const float2 (&v)[4], const Enc& en) {
  if (en.qt == kQInt8) {
    float2 q[4];
    return encode8_i8(v, en, q);
  }
  return encode8_f8(v, en);
}

// 8 values -> 8 code bytes packed in a uint2 (little-endian byte order = k order).
__device__ __forceinline__ uint2 encode8(const float (&v)[8], const Enc& en) {
  const float2 p[4] = {make_float2(v[0], v[1]), make_float2(v[2], v[3]), make_float2(v[4], v[5]),
                       make_float2(v[6], v[7])};
  return encode8(p, en);
}

// Saturation of the sums of |code| (any value above 2^24 / 128 means
// "accumulate in chunks" to the GEMM that reads them).
constexpr int kAbsSumCap = 1 << 24;

// Sum of |code| and of code^2 of 8 INT8 codes: |c| = c * (+1 or -1), the
// second factor's bytes 0x01 | the code's sign replicated (byte_perm selector
// nibbles with bit 3 set copy the selected byte's sign bit).
__device__ __forceinline__ int2 code_sums8(uint2 c) {
  const int sx = static_cast<int>(__byte_perm(c.x, 0u, 0xBA98) | 0x01010101u);
  const int sy = static_cast<int>(__byte_perm(c.y, 0u, 0xBA98) | 0x01010101u);
  const int cx = static_cast<int>(c.x), cy = static_cast<int>(c.y);
  return make_int2(__dp4a(cy, sy, __dp4a(cx, sx, 0)), __dp4a(cy, cy, __dp4a(cx, cx, 0)));
}

// Store the 8 codes of v (and, for INT8 when x16 is given, the same 8 codes
// as fp16 -- exact, integers of magnitude <= 127 -- for the tensor-core GEMM
// to read).  Returns the sum of |code| and the sum of code^2 of the 8 INT8
// codes when x16 is given, else zeros.
__device__ __forceinline__ int2 store8(uint8_t* __restrict__ q, uint8_t* __restrict__ x16, size_t idx,
                                       const float2 (&v)[4], const Enc& en) {
  if (en.qt != kQInt8) {
    reinterpret_cast<uint2*>(q)[idx] = encode8_f8(v, en);
    return make_int2(0, 0);
  }
  float2 qf[4];
  const uint2 c = encode8_i8(v, en, qf);
  reinterpret_cast<uint2*>(q)[idx] = c;
  if (x16 == nullptr) return make_int2(0, 0);
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 p = __float22half2_rn(qf[i]);  // .x in the low half
    h[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
  reinterpret_cast<uint4*>(x16)[idx] = make_uint4(h[0], h[1], h[2], h[3]);
  return code_sums8(c);
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

__device__ __forceinline__ void bf16x8_to_f2(const uint4 u, float2 (&x)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
}

// Largest |x| of 8 bf16 values folded into m (two lanes; NaN never wins, as in fmaxf).
__device__ __forceinline__ __nv_bfloat162 absmax_bf16x8(const uint4 u, __nv_bfloat162 m) {
  const uint32_t w[4] = {u.x & 0x7FFF7FFFu, u.y & 0x7FFF7FFFu, u.z & 0x7FFF7FFFu, u.w & 0x7FFF7FFFu};
#pragma unroll
  for (int e = 0; e < 4; ++e) m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162*>(&w[e]));
  return m;
}

// max |fl(a * pre)| over the values a whose largest magnitude is amax: rounding
// is monotone, so it is fl(amax * |pre|) (and 0 for pre = 0, where non-finite
// a would give NaN products, which a max ignores).
__device__ __forceinline__ float scaled_absmax(float amax, float pre) {
  return pre == 0.0f ? 0.0f : __fmul_rn(amax, fabsf(pre));
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

// Shared-memory scratch of a row: the block reductions' partials and the
// per-range code-sum counters.
struct RowScratch {
  float red[66];
  unsigned long long cnt[2 * kMaxSums];
};

// Per-token quantization of row m of X (bf16, row stride ldx): v = x * pre,
// codes to Xq (stride K), scale to sx[m]; for INT8 with x16, also the fp16
// copy of the codes and their sums.  Every thread of the block calls it.
template <int NC>
__device__ __forceinline__ void quant_act_row(int m, const __nv_bfloat16* __restrict__ X, int K, long long ldx,
                                              float pre, int qt, uint8_t* __restrict__ Xq, float* __restrict__ sx,
                                              uint8_t* __restrict__ x16, const CodeSums& sums, RowScratch& sh) {

  __syncthreads();  // the previous row's reductions and sums are done with the scratch
  sums_begin(sh.cnt, sums);
  const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * ldx);
  const int nvec = K >> 3;
  uint4 cache[NC];
  fill_cache(row, nvec, cache);
  // the largest |x| on the bf16 values themselves; the pre-scale is applied once
  __nv_bfloat162 m2 = __floats2bfloat162_rn(0.0f, 0.0f);
  for_vectors(row, nvec, cache, [&](const uint4 u, int) { m2 = absmax_bf16x8(u, m2); });
  float amax = scaled_absmax(fmaxf(__bfloat162float(m2.x), __bfloat162float(m2.y)), pre);
  amax = block_reduce<true>(amax, sh.red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sx[m] = en.scale;
  uint8_t* out = Xq + static_cast<size_t>(m) * K;
  uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * K * 2 : nullptr;
  const float2 pre2 = splat2(pre);
  for_vectors_warp(row, nvec, cache, [&](const uint4 u, int idx, bool valid) {
    int2 v = make_int2(0, 0);
    if (valid) {
      float2 x[4];
      bf16x8_to_f2(u, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = mul2(x[e], pre2);
      v = store8(out, out16, idx, x, en);
    }
    sums_add_warp(sh.cnt, sums, idx, v);
  });
  sums_end(sh.cnt, sums, m);
}

// RMSNorm of row m with the folded gain gamma', then per-token quantization
// (ms_out[m], when given, receives the row's mean of squares).
template <int NC>
__device__ __forceinline__ void rmsnorm_quant_row(int m, const __nv_bfloat16* __restrict__ X, int K, long long ldx,
                                                  const float* __restrict__ gamma, float eps, int qt,
                                                  uint8_t* __restrict__ Xq, float* __restrict__ sx,
                                                  float* __restrict__ ms_out, uint8_t* __restrict__ x16,
                                                  const CodeSums& sums, RowScratch& sh) {

  __syncthreads();  // the previous row's reductions and sums are done with the scratch
  sums_begin(sh.cnt, sums);
  const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<size_t>(m) * ldx);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  const int nvec = K >> 3;
  uint4 cache[NC];
  fill_cache(row, nvec, cache);
  // mean of squares.  Each x^2 is exact in fp32 (a bf16 has an 8-bit
  // significand); the sum is carried as an unevaluated pair s + c (error-free
  // two-sum per term, Knuth) and divided by K in fp64, so ms is the fp32
  // rounding of the mean to within ~2^-44 relative -- the same fp32 value a
  // plain fp64 sum gives, except when the mean lies that close to a rounding
  // midpoint.
  float2 ss2 = make_float2(0.0f, 0.0f), sc2 = make_float2(0.0f, 0.0f);  // even / odd k
  for_vectors(row, nvec, cache, [&](const uint4 u, int) {
    float2 x[4];
    bf16x8_to_f2(u, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) two_sum_acc2(ss2, sc2, mul2(x[e], x[e]));
  });
  float ss = ss2.x, sc = sc2.x;
  two_sum_acc(ss, sc, ss2.y);
  sc = __fadd_rn(sc, sc2.y);
  // the gain of the vectors this thread normalises is read while the sums are reduced
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    if (idx < nvec) asm volatile("prefetch.global.L1 [%0];" ::"l"(g4 + 2 * idx));
  }
  float ms, r;
  block_mean_sq(ss, sc, sh.red, K, eps, ms, r);
  if (threadIdx.x == 0 && ms_out) ms_out[m] = ms;
  // v = (x * r) * gamma'
  const float2 r2 = splat2(r);
  auto normed = [&](const uint4 u, int idx, float2 (&x)[4]) {
    bf16x8_to_f2(u, x);
    const float4 ga = __ldg(g4 + 2 * idx), gb = __ldg(g4 + 2 * idx + 1);
    const float2 g[4] = {make_float2(ga.x, ga.y), make_float2(ga.z, ga.w), make_float2(gb.x, gb.y),
                         make_float2(gb.z, gb.w)};
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = mul2(mul2(x[e], r2), g[e]);
  };
  float amax = 0.0f;
  for_vectors(row, nvec, cache, [&](const uint4 u, int idx) {
    float2 x[4];
    normed(u, idx, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fmaxf(fabsf(x[e].x), fabsf(x[e].y)));
  });
  amax = block_reduce<true>(amax, sh.red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sx[m] = en.scale;
  uint8_t* out = Xq + static_cast<size_t>(m) * K;
  uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * K * 2 : nullptr;
  for_vectors_warp(row, nvec, cache, [&](const uint4 u, int idx, bool valid) {
    int2 v = make_int2(0, 0);
    if (valid) {
      float2 x[4];
      normed(u, idx, x);
      v = store8(out, out16, idx, x, en);
    }
    sums_add_warp(sh.cnt, sums, idx, v);
  });
  sums_end(sh.cnt, sums, m);
}

__device__ __forceinline__ float silu_ratio(float g, float den) {
  return den < 0x1p126f ? __fdividef(g, den) : 0.0f;
}

__device__ __forceinline__ void silu_mul8(const uint4 gu, const uint4 uu, float2 (&h)[4]) {
  float2 g[4], u[4];
  bf16x8_to_f2(gu, g);
  bf16x8_to_f2(uu, u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    // g / (1 + exp(-g)) to within ~2 units in the last place (h is held to a
    // relative 2e-6 of the exact value; the codes are decided on this h).  A
    // denominator beyond 2^126 (g < -87.3) makes |h| < 2e-36: 0.
    const float2 den = add2(splat2(1.0f), make_float2(expf(-g[e].x), expf(-g[e].y)));
    h[e] = mul2(make_float2(silu_ratio(g[e].x, den.x), silu_ratio(g[e].y, den.y)), u[e]);
  }
}

// SiLU(gate) * up of row m of GU ([M, 2I], gate | up, row stride ldgu), then
// per-token quantization with the pre-scale (h_out, when given, receives h).
template <int NC>
__device__ __forceinline__ void silu_mul_quant_row(int m, const __nv_bfloat16* __restrict__ GU, int I, long long ldgu,
                                                   float pre, int qt, uint8_t* __restrict__ Xq,
                                                   float* __restrict__ sx, float* __restrict__ h_out,
                                                   uint8_t* __restrict__ x16, const CodeSums& sums, RowScratch& sh) {

  __syncthreads();  // the previous row's reductions and sums are done with the scratch
  sums_begin(sh.cnt, sums);
  const uint4* grow = reinterpret_cast<const uint4*>(GU + static_cast<size_t>(m) * ldgu);
  const uint4* urow = reinterpret_cast<const uint4*>(GU + static_cast<size_t>(m) * ldgu + I);
  const int nvec = I >> 3;
  uint4 cg[NC], cu[NC];
  fill_cache(grow, nvec, cg);
  fill_cache(urow, nvec, cu);
  // pass 1: h = silu(g) * u, kept in registers for the cached positions; the
  // largest |h| (the pre-scale is applied to it once)
  float2 hc[NC][4];
  float amax = 0.0f;
  auto take = [&](const float2 (&h)[4], int idx) {
    if (h_out) {
      float4* ho = reinterpret_cast<float4*>(h_out + static_cast<size_t>(m) * I) + 2 * idx;
      ho[0] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
      ho[1] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fmaxf(fabsf(h[e].x), fabsf(h[e].y)));
  };
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    if (idx < nvec) {
      silu_mul8(cg[c], cu[c], hc[c]);
      take(hc[c], idx);
    }
  }
  for (int idx = threadIdx.x + NC * blockDim.x; idx < nvec; idx += blockDim.x) {
    float2 h[4];
    silu_mul8(__ldg(grow + idx), __ldg(urow + idx), h);
    take(h, idx);
  }
  amax = block_reduce<true>(scaled_absmax(amax, pre), sh.red);
  const Enc en = make_enc(amax, qt);
  if (threadIdx.x == 0) sx[m] = en.scale;
  uint8_t* out = Xq + static_cast<size_t>(m) * I;
  uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * I * 2 : nullptr;
  const float2 pre2 = splat2(pre);
  // pass 2: codes (warp-uniform steps, see for_vectors_warp)
  auto put = [&](float2 (&h)[4], int idx, bool valid) {
    int2 v = make_int2(0, 0);
    if (valid) {
#pragma unroll
      for (int e = 0; e < 4; ++e) h[e] = mul2(h[e], pre2);
      v = store8(out, out16, idx, h, en);
    }
    sums_add_warp(sh.cnt, sums, idx, v);
  };
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int idx = threadIdx.x + c * blockDim.x;
    put(hc[c], idx, idx < nvec);
  }
  for (int i0 = NC * blockDim.x + (threadIdx.x & ~31); i0 < nvec; i0 += blockDim.x) {
    const int idx = i0 + (threadIdx.x & 31);
    float2 h[4] = {};
    if (idx < nvec) silu_mul8(__ldg(grow + idx), __ldg(urow + idx), h);
    put(h, idx, idx < nvec);
  }
  sums_end(sh.cnt, sums, m);
}

}  // namespace rq
}  // namespace qurl
