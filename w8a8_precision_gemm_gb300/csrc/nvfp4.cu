// nvfp4.cu -- the 4-bit (W4A4) variant of the quantized linear layer: NVFP4
// rows and their exact widening to fp16 for the tensor-core GEMM.
//
// Method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
// Quantized Rollout", section "局限与展望" (4-bit quantization named as the
// next, larger speedup, not explored there) and the QeRL entry of the
// related-papers list on the fugumt page of the same paper (NVFP4 in RL
// rollout).  The pages do not define the format; the reading taken is
// NVIDIA's published NVFP4 layout with the pages' per-channel / per-token
// second-level scale:
//   * E2M1 element codes (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; sign bit 3),
//     two per byte, value 2j in the low nibble of byte j;
//   * one E4M3 scale per 16 consecutive values of a row (a block);
//   * one fp32 scale g per row: g = max|v| / 2688 (6 * 448), 1 for a zero row.
// Block b: s_b = e4m3_RNE_satfinite(max|v_b| / fl(6 g)); step e_b =
// fl(dec(s_b) * g); code = e2m1_RNE_satfinite(fl(v / e_b)), 0 where e_b = 0.
//
// The GEMM multiplies dec(code) * dec(s_b) -- at most 6 significant bits, in
// [2^-10, 2688] -- which fp16 holds exactly, on the fp16 tensor path (the CTA
// pair kernel of the INT8 prefill, accumulating in fp32); g_x and g_w enter
// its dequantizing epilogue as the token and channel scales.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "rowquant.cuh"

namespace qurl {
namespace {

constexpr int kNvThreads = 256;

// fl(v / d) for a step d in [2^-80, 2^100] by one FMA correction of the
// reciprocal product (correctly rounded by Markstein's theorem wherever the
// residual does not underflow, |v| >= 2^-102: so for every quotient of 2^-3 or
// more, all that can round to a nonzero E2M1 code), sign of v kept.
__device__ __forceinline__ float2 quotient2(float2 v, float d, float inv) {
  const float2 r = __fmul2_rn(v, make_float2(inv, inv));
  const float2 res = __ffma2_rn(r, make_float2(-d, -d), v);
  float2 q = __ffma2_rn(res, make_float2(inv, inv), r);
  q.x = copysignf(q.x, v.x);
  q.y = copysignf(q.y, v.y);
  return q;
}

// 16 values of one block -> 8 code bytes (value 2j in the low nibble of byte j).
__device__ __forceinline__ uint2 e2m1_codes16(const float (&v)[16], float e) {
  uint32_t w[2] = {0u, 0u};
  if (e == 0.0f) return make_uint2(0u, 0u);
  const bool fma_ok = e >= 0x1p-80f && e <= 0x1p100f;
  const float inv = __frcp_rn(e);
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const float2 x = make_float2(v[2 * p], v[2 * p + 1]);
    const float2 q = fma_ok ? quotient2(x, e, inv) : make_float2(__fdiv_rn(x.x, e), __fdiv_rn(x.y, e));
    const uint32_t b = __nv_cvt_float2_to_fp4x2(q, __NV_E2M1, cudaRoundNearest) & 0xFFu;  // .x low nibble
    w[p >> 2] |= b << (8 * (p & 3));
  }
  return make_uint2(w[0], w[1]);
}

// One row per CTA: pass 1 the row's largest |v|, pass 2 one block of 16
// values per thread step.  Rows of bf16 activations (v = x * pre) or fp32
// weights (v = w).
template <bool kF32>
__global__ void __launch_bounds__(kNvThreads) nvfp4_quant_kernel(const void* __restrict__ X, int K, long long ldx,
                                                                 float pre, uint8_t* __restrict__ q4,
                                                                 uint8_t* __restrict__ sblk, float* __restrict__ g) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[66];
  const int m = blockIdx.x;
  const char* row = reinterpret_cast<const char*>(X) + static_cast<size_t>(m) * ldx * (kF32 ? 4 : 2);
  const int nblk = K >> 4;
  auto load16 = [&](int b, float (&v)[16]) {
    if (kF32) {
      const float4* p = reinterpret_cast<const float4*>(row) + 4 * b;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 t = __ldg(p + i);
        v[4 * i] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
      }
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(row) + 2 * b;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float2 x[4];
        rq::bf16x8_to_f2(__ldg(p + i), x);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 y = __fmul2_rn(x[e], make_float2(pre, pre));
          v[8 * i + 2 * e] = y.x;
          v[8 * i + 2 * e + 1] = y.y;
        }
      }
    }
  };
  float amax = 0.0f;
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
    float v[16];
    load16(b, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = rq::block_reduce<true>(amax, red);
  const float gs = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  const float d6 = __fmul_rn(6.0f, gs);
  if (threadIdx.x == 0) g[m] = gs;
  uint2* out = reinterpret_cast<uint2*>(q4 + static_cast<size_t>(m) * (K >> 1));
  uint8_t* sb = sblk + static_cast<size_t>(m) * nblk;
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
    float v[16];
    load16(b, v);
    float ab = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
    const uint8_t s = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(ab, d6), __NV_SATFINITE, __NV_E4M3));
    const float ds = __half2float(__half(__nv_cvt_fp8_to_halfraw(s, __NV_E4M3)));
    sb[b] = s;
    out[b] = e2m1_codes16(v, __fmul_rn(ds, gs));
  }
}

// One thread per block of 16: codes and block scale -> 16 fp16 values
// dec(code) * dec(scale), exact (at most 6 significant bits, in [2^-10, 2688]).
__global__ void __launch_bounds__(256) nvfp4_widen_kernel(const uint8_t* __restrict__ q4,
                                                          const uint8_t* __restrict__ sblk, long long nblk,
                                                          uint8_t* __restrict__ out16) {
  griddep_wait();
  griddep_launch_dependents();
  for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nblk;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(q4) + b);
    const __half s = __half(__nv_cvt_fp8_to_halfraw(__ldg(sblk + b), __NV_E4M3));
    const __half2 s2 = __halves2half2(s, s);
    uint32_t h[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const uint32_t byte = ((p < 4 ? c.x : c.y) >> (8 * (p & 3))) & 0xFFu;
      const __half2 v = __half2(__nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte), __NV_E2M1));
      const __half2 r = __hmul2(v, s2);
      h[p] = *reinterpret_cast<const uint32_t*>(&r);
    }
    uint4* d = reinterpret_cast<uint4*>(out16) + 2 * b;
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace

cudaError_t launch_nvfp4_quant(const void* X, bool x_f32, int R, int K, long long ldx, float pre, void* q4,
                               void* sblk, float* g, cudaStream_t st) {
  int t = 32;
  while (t < kNvThreads && t < (K >> 4)) t *= 2;
  if (x_f32)
    return launch_pdl(nvfp4_quant_kernel<true>, dim3(R), dim3(t), 0, st, X, K, ldx, pre,
                      reinterpret_cast<uint8_t*>(q4), reinterpret_cast<uint8_t*>(sblk), g);
  return launch_pdl(nvfp4_quant_kernel<false>, dim3(R), dim3(t), 0, st, X, K, ldx, pre,
                    reinterpret_cast<uint8_t*>(q4), reinterpret_cast<uint8_t*>(sblk), g);
}

cudaError_t launch_nvfp4_widen(const void* q4, const void* sblk, int R, int K, void* out16, int num_sms,
                               cudaStream_t st) {
  const long long nblk = static_cast<long long>(R) * (K >> 4);
  long long blocks = (nblk + 255) / 256;
  const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(nvfp4_widen_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                    reinterpret_cast<const uint8_t*>(q4), reinterpret_cast<const uint8_t*>(sblk), nblk,
                    reinterpret_cast<uint8_t*>(out16));
}

}  // namespace qurl
