// quant.cu -- the memory-bound kernels of the W8A8 path:
//   * per-token activation quantization (optionally with a UAQ pre-scale),
//   * RMSNorm with the UAQ-folded gain -> per-token quantization,
//   * SiLU(gate) * up -> per-token quantization,
//     (one row per CTA; the row arithmetic is in rowquant.cuh),
//   * UAQ weight fold W' = W/s + per-output-channel weight quantization,
//   * gain fold gamma' = gamma * s,
//   * code-flip count of two code buffers,
//   * FP8 key/value cache quantization and its read-back.
//
// Method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
// Quantized Rollout", sections "更新感知量化 (UAQ)" (W X = (W/s)(sX), s folded
// into the norm gain), "损失函数 / 训练策略" (per-channel weight and per-token
// activation INT8/FP8 quantization, s = 1.5) and "局限与展望" (FP8 KV cache).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "rowquant.cuh"

namespace qurl {
namespace {

constexpr int kVPT = 8;           // 16-byte vectors cached per thread
constexpr int kRowThreads = 512;  // most threads of a row CTA (register budget of the row kernels)
constexpr int kSlimVPT = 5;       // e.g. the 5120-wide rows of the 32B class at 128 threads
// The 5120-wide rows at 128 threads: nine resident CTAs a SM (at most 56
// registers a thread) instead of eight at 64.  Measured at M = 8192 (RMSNorm,
// INT8 / FP8): 50.8 / 47.6 us against 54.5 / 50.5; ten (47 registers) and
// twelve (40) spill and measured slower.
constexpr int kDenseRows = 9;

using rq::Enc;
using rq::block_reduce;
using rq::bf16x8_to_f32;
using rq::encode8;
using rq::make_enc;
using rq::warp_max;

// ------------------------------------------------------------------ activation quant

// NC: 16-byte vectors a thread caches (kVPT, or kSlimVPT for rows that need
// no more: fewer registers, more resident CTAs).
template <int NC, int MAXT = kRowThreads, int MINB = 1>
__global__ void __launch_bounds__(MAXT, MINB) quant_act_kernel(const __nv_bfloat16* __restrict__ X, int K, long long ldx, float pre, int qt,
                                 uint8_t* __restrict__ Xq, float* __restrict__ sx, uint8_t* __restrict__ x16,
                                 const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ rq::RowScratch sh;
  rq::quant_act_row<NC>(blockIdx.x, X, K, ldx, pre, qt, Xq, sx, x16, sums, sh);
}

// ------------------------------------------------------------------ RMSNorm -> quant

template <int NC, int MAXT = kRowThreads, int MINB = 1>
__global__ void __launch_bounds__(MAXT, MINB) rmsnorm_quant_kernel(const __nv_bfloat16* __restrict__ X, int K, long long ldx,
                                     const float* __restrict__ gamma, float eps, int qt, uint8_t* __restrict__ Xq,
                                     float* __restrict__ sx, float* __restrict__ ms_out, uint8_t* __restrict__ x16,
                                     const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ rq::RowScratch sh;
  rq::rmsnorm_quant_row<NC>(blockIdx.x, X, K, ldx, gamma, eps, qt, Xq, sx, ms_out, x16, sums, sh);
}

// ------------------------------------------------------------------ SiLU * up -> quant

// MINB = 2: two blocks per SM (at most 64 registers a thread) when there are
// more rows than SMs, so a batch of up to two rows per SM runs as one wave.
template <int MINB>
__global__ void __launch_bounds__(kRowThreads, MINB) silu_mul_quant_kernel(const __nv_bfloat16* __restrict__ GU, int I, long long ldgu, float pre,
                                      int qt, uint8_t* __restrict__ Xq, float* __restrict__ sx,
                                      float* __restrict__ h_out, uint8_t* __restrict__ x16,
                                      const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ rq::RowScratch sh;
  rq::silu_mul_quant_row<kVPT / 2>(blockIdx.x, GU, I, ldgu, pre, qt, Xq, sx, h_out, x16, sums, sh);
}

// Rows of more than 2048 positions at more rows than SMs: 1024 threads (one
// CTA per SM at 64 registers), so the register cache holds rows of up to 4096
// positions whole and pass 2 recomputes none of them.
__global__ void __launch_bounds__(1024, 1) silu_mul_quant_1k_kernel(const __nv_bfloat16* __restrict__ GU, int I,
                                                                   long long ldgu, float pre, int qt,
                                                                   uint8_t* __restrict__ Xq, float* __restrict__ sx,
                                                                   float* __restrict__ h_out,
                                                                   uint8_t* __restrict__ x16, const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ rq::RowScratch sh;
  rq::silu_mul_quant_row<kVPT / 2>(blockIdx.x, GU, I, ldgu, pre, qt, Xq, sx, h_out, x16, sums, sh);
}

// Rows of 8192 .. kSiluStreamMaxI positions at more rows than SMs: one
// persistent CTA of 1024 threads per SM walks rows blockIdx.x + j gridDim.x.
// Each gate | up row arrives in shared memory by one bulk copy, two rows
// ahead: while a row is computed, reduced and its codes stored, the next one
// is already in flight, so the SM keeps reading HBM through the arithmetic,
// the block reductions and the stores (one resident row kernel per SM leaves
// HBM idle across each of those phases).  Same arithmetic, in the same order,
// as the row kernels above.
constexpr int kSiluStreamNC = 4;  // vectors of h a thread holds: rows of up to 4 x 1024 x 8 positions
constexpr int kSiluStreamMaxI = 27648;  // two gate | up rows of bf16: 8 I bytes of shared memory

__device__ __forceinline__ void drain_bulk(uint64_t* bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, kDevOk, kDevTimeout);
      return;
    }
  }
}

__global__ void __launch_bounds__(1024, 1) silu_mul_quant_stream_kernel(const __nv_bfloat16* __restrict__ GU, int M,
                                                                       int I, long long ldgu, float pre, int qt,
                                                                       uint8_t* __restrict__ Xq, float* __restrict__ sx,
                                                                       float* __restrict__ h_out,
                                                                       uint8_t* __restrict__ x16, const CodeSums sums,
                                                                       int* status) {
  extern __shared__ __align__(16) uint8_t rows_smem[];  // [2][gate I | up I] bf16
  __shared__ rq::RowScratch sh;
  __shared__ uint64_t full[2];
  __shared__ int stop;
  const uint32_t row_bytes = 4u * static_cast<uint32_t>(I);
  const int nvec = I >> 3;
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_barrier_init();
    stop = 0;
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  int issued[2] = {0, 0};  // copies issued per buffer (thread 0)
  auto issue = [&](int j) {
    const int m = blockIdx.x + j * static_cast<int>(gridDim.x);
    if (m >= M) return;
    mbar_arrive_expect_tx(&full[j & 1], row_bytes);
    bulk_load_1d(rows_smem + (j & 1) * row_bytes, GU + static_cast<size_t>(m) * ldgu, row_bytes, &full[j & 1]);
    ++issued[j & 1];
  };
  if (threadIdx.x == 0) {
    issue(0);
    issue(1);
  }
  const float2 pre2 = rq::splat2(pre);
  int j = 0;
  for (;; ++j) {
    const int m = blockIdx.x + j * static_cast<int>(gridDim.x);
    if (m >= M) break;
    if (threadIdx.x == 0 && !mbar_wait(&full[j & 1], (j >> 1) & 1, status)) stop = 1;
    __syncthreads();  // also: the previous row's sums are written before the counters are reset
    if (stop) break;
    rq::sums_begin(sh.cnt, sums);
    const uint4* g = reinterpret_cast<const uint4*>(rows_smem + (j & 1) * row_bytes);
    const uint4* u = g + nvec;
    // pass 1: h = silu(g) * u into registers; the largest |h|
    float2 hc[kSiluStreamNC][4];
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < kSiluStreamNC; ++c) {
      const int idx = threadIdx.x + c * 1024;
      if (idx < nvec) {
        rq::silu_mul8(g[idx], u[idx], hc[c]);
        if (h_out) {
          float4* ho = reinterpret_cast<float4*>(h_out + static_cast<size_t>(m) * I) + 2 * idx;
          ho[0] = make_float4(hc[c][0].x, hc[c][0].y, hc[c][1].x, hc[c][1].y);
          ho[1] = make_float4(hc[c][2].x, hc[c][2].y, hc[c][3].x, hc[c][3].y);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fmaxf(fabsf(hc[c][e].x), fabsf(hc[c][e].y)));
      }
    }
    amax = block_reduce<true>(rq::scaled_absmax(amax, pre), sh.red);
    // every thread has read this buffer: the row after next streams into it
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();
      issue(j + 2);
    }
    const Enc en = make_enc(amax, qt);
    if (threadIdx.x == 0) sx[m] = en.scale;
    uint8_t* out = Xq + static_cast<size_t>(m) * I;
    uint8_t* out16 = x16 ? x16 + static_cast<size_t>(m) * I * 2 : nullptr;
    // pass 2: codes (warp-uniform steps: the code sums reduce over the warp)
#pragma unroll
    for (int c = 0; c < kSiluStreamNC; ++c) {
      const int idx = threadIdx.x + c * 1024;
      int2 v = make_int2(0, 0);
      if (idx < nvec) {
#pragma unroll
        for (int e = 0; e < 4; ++e) hc[c][e] = rq::mul2(hc[c][e], pre2);
        v = rq::store8(out, out16, idx, hc[c], en);
      }
      rq::sums_add_warp(sh.cnt, sums, idx, v);
    }
    rq::sums_end(sh.cnt, sums, m);
  }
  if (stop && threadIdx.x == 0) {
    // a copy timed out (the status is latched): wait, bounded, for the copies
    // still in flight before the shared memory is released
    for (int b = 0; b < 2; ++b) {
      const int consumed = (j + 1 - b) / 2;  // rows 0 .. j - 1 of buffer b (j & 1 == b)
      if (issued[b] > consumed) drain_bulk(&full[b], (issued[b] - 1) & 1, status);
    }
  }
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
  // W' = W / s; s = 1 (the per-step re-quantization of the folded weights)
  // divides exactly into w itself, so that case skips the division
  const bool unit = (s == 1.0f);
  // pass 1: absmax of W' (reads only)
  float amax = 0.0f;
  for (int idx = threadIdx.x; idx < nvec; idx += blockDim.x) {
    float w[8];
    load_w8<kF32>(row, idx, w);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(unit ? w[e] : __fdiv_rn(w[e], s)));
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
    if (!unit) {
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = __fdiv_rn(w[e], s);
    }
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
  const int t = row_threads(K / 8, M);
  if (t == 128 && K / 8 <= kSlimVPT * t)
    return launch_pdl(quant_act_kernel<kSlimVPT, 128, kDenseRows>, dim3(M), dim3(t), 0, st,
                      reinterpret_cast<const __nv_bfloat16*>(X), K, ldx, pre, qt, reinterpret_cast<uint8_t*>(Xq), sx,
                      reinterpret_cast<uint8_t*>(x16), sums);
  return launch_pdl(K / 8 <= kSlimVPT * t ? quant_act_kernel<kSlimVPT> : quant_act_kernel<kVPT>, dim3(M), dim3(t),
                    0, st, reinterpret_cast<const __nv_bfloat16*>(X), K, ldx, pre, qt, reinterpret_cast<uint8_t*>(Xq),
                    sx, reinterpret_cast<uint8_t*>(x16), sums);
}

cudaError_t launch_rmsnorm_quant(const void* X, int M, int K, long long ldx, const float* gamma, float eps,
                                 int qt, void* Xq, float* sx, float* ms_out, void* x16, CodeSums sums,
                                 cudaStream_t st) {
  if (x16 == nullptr) sums.asum = nullptr;
  const int t = row_threads(K / 8, M);
  if (t == 128 && K / 8 <= kSlimVPT * t)
    return launch_pdl(rmsnorm_quant_kernel<kSlimVPT, 128, kDenseRows>, dim3(M), dim3(t), 0, st,
                      reinterpret_cast<const __nv_bfloat16*>(X), K, ldx, gamma, eps, qt,
                      reinterpret_cast<uint8_t*>(Xq), sx, ms_out, reinterpret_cast<uint8_t*>(x16), sums);
  return launch_pdl(K / 8 <= kSlimVPT * t ? rmsnorm_quant_kernel<kSlimVPT> : rmsnorm_quant_kernel<kVPT>, dim3(M),
                    dim3(t), 0, st, reinterpret_cast<const __nv_bfloat16*>(X), K, ldx, gamma, eps, qt,
                    reinterpret_cast<uint8_t*>(Xq), sx, ms_out, reinterpret_cast<uint8_t*>(x16), sums);
}

cudaError_t launch_silu_mul_quant(const void* GU, int M, int I, long long ldgu, float pre, int qt, void* Xq,
                                  float* sx, float* h_out, void* x16, CodeSums sums, int* status, cudaStream_t st) {
  if (x16 == nullptr) sums.asum = nullptr;
  // two vectors (gate, up) are cached per position: half as many per thread
  const int t = row_threads(I / 8, M, kVPT / 2);
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  const int nvec = I / 8;
  if (sms > 0 && M > sms && status != nullptr && nvec > kRowThreads * (kVPT / 2) && I <= kSiluStreamMaxI &&
      dev >= 0 && dev < 64) {
    static bool attr_done[64] = {};
    const size_t smem = 8 * static_cast<size_t>(I);
    if (!attr_done[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(silu_mul_quant_stream_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(8 * kSiluStreamMaxI));
      if (e != cudaSuccess) return e;
      attr_done[dev] = true;
    }
    return launch_pdl(silu_mul_quant_stream_kernel, dim3(sms), dim3(1024), smem, st,
                      reinterpret_cast<const __nv_bfloat16*>(GU), M, I, ldgu, pre, qt, reinterpret_cast<uint8_t*>(Xq),
                      sx, h_out, reinterpret_cast<uint8_t*>(x16), sums, status);
  }
  if (sms > 0 && M > sms && nvec > kRowThreads * (kVPT / 2) && nvec <= 1024 * (kVPT / 2))
    return launch_pdl(silu_mul_quant_1k_kernel, dim3(M), dim3(1024), 0, st,
                      reinterpret_cast<const __nv_bfloat16*>(GU), I, ldgu, pre, qt, reinterpret_cast<uint8_t*>(Xq),
                      sx, h_out, reinterpret_cast<uint8_t*>(x16), sums);
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
