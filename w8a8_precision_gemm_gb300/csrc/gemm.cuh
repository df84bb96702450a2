// gemm.cuh -- the W8A8 GEMM with dequantizing epilogue on the sm_103a
// tensor cores (tcgen05 / TMEM, fed by TMA).
//
//   acc[m,n] = sum_k Xq[m,k] * Wq[n,k];   Y[m,n] = bf16((fp32(acc) * sx[m]) * sw[n])
//
// One CTA computes a 128 x BN tile of the accumulator for one range of K
// k-blocks ("split").  Warp roles:
//   warp 0      TMA producer: streams A and B tiles into a STAGES-deep ring.
//   warp 1      MMA issuer (one thread) and TMEM owner.
//   warps 2-5   epilogue: TMEM -> registers -> scales -> bf16 (or raw partials).
//   warps 6-13  (INT8 only) converters: int8 tiles -> fp16 tiles in the 128-byte
//               swizzled K-major layout the MMA reads.
//
// FP8-E4M3 runs tcgen05.mma kind::f8f6f4 directly on the TMA-loaded codes,
// fp32 accumulation in TMEM.
//
// INT8: this toolchain has no tcgen05 kind::i8 for sm_103a, so the int8 codes
// are widened to fp16 (every integer of magnitude <= 2048 is exact in fp16)
// and multiplied with kind::f16 into fp32 TMEM accumulators.  Each product is
// an integer of magnitude <= 128^2 and every partial sum over a chunk of 1024
// k stays within 1024 * 128^2 = 2^24, so the fp32 accumulation of one chunk
// is exact; the epilogue warps drain each chunk from TMEM,
// convert it to int32 and add it to an int32 running sum that also lives in
// TMEM.  Two TMEM partial buffers let the MMA fill one chunk while the other
// is drained.  The int32 result is therefore exact.
//
// Orientation: with SWAP the weight tile is the MMA's M side (128 output
// channels per CTA) and the tokens are its N side (BN <= 256) -- the layout for
// small-M decode, where every weight byte is read once.  Without SWAP the
// tokens are the M side (FP8 prefill; INT8 prefill without a workspace -- with
// one, INT8 at every M runs the TMEM-operand kernel of gemm_i8t.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "fused_quant.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace qurl {

// One work unit of a persistent GEMM CTA: a 128 x BN accumulator tile over
// one K split.  Units are numbered token tile fastest, so CTAs running at the
// same time share weight tiles (L2 reuse when there are several token tiles).
// Tile v's coordinates in the unit order of the CTA-pair prefill kernels:
// groups of `group` token tiles, then channel tiles, token tile fastest -- the
// pairs running together cover a few channel tiles of one token group, so a
// channel tile's weights are read from HBM once per token group and the
// group's activations stay in L2 while its channel tiles go by.  Only the last
// group can be short; group >= tiles_tok is token tile fastest over all.
__host__ __device__ __forceinline__ void group_tile(int tiles_tok, int tiles_ch, int group, int v, int& tok,
                                                    int& ch) {
  const int gi = v / (group * tiles_ch);
  const int gs = min(group, tiles_tok - gi * group);
  const int r = v - gi * group * tiles_ch;
  ch = r / gs;
  tok = gi * group + (r - ch * gs);
}

struct Unit {
  int a0, b0;    // first row of the A tile / of the B tile
  int kb0, nkb;  // k-block range
  int split;
};

template <bool SWAP, int BN>
__device__ __forceinline__ Unit unit_of(const GemmArgs& a, int u) {
  const int tok = u % a.tiles_tok;
  const int rest = u / a.tiles_tok;
  const int ch = rest % a.tiles_ch;
  const int sp = rest / a.tiles_ch;
  Unit w;
  w.a0 = (SWAP ? ch : tok) * 128;
  w.b0 = (SWAP ? tok : ch) * BN;
  w.kb0 = sp * a.kb_per_split;
  w.nkb = min(a.num_kb - w.kb0, a.kb_per_split);
  w.split = sp;
  return w;
}

// The units one CTA processes: blockIdx.x, blockIdx.x + gridDim.x, ... < end.
struct UnitRange {
  int u, stride, end;
};

__device__ __forceinline__ UnitRange unit_range(const GemmArgs& a) {
  return {static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), a.tiles_tok * a.tiles_ch * a.splits};
}

template <int QT, bool SWAP, int BN, int STAGES>
struct GemmCfg {
  static constexpr bool kInt8 = (QT == 0);
  static constexpr int BM = 128;                        // MMA M (rows of the A tile)
  static constexpr int BK = kInt8 ? 64 : 128;           // k per k-block (= bytes per code row)
  static constexpr int CSTAGES = kInt8 ? 3 : 0;         // fp16 stages (INT8)
  static constexpr int A_STAGE = BM * BK;               // bytes of a staged code tile
  static constexpr int B_STAGE = BN * BK;
  static constexpr int A_CONV = BM * 128;               // fp16 tile: rows x 64 halves
  static constexpr int B_CONV = BN * 128;
  static constexpr int SMEM_TILES = CSTAGES * (A_CONV + B_CONV) + STAGES * (A_STAGE + B_STAGE);
  static constexpr int SMEM_BYTES = SMEM_TILES + 1024;  // slack for 1024-byte alignment
  static constexpr int NUM_CONV = 256;                  // INT8 converter threads (warps 6-13), two groups
  static constexpr int CONV_GROUP = 128;                // threads of one group (alternate k-blocks)
  static constexpr int NUM_THREADS = kInt8 ? 192 + NUM_CONV : 192;
  static constexpr int TMEM_USED = kInt8 ? 3 * BN : 2 * BN;  // two accumulator buffers (+ int32 sum)
  static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                   : TMEM_USED <= 64  ? 64
                                   : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256
                                                      : 512;
  static constexpr int CHUNK_KB = kInt8 ? (1024 / BK) : (1 << 30);  // k-blocks per exact chunk
  static constexpr int MMA_K_BYTES = 32;                // k per MMA: 32 e4m3 or 16 f16
  static constexpr int MMAS_PER_KB = 128 / MMA_K_BYTES; // a k-block row is 128 bytes in smem
  static constexpr uint32_t IDESC = umma_idesc_f32acc(0, 0, BM, BN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(TMEM_USED <= 512, "TMEM has 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

template <int STAGES, int CSTAGES>
struct GemmBarriers {
  uint64_t full[STAGES];    // TMA -> consumer (tx bytes)
  uint64_t empty[STAGES];   // consumer -> TMA
  uint64_t cfull[CSTAGES > 0 ? CSTAGES : 1];   // converters -> MMA
  uint64_t cempty[CSTAGES > 0 ? CSTAGES : 1];  // MMA -> converters
  uint64_t pfull[2];        // MMA -> epilogue (accumulator chunk ready)
  uint64_t pempty[2];       // epilogue -> MMA (TMEM buffer drained)
  uint64_t done;            // MMA drain on the error path
  uint32_t tmem_base;
};

// Wait (bounded, ignoring latched errors) for async copies/MMAs a thread has
// issued itself, so nothing is in flight when the CTA leaves.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, kDevOk, kDevTimeout);
      return;
    }
  }
}

// Warp-uniform bounded wait: every lane polls, then the warp agrees.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status) {
  const bool ok = mbar_wait(bar, parity, status);
  return __all_sync(0xFFFFFFFFu, ok) != 0;
}

__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

// Bounded wait until *count > j (a counter another warp of the CTA raises).
__device__ __forceinline__ bool wait_count(const uint32_t* count, uint32_t j, int* status) {
  if (ld_acquire_cta(count) > j) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_cta(count) > j) return true;
    if ((it & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(status) != kDevOk) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(status, kDevOk, kDevTimeout);
        return false;
      }
    }
  }
}

// 16 int8 codes -> 16 fp16 values, exactly: with u = c + 128 in [0, 255], the
// fp16 with bits 0x6400 | u is 1024 + u; subtracting 1152 leaves c.
__device__ __forceinline__ void i8x16_to_f16x16(const uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
  uint32_t o[8];
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p0 = __byte_perm(w[i], 0x64646464u, 0x4140);
    const uint32_t p1 = __byte_perm(w[i], 0x64646464u, 0x4342);
    __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), bias);
    __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), bias);
    o[2 * i] = *reinterpret_cast<uint32_t*>(&h0);
    o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&h1);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Widen a staged int8 tile (rows x 64 bytes, row-major, unswizzled) into an
// fp16 tile of rows x 128 bytes in the 128-byte swizzled K-major layout: the
// 16-byte chunk c of row r lives at (r/8)*1024 + (r%8)*128 + ((c ^ (r%8))*16).
// nthreads threads; thread t converts 16 codes (chunk t%4) of rows t/4,
// t/4 + nthreads/4, ...  A quarter-warp reads 128 contiguous bytes and writes 8
// distinct chunk positions, so neither side has bank conflicts.
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int rows, int t, int nthreads) {
  const int j = t & 3;
  for (int r = t >> 2; r < rows; r += nthreads >> 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + r * 64 + j * 16);
    uint4 lo, hi;
    i8x16_to_f16x16(v, lo, hi);
    uint8_t* row = dst + (r >> 3) * 1024 + (r & 7) * 128;
    *reinterpret_cast<uint4*>(row + (((2 * j) ^ (r & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
  }
}

// One step of a warp transpose.  Before it each lane holds nb = 2^S
// consecutive channels (the lane's own number with its low S bits cleared,
// plus ci) of nt = 32 / nb tokens (its low S bits, plus ti * nb), as
// x[ci * nt + ti]; lane pairs at distance nb swap the half of their tokens the
// other one keeps, leaving 2 nb channels of nt / 2 tokens.
template <int S>
__device__ __forceinline__ void transpose_step(uint32_t (&x)[32], int lane) {
  constexpr int nb = 1 << S, nt = 32 >> S, h = nt / 2;
  const bool bit = ((lane >> S) & 1) != 0;
  uint32_t y[32];
#pragma unroll
  for (int ci = 0; ci < nb; ++ci) {
#pragma unroll
    for (int t2 = 0; t2 < h; ++t2) {
      const uint32_t e = x[ci * nt + 2 * t2], o = x[ci * nt + 2 * t2 + 1];
      const uint32_t keep = bit ? o : e;
      const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, bit ? e : o, nb);
      y[ci * h + t2] = bit ? recv : keep;         // channel ci: this lane's if bit == 0
      y[(nb + ci) * h + t2] = bit ? keep : recv;  // channel nb + ci: this lane's if bit == 1
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = y[j];
}

template <typename T>
__device__ __forceinline__ float acc_to_float(uint32_t bits) {
  if constexpr (std::is_same<T, int>::value) return static_cast<float>(static_cast<int>(bits));
  else return __uint_as_float(bits);
}

// The swap orientation's block of one warp: lane L holds channel a0 + (i & ~31)
// + L for the tokens b0 + c0 + j, j < 32.  One store per lane and token would
// write 2 (bf16) or 4 bytes per lane; three transpose steps first leave each
// lane 8 consecutive channels ((L & ~7) + ci) of 4 tokens ((L & 7) + 8 t), so
// each store writes 16 contiguous bytes.  sx_lane / sw_lane: lane L's scale of
// token b0 + c0 + L and of channel a0 + (i & ~31) + L (loaded by the caller
// ahead of time; used in mode kModeBf16).  Called by all 32 lanes of the warp.
template <int BN, typename T>
__device__ __forceinline__ void emit32_swap(const GemmArgs& a, int mode, int a0, int b0, int split, int i, int c0,
                                            const T (&v)[32], float sx_lane, float sw_lane) {
  const int M = a.M, N = a.N;
  const int L = threadIdx.x & 31;
  uint32_t x[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = *reinterpret_cast<const uint32_t*>(&v[j]);
  transpose_step<0>(x, L);
  transpose_step<1>(x, L);
  transpose_step<2>(x, L);
  const int n0 = a0 + (i & ~31) + (L & ~7);  // the lane's first channel; x[ci * 4 + t]
  if (mode == kModeAcc) {
    T* part = reinterpret_cast<T*>(a.part) + static_cast<size_t>(split) * M * N;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int jj = (L & 7) + 8 * t;
      const int m = b0 + c0 + jj;
      if (c0 + jj >= BN || m >= M) continue;
      T* dst = part + static_cast<size_t>(m) * N + n0;
      if (n0 + 8 <= N && (N & 3) == 0) {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(x[t], x[4 + t], x[8 + t], x[12 + t]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(x[16 + t], x[20 + t], x[24 + t], x[28 + t]);
      } else {
#pragma unroll
        for (int ci = 0; ci < 8; ++ci)
          if (n0 + ci < N) dst[ci] = *reinterpret_cast<const T*>(&x[ci * 4 + t]);
      }
    }
    return;
  }
  // dequantizing epilogue: y = bf16((fp32(acc) * sx[m]) * sw[n])
  float swv[8];
#pragma unroll
  for (int ci = 0; ci < 8; ++ci) swv[ci] = __shfl_sync(0xFFFFFFFFu, sw_lane, (L & ~7) + ci);
  float sxv[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) sxv[t] = __shfl_sync(0xFFFFFFFFu, sx_lane, (L & 7) + 8 * t);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int jj = (L & 7) + 8 * t;
    const int m = b0 + c0 + jj;
    if (c0 + jj >= BN || m >= M) continue;
    const float sxm = sxv[t];
    uint32_t packed[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float y0 = __fmul_rn(__fmul_rn(acc_to_float<T>(x[(2 * h) * 4 + t]), sxm), swv[2 * h]);
      const float y1 = __fmul_rn(__fmul_rn(acc_to_float<T>(x[(2 * h + 1) * 4 + t]), sxm), swv[2 * h + 1]);
      __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);  // one paired RNE conversion
      packed[h] = *reinterpret_cast<uint32_t*>(&p);
    }
    __nv_bfloat16* dst = a.Y + static_cast<size_t>(m) * a.ldy + n0;
    if (n0 + 8 <= N) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    } else {
#pragma unroll
      for (int ci = 0; ci < 8; ++ci)
        if (n0 + ci < N) dst[ci] = reinterpret_cast<const __nv_bfloat16*>(packed)[ci];
    }
  }
}

// Scales the swap epilogue hands to emit32_swap: this lane's token b0 + c0 +
// lane, and its channel n (0 where out of range or not needed).
// (coherent loads: in a fused call this grid itself wrote sx)
__device__ __forceinline__ float token_scale(const GemmArgs& a, int mode, int m) {
  return (mode == kModeBf16 && m < a.M) ? __ldcg(a.sx + m) : 0.0f;
}
__device__ __forceinline__ float channel_scale(const GemmArgs& a, int mode, int n) {
  return (mode == kModeBf16 && n < a.N) ? __ldg(a.sw + n) : 0.0f;
}

// Prefill orientation: write 32 accumulator values of one tile row.  i = row
// of the A tile (TMEM lane = token), columns c0..c0+31 of the B tile.
// (part_base, when given, replaces a.part: a whole-K unit of a call that also
// has split units writes its raw sums straight to the accumulator output)
template <int BN, typename T>
__device__ __forceinline__ void emit32(const GemmArgs& a, int mode, int a0, int b0, int split, int i, int c0,
                                       const T (&v)[32], void* part_base = nullptr) {
  const int M = a.M, N = a.N;
  if (mode == kModeAcc) {
    T* part = reinterpret_cast<T*>(part_base ? part_base : a.part) + static_cast<size_t>(split) * M * N;
    const int m = a0 + i;
    if (m < M) {
      T* dst = part + static_cast<size_t>(m) * N + (b0 + c0);
      const int nvalid = min(32, min(BN - c0, N - (b0 + c0)));
      if (nvalid == 32 && (N & 3) == 0) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<uint4*>(dst + j) =
              make_uint4(*reinterpret_cast<const uint32_t*>(&v[j]), *reinterpret_cast<const uint32_t*>(&v[j + 1]),
                         *reinterpret_cast<const uint32_t*>(&v[j + 2]),
                         *reinterpret_cast<const uint32_t*>(&v[j + 3]));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) dst[j] = v[j];
      }
    }
    return;
  }
  // dequantizing epilogue: y = bf16((fp32(acc) * sx[m]) * sw[n])
  {
    const int m = a0 + i;
    if (m >= M) return;
    const float sxm = __ldg(a.sx + m);
    __nv_bfloat16* dst = a.Y + static_cast<size_t>(m) * a.ldy + (b0 + c0);
    const int nvalid = min(32, min(BN - c0, N - (b0 + c0)));
    if (nvalid == 32) {
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float y0 = __fmul_rn(__fmul_rn(static_cast<float>(v[j]), sxm), __ldg(a.sw + b0 + c0 + j));
        const float y1 = __fmul_rn(__fmul_rn(static_cast<float>(v[j + 1]), sxm), __ldg(a.sw + b0 + c0 + j + 1));
        __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);  // one paired RNE conversion
        packed[j / 2] = *reinterpret_cast<uint32_t*>(&p);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        reinterpret_cast<uint4*>(dst)[q] =
            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nvalid) {
          const float y = __fmul_rn(__fmul_rn(static_cast<float>(v[j]), sxm), __ldg(a.sw + b0 + c0 + j));
          dst[j] = __float2bfloat16_rn(y);
        }
    }
  }
}

// The dequantizing write of 32 columns of one tile row whose scales are
// already in registers (loaded while the accumulator filled): sxm = sx[m],
// sw_lane = sw[n0 + lane] (0 past N).  The same products in the same order as
// emit32's; every lane of the warp calls it (the channel scales are shuffled).
template <typename T>
__device__ __forceinline__ void emit32_prescaled(const GemmArgs& a, int m, int n0, const T (&v)[32], float sxm,
                                                 float sw_lane) {
  const bool row = m < a.M;
  const int nvalid = min(32, a.N - n0);
  __nv_bfloat16* dst = a.Y + static_cast<size_t>(row ? m : 0) * a.ldy + n0;
  if (nvalid == 32) {
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float s0 = __shfl_sync(0xFFFFFFFFu, sw_lane, j), s1 = __shfl_sync(0xFFFFFFFFu, sw_lane, j + 1);
      const float y0 = __fmul_rn(__fmul_rn(static_cast<float>(v[j]), sxm), s0);
      const float y1 = __fmul_rn(__fmul_rn(static_cast<float>(v[j + 1]), sxm), s1);
      __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);
      packed[j / 2] = *reinterpret_cast<uint32_t*>(&p);
    }
    if (row) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        reinterpret_cast<uint4*>(dst)[q] =
            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float sj = __shfl_sync(0xFFFFFFFFu, sw_lane, j);
      if (row && j < nvalid) dst[j] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(static_cast<float>(v[j]), sxm), sj));
    }
  }
}

template <int QT, bool SWAP, int BN, int STAGES>
__global__ void __launch_bounds__(GemmCfg<QT, SWAP, BN, STAGES>::NUM_THREADS, 1)
    w8a8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs args) {
  using C = GemmCfg<QT, SWAP, BN, STAGES>;
  __shared__ GemmBarriers<STAGES, C::CSTAGES> bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* convA = smem;                                   // [CSTAGES][A_CONV]  (INT8)
  uint8_t* convB = convA + C::CSTAGES * C::A_CONV;         // [CSTAGES][B_CONV]  (INT8)
  uint8_t* stA = convB + C::CSTAGES * C::B_CONV;           // [STAGES][A_STAGE]
  uint8_t* stB = stA + STAGES * C::A_STAGE;                // [STAGES][B_STAGE]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const UnitRange R = unit_range(args);
  int* status = args.status;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], C::kInt8 ? C::CONV_GROUP : 1);
    }
#pragma unroll
    for (int s = 0; s < (C::CSTAGES > 0 ? C::CSTAGES : 1); ++s) {
      mbar_init(&bars.cfull[s], C::CONV_GROUP);
      mbar_init(&bars.cempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.pfull[b], 1);
      mbar_init(&bars.pempty[b], 128);
    }
    mbar_init(&bars.done, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  griddep_launch_dependents();
  // a fused call quantizes its input rows first (decode orientation; FP8)
  const bool fused = SWAP && !C::kInt8 && args.fq.kind != kFuseNone;
  if (warp != 0 || fused) griddep_wait();

  const uint64_t polA = SWAP ? l2_policy_evict_first() : l2_policy_evict_last();
  const uint64_t polB = SWAP ? l2_policy_evict_last() : l2_policy_evict_normal();
  // Weight tiles of the first stages may stream in while the previous kernel
  // (which, per w_prefetch, does not write Wq) is finishing, or, in a fused
  // call, while this kernel quantizes its input rows.
  int npre = 0;  // meaningful in the producer thread
  if (warp == 0 && lane == 0 && (args.w_prefetch || fused) && !args.fault && R.u < R.end) {
    const Unit w = unit_of<SWAP, BN>(args, R.u);
    npre = min(STAGES, w.nkb);
    for (int it = 0; it < npre; ++it) {
      mbar_arrive_expect_tx(&bars.full[it], C::A_STAGE + C::B_STAGE);
      const int kc = (w.kb0 + it) * C::BK;
      if (SWAP)
        tma_load_2d(stA + it * C::A_STAGE, &tmA, kc, w.a0, &bars.full[it], polA);
      else
        tma_load_2d(stB + it * C::B_STAGE, &tmB, kc, w.b0, &bars.full[it], polB);
    }
  }
  bool run = true;
  if constexpr (SWAP && !C::kInt8) {
    if (fused)  // the token stages are free until the handoff: they hold the rows' reduction scratch
      run = fused_quant_prologue<4>(args.fq, args.fsums, args.M, args.K, QT,
                                    *reinterpret_cast<rq::RowScratch*>(stB), args.status, args.fault);
  }

  if (!run) {
    // the handoff ran out (the timeout is latched): no role runs; the weight
    // copies already issued land before the CTA leaves (their barriers also
    // count the token halves never issued: bounded waits)
    if (warp == 0 && lane == 0)
      for (int j = 0; j < npre; ++j) mbar_wait_drain(&bars.full[j], 0, args.status);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if (!fused) griddep_wait();
      int g = 0;  // k-blocks issued by this CTA (ring position)
      bool ok = true;
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<SWAP, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          const int s = g % STAGES;
          const int kc = (w.kb0 + it) * C::BK;
          if (args.fault && g == 0) continue;  // injected fault: this stage never fills
          if (g < npre) {  // the weight half is in flight; add the activation half
            if (SWAP)
              tma_load_2d(stB + s * C::B_STAGE, &tmB, kc, w.b0, &bars.full[s], polB);
            else
              tma_load_2d(stA + s * C::A_STAGE, &tmA, kc, w.a0, &bars.full[s], polA);
            continue;
          }
          if (!mbar_wait(&bars.empty[s], ((g / STAGES) & 1) ^ 1, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.full[s], C::A_STAGE + C::B_STAGE);
          tma_load_2d(stA + s * C::A_STAGE, &tmA, kc, w.a0, &bars.full[s], polA);
          tma_load_2d(stB + s * C::B_STAGE, &tmB, kc, w.b0, &bars.full[s], polB);
        }
      }
      if (!ok) {  // let the copies still in flight land before the CTA leaves
        for (int it = max(0, g - STAGES); it < g; ++it)
          mbar_wait_drain(&bars.full[it % STAGES], (it / STAGES) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int g = 0;   // k-blocks consumed
      int cg = 0;  // accumulator chunks started (buffer cg & 1)
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<SWAP, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          const int kin = it % C::CHUNK_KB;
          const int buf = cg & 1;
          if (kin == 0 && cg >= 2) {  // the epilogue must have drained this buffer's previous chunk
            if (!mbar_wait(&bars.pempty[buf], ((cg >> 1) - 1) & 1, status)) {
              ok = false;
              break;
            }
          }
          const uint32_t d = tmem + buf * BN;
          if constexpr (!C::kInt8) {
            const int s = g % STAGES;
            if (!mbar_wait(&bars.full[s], (g / STAGES) & 1, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_addr(stA + s * C::A_STAGE);
            const uint32_t sb = smem_addr(stB + s * C::B_STAGE);
#pragma unroll
            for (int kk = 0; kk < C::MMAS_PER_KB; ++kk)
              umma_f8f6f4(d, umma_desc_sw128(sa + kk * C::MMA_K_BYTES), umma_desc_sw128(sb + kk * C::MMA_K_BYTES),
                          C::IDESC, (kin | kk) != 0);
            umma_commit(&bars.empty[s]);
          } else {
            const int cs = g % C::CSTAGES;
            if (!mbar_wait(&bars.cfull[cs], (g / C::CSTAGES) & 1, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_addr(convA + cs * C::A_CONV);
            const uint32_t sb = smem_addr(convB + cs * C::B_CONV);
#pragma unroll
            for (int kk = 0; kk < C::MMAS_PER_KB; ++kk)
              umma_f16(d, umma_desc_sw128(sa + kk * C::MMA_K_BYTES), umma_desc_sw128(sb + kk * C::MMA_K_BYTES),
                       C::IDESC, (kin | kk) != 0);
            umma_commit(&bars.cempty[cs]);
          }
          if (kin == C::CHUNK_KB - 1 || it == w.nkb - 1) {
            umma_commit(&bars.pfull[buf]);
            ++cg;
          }
        }
      }
      if (!ok) {  // no MMA may still be writing TMEM when it is released
        umma_commit(&bars.done);
        mbar_wait_drain(&bars.done, 0, status);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int i = q * 32 + lane;          // row of the A tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tR = lane_base + 2 * BN;  // INT8: int32 running sum
    const int emode = args.mode;
    int cg = 0;
    bool ok = true;
    for (int u = R.u; u < R.end && ok; u += R.stride) {
      const Unit w = unit_of<SWAP, BN>(args, u);
      const int nch = (w.nkb + C::CHUNK_KB - 1) / C::CHUNK_KB;
      // swap: scales of this lane's channel and of its token in the first
      // 32-token block, loaded while the accumulator is being filled
      const float sw_lane = SWAP ? channel_scale(args, emode, w.a0 + i) : 0.0f;
      const float sx_first = SWAP ? token_scale(args, emode, w.b0 + lane) : 0.0f;
      for (int c = 0; c < nch; ++c, ++cg) {
        const int buf = cg & 1;
        if (!warp_wait(&bars.pfull[buf], (cg >> 1) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool last = (c == nch - 1);
        float sx_lane = sx_first;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          // the next block's token scale, in flight while this block is written
          const float sx_next = (SWAP && last && c0 + 32 < BN) ? token_scale(args, emode, w.b0 + c0 + 32 + lane) : 0.0f;
          uint32_t p[32];
          tmem_ld32(lane_base + buf * BN + c0, p);
          if constexpr (!C::kInt8) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(p[j]);
            if constexpr (SWAP)
              emit32_swap<BN, float>(args, emode, w.a0, w.b0, w.split, i, c0, v, sx_lane, sw_lane);
            else
              emit32<BN, float>(args, emode, w.a0, w.b0, w.split, i, c0, v);
          } else {
            int v[32];
            if (c > 0) {
              uint32_t rs[32];
              tmem_ld32(tR + c0, rs);
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = static_cast<int>(rs[j]) + __float2int_rn(__uint_as_float(p[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float2int_rn(__uint_as_float(p[j]));
            }
            if (!last) {
              uint32_t wv[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) wv[j] = static_cast<uint32_t>(v[j]);
              tmem_st32(tR + c0, wv);
            } else if constexpr (SWAP) {
              emit32_swap<BN, int>(args, emode, w.a0, w.b0, w.split, i, c0, v, sx_lane, sw_lane);
            } else {
              emit32<BN, int>(args, emode, w.a0, w.b0, w.split, i, c0, v);
            }
          }
          sx_lane = sx_next;
        }
        if (C::kInt8 && !last) tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.pempty[buf]);
      }
    }
  } else {
    // ------------------------------------------------------------ converters (INT8)
    // Two groups of 128 threads take alternate k-blocks, so two k-blocks are
    // widened at a time.
    if constexpr (C::kInt8) {
      const int t = (threadIdx.x - 192) & (C::CONV_GROUP - 1);
      const int grp = (threadIdx.x - 192) / C::CONV_GROUP;
      int g = 0;
      bool ok = true;
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<SWAP, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          if ((g & 1) != grp) continue;
          const int s = g % STAGES;
          if (!warp_wait(&bars.full[s], (g / STAGES) & 1, status)) {
            ok = false;
            break;
          }
          const int cs = g % C::CSTAGES;
          if (!warp_wait(&bars.cempty[cs], ((g / C::CSTAGES) & 1) ^ 1, status)) {
            ok = false;
            break;
          }
          convert_tile(stA + s * C::A_STAGE, convA + cs * C::A_CONV, C::BM, t, C::CONV_GROUP);
          convert_tile(stB + s * C::B_STAGE, convB + cs * C::B_CONV, BN, t, C::CONV_GROUP);
          fence_proxy_async_smem();
          mbar_arrive(&bars.empty[s]);
          mbar_arrive(&bars.cfull[cs]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Split-K reduction in a fixed order (z = 0, 1, ...), then either the
// dequantizing epilogue (Y != nullptr) or the raw sum (acc_out).  Every thread
// takes 4 consecutive outputs (16-byte loads of each partial) when N % 4 == 0.
template <typename T>
__global__ void splitk_reduce_kernel(const T* __restrict__ part, int splits, int M, int N,
                                     const float* __restrict__ sx, const float* __restrict__ sw,
                                     __nv_bfloat16* __restrict__ Y, long long ldy, T* __restrict__ acc_out) {
  griddep_wait();
  griddep_launch_dependents();
  const size_t total = static_cast<size_t>(M) * N;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const bool vec = (N & 3) == 0;
  const size_t items = vec ? total / 4 : total;
  for (size_t it = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items; it += stride) {
    const int w = vec ? 4 : 1;
    const size_t idx = it * w;
    T s[4] = {};
    for (int z = 0; z < splits; ++z) {
      const T* p = part + static_cast<size_t>(z) * total + idx;
      if (vec) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(p));
        s[0] += *reinterpret_cast<const T*>(&v.x);
        s[1] += *reinterpret_cast<const T*>(&v.y);
        s[2] += *reinterpret_cast<const T*>(&v.z);
        s[3] += *reinterpret_cast<const T*>(&v.w);
      } else {
        s[0] += __ldcg(p);
      }
    }
    const int m = static_cast<int>(idx / N);
    const int n0 = static_cast<int>(idx - static_cast<size_t>(m) * N);
    for (int e = 0; e < w; ++e) {
      if (Y != nullptr) {
        const float y = __fmul_rn(__fmul_rn(static_cast<float>(s[e]), __ldg(sx + m)), __ldg(sw + n0 + e));
        Y[static_cast<size_t>(m) * ldy + n0 + e] = __float2bfloat16_rn(y);
      } else {
        acc_out[idx + e] = s[e];
      }
    }
  }
}

// The unit grid (token tiles, channel tiles, splits) becomes a persistent
// launch of one CTA per SM (fewer when there are fewer units).
int persistent_ctas(const GemmArgs& a);

// attr_done: the caller's per-instantiation flags (one per device) recording
// that the kernel's dynamic shared-memory limit has been raised -- every kernel
// needs its own, although many share this function's signature type.
template <typename Kern>
cudaError_t launch_persistent(Kern kern, int threads, int smem, const CUtensorMap& ta, const CUtensorMap& tb,
                              const GemmArgs& args_in, dim3 grid, cudaStream_t stream, bool (&attr_done)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  GemmArgs args = args_in;
  args.tiles_tok = grid.x;
  args.tiles_ch = grid.y;
  args.splits = grid.z;
  return launch_pdl(kern, dim3(persistent_ctas(args)), dim3(threads), smem, stream, ta, tb, args);
}

template <int QT, bool SWAP, int BN, int STAGES>
cudaError_t launch_gemm_inst(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args, dim3 grid,
                             cudaStream_t stream) {
  using C = GemmCfg<QT, SWAP, BN, STAGES>;
  static bool attr_done[64] = {};
  return launch_persistent(w8a8_gemm_kernel<QT, SWAP, BN, STAGES>, C::NUM_THREADS, C::SMEM_BYTES, ta, tb, args,
                           grid, stream, attr_done);
}

}  // namespace qurl
