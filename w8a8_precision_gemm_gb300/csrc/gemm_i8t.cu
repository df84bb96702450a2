// gemm_i8t.cu -- the INT8 W8A8 GEMM for decode (weights on the MMA M side),
// with the weight operand widened into TMEM.
//
// Per 128-deep k-block a CTA
//   * TMA-loads its 128 weight rows of int8 codes (16 KB, 128-byte swizzle) and
//     the tokens' codes already widened to fp16 (BN rows x 256 B, two swizzled
//     halves) -- the fp16 copy of the activation codes is made once per call,
//     not once per CTA;
//   * converter warps (one thread per weight row = TMEM lane) read the row's
//     128 codes from shared memory, widen them to fp16 (exact) and store them
//     into a TMEM stage with tcgen05.st: the MMA takes its A operand from TMEM,
//     so the widened weights never travel through shared memory;
//   * the MMA warp issues tcgen05.mma kind::f16 [d], [a_tmem], b_desc with fp32
//     accumulation; every 1024-deep chunk is exact (|partial| < 1024 * 127^2 <
//     2^24) and the epilogue warps drain it into an int32 running sum in TMEM,
//     exactly as in the shared-memory INT8 kernel (gemm.cuh).
// Shared-memory traffic per weight byte: 1 (TMA) + 1 (converter read) + 4
// (fp16 activations in and out, amortised over the 128 weight rows of the
// tile at BN = 64) -- half of widening both operands in shared memory.
#include "gemm.cuh"

namespace qurl {

template <int BN, int STAGES, int ASTAGES>
struct I8tCfg {
  static constexpr int BM = 128;
  static constexpr int BK = 128;                          // k per k-block
  static constexpr int W_STAGE = BM * BK;                 // int8 weight tile
  static constexpr int X_HALF = BN * 128;                 // fp16 [BN][64] swizzled half
  static constexpr int X_STAGE = 2 * X_HALF;
  static constexpr int SMEM_BYTES = STAGES * (W_STAGE + X_STAGE) + 1024;
  static constexpr int NUM_THREADS = 448;  // TMA, MMA, 4 epilogue warps, 8 converter warps
  static constexpr int A_BASE = ((3 * BN + 63) / 64) * 64;  // TMEM column of the first A stage
  static constexpr int A_COLS = 64;                       // 128 fp16 per lane per k-block
  static constexpr int TMEM_USED = A_BASE + ASTAGES * A_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
  static constexpr int CHUNK_KB = 1024 / BK;
  static constexpr uint32_t IDESC = umma_idesc_f32acc(0, 0, BM, BN);  // f16 x f16 -> f32
  static_assert(TMEM_USED <= 512, "TMEM has 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int STAGES, int ASTAGES>
struct I8tBarriers {
  uint64_t full[STAGES];     // TMA (weights + fp16 activations) landed
  uint64_t empty[STAGES];    // a converter group read the weights (128) and the MMA read the activations (1)
  uint64_t afull[ASTAGES];   // converters -> MMA: A stage written to TMEM
  uint64_t aempty[ASTAGES];  // MMA -> converters: A stage consumed
  uint64_t pfull[2];
  uint64_t pempty[2];
  uint64_t done;
  uint32_t tmem_base;
};

template <int BN, int STAGES, int ASTAGES>
__global__ void __launch_bounds__(448, 1)
    w8a8_gemm_i8t_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX16,
                         const GemmArgs args) {
  using C = I8tCfg<BN, STAGES, ASTAGES>;
  __shared__ I8tBarriers<STAGES, ASTAGES> bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stW = smem;                           // [STAGES][W_STAGE]
  uint8_t* stX = stW + STAGES * C::W_STAGE;      // [STAGES][X_STAGE]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const UnitRange R = unit_range(args);
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 129);  // one converter group (128 threads) + the MMA's commit
    }
    for (int s = 0; s < ASTAGES; ++s) {
      mbar_init(&bars.afull[s], 128);
      mbar_init(&bars.aempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.pfull[b], 1);
      mbar_init(&bars.pempty[b], 128);
    }
    mbar_init(&bars.done, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX16);
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
  if (warp != 0) griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t polW = l2_policy_evict_first();
      const uint64_t polX = l2_policy_evict_last();
      // weight tiles of the first stages stream in while the previous kernel
      // (which, per w_prefetch, does not write Wq) is finishing
      int npre = 0;
      if (args.w_prefetch && !args.fault && R.u < R.end) {
        const Unit w = unit_of<true, BN>(args, R.u);
        npre = min(STAGES, w.nkb);
        for (int it = 0; it < npre; ++it) {
          mbar_arrive_expect_tx(&bars.full[it], C::W_STAGE + C::X_STAGE);
          tma_load_2d(stW + it * C::W_STAGE, &tmW, (w.kb0 + it) * C::BK, w.a0, &bars.full[it], polW);
        }
      }
      griddep_wait();
      int g = 0;
      bool ok = true;
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<true, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          const int s = g % STAGES;
          const int kb = w.kb0 + it;
          if (args.fault && g == 0) continue;  // injected fault: this stage never fills
          if (g >= npre) {
            if (!mbar_wait(&bars.empty[s], ((g / STAGES) & 1) ^ 1, status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars.full[s], C::W_STAGE + C::X_STAGE);
            tma_load_2d(stW + s * C::W_STAGE, &tmW, kb * C::BK, w.a0, &bars.full[s], polW);
          }
          uint8_t* xs = stX + s * C::X_STAGE;
          tma_load_2d(xs, &tmX16, kb * C::BK * 2, w.b0, &bars.full[s], polX);
          tma_load_2d(xs + C::X_HALF, &tmX16, kb * C::BK * 2 + 128, w.b0, &bars.full[s], polX);
        }
      }
      if (!ok) {
        for (int it = max(0, g - STAGES); it < g; ++it)
          mbar_wait_drain(&bars.full[it % STAGES], (it / STAGES) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int g = 0, cg = 0;
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<true, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          const int kin = it % C::CHUNK_KB;
          const int buf = cg & 1;
          if (kin == 0 && cg >= 2) {
            if (!mbar_wait(&bars.pempty[buf], ((cg >> 1) - 1) & 1, status)) {
              ok = false;
              break;
            }
          }
          const int s = g % STAGES;
          const int as = g % ASTAGES;
          if (!mbar_wait(&bars.full[s], (g / STAGES) & 1, status) ||
              !mbar_wait(&bars.afull[as], (g / ASTAGES) & 1, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + buf * BN;
          const uint32_t a_t = tmem + C::A_BASE + as * C::A_COLS;
          const uint32_t xs = smem_addr(stX + s * C::X_STAGE);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t b_addr = xs + (kk >> 2) * C::X_HALF + (kk & 3) * 32;
            umma_f16_tmem_a(d, a_t + kk * 8, umma_desc_sw128(b_addr), C::IDESC, (kin | kk) != 0);
          }
          umma_commit(&bars.empty[s]);
          umma_commit(&bars.aempty[as]);
          if (kin == C::CHUNK_KB - 1 || it == w.nkb - 1) {
            umma_commit(&bars.pfull[buf]);
            ++cg;
          }
        }
      }
      if (!ok) {
        umma_commit(&bars.done);
        mbar_wait_drain(&bars.done, 0, status);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue (chunk drains)
    const int q = warp & 3;
    const int i = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tR = lane_base + 2 * BN;
    const int emode = args.mode;
    int cg = 0;
    bool ok = true;
    for (int u = R.u; u < R.end && ok; u += R.stride) {
      const Unit w = unit_of<true, BN>(args, u);
      const int nch = (w.nkb + C::CHUNK_KB - 1) / C::CHUNK_KB;
      for (int c = 0; c < nch; ++c, ++cg) {
        const int buf = cg & 1;
        if (!warp_wait(&bars.pfull[buf], (cg >> 1) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool last = (c == nch - 1);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t p[32];
          tmem_ld32(lane_base + buf * BN + c0, p);
          int v[32];
          if (c > 0) {
            uint32_t rs[32];
            tmem_ld32(tR + c0, rs);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = static_cast<int>(rs[j]) + __float2int_rn(__uint_as_float(p[j]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float2int_rn(__uint_as_float(p[j]));
          }
          if (!last) {
            uint32_t wv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) wv[j] = static_cast<uint32_t>(v[j]);
            tmem_st32(tR + c0, wv);
          } else {
            emit32<true, BN, int>(args, emode, w.a0, w.b0, w.split, i, c0, v);
          }
        }
        if (!last) tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.pempty[buf]);
      }
    }
  } else {
    // ------------------------------------------------------------ converters: weights -> fp16 in TMEM
    // Two groups of four warps (one per TMEM lane quadrant, one weight row per
    // lane) take alternate k-blocks, so two k-blocks are widened at a time: a
    // group's k-block is a serial chain (wait, load, widen, tcgen05.st, wait,
    // signal) and the groups overlap theirs.
    const int q = warp & 3;
    const int grp = (warp - 6) >> 2;
    const int i = q * 32 + lane;  // weight row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int g = 0;
    bool ok = true;
    for (int u = R.u; u < R.end && ok; u += R.stride) {
      const Unit w = unit_of<true, BN>(args, u);
      for (int it = 0; it < w.nkb; ++it, ++g) {
        if ((g & 1) != grp) continue;
        const int s = g % STAGES;
        const int as = g % ASTAGES;
        if (!warp_wait(&bars.full[s], (g / STAGES) & 1, status) ||
            !warp_wait(&bars.aempty[as], ((g / ASTAGES) & 1) ^ 1, status)) {
          ok = false;
          break;
        }
        const uint8_t* wrow = stW + s * C::W_STAGE + (i >> 3) * 1024 + (i & 7) * 128;
        const uint32_t a_t = lane_base + C::A_BASE + as * C::A_COLS;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = half * 4 + jj;  // 16-byte chunk = k 16j .. 16j+15
            const uint4 raw = *reinterpret_cast<const uint4*>(wrow + ((j ^ (i & 7)) << 4));
            uint4 lo, hi;
            i8x16_to_f16x16(raw, lo, hi);
            v[8 * jj + 0] = lo.x; v[8 * jj + 1] = lo.y; v[8 * jj + 2] = lo.z; v[8 * jj + 3] = lo.w;
            v[8 * jj + 4] = hi.x; v[8 * jj + 5] = hi.y; v[8 * jj + 6] = hi.z; v[8 * jj + 7] = hi.w;
          }
          tmem_st32(a_t + half * 32, v);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.afull[as]);
        mbar_arrive(&bars.empty[s]);
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

// int8 codes -> fp16 (exact), [M, K] dense -> [M, K] dense.
__global__ void i8_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t nvec) {
  griddep_launch_dependents();
  griddep_wait();
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    uint4 lo, hi;
    i8x16_to_f16x16(__ldg(src + i), lo, hi);
    dst[2 * i] = lo;
    dst[2 * i + 1] = hi;
  }
}

template <int BN, int STAGES, int ASTAGES>
cudaError_t launch_i8t_inst(const CUtensorMap& tw, const CUtensorMap& tx, const GemmArgs& args, dim3 grid,
                            cudaStream_t stream) {
  using C = I8tCfg<BN, STAGES, ASTAGES>;
  static bool attr_done[64] = {};
  return launch_persistent(w8a8_gemm_i8t_kernel<BN, STAGES, ASTAGES>, C::NUM_THREADS, C::SMEM_BYTES, tw, tx, args,
                           grid, stream, attr_done);
}

cudaError_t launch_gemm_i8t(int bn, const CUtensorMap& tw, const CUtensorMap& tx16, const GemmArgs& a, dim3 grid,
                            cudaStream_t st) {
  switch (bn) {
    case 16: return launch_i8t_inst<16, 6, 4>(tw, tx16, a, grid, st);
    case 32: return launch_i8t_inst<32, 6, 4>(tw, tx16, a, grid, st);
    case 64: return launch_i8t_inst<64, 5, 4>(tw, tx16, a, grid, st);
    case 128: return launch_i8t_inst<128, 4, 2>(tw, tx16, a, grid, st);
    default: break;
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_i8_to_f16(const void* src, void* dst, size_t n, int num_sms, cudaStream_t st) {
  const size_t nvec = n / 16;
  size_t blocks = (nvec + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms > 0 ? num_sms : 152) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(i8_to_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                    reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), nvec);
}

}  // namespace qurl
