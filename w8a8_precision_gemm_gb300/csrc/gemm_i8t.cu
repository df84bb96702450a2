// gemm_i8t.cu -- the INT8 W8A8 GEMM for decode (weights on the MMA M side),
// with the weight operand widened into TMEM.
//
// Per 256-deep k stage a CTA
//   * TMA-loads its 128 weight rows of int8 codes (two 128-byte-swizzled
//     boxes, 32 KB) into a ring of their own, and the tokens' codes already
//     widened to fp16 (BN rows x 512 B as four swizzled boxes) into a second
//     ring -- the fp16 copy is made once per call, not once per CTA;
//   * converter warps (one thread per weight row = TMEM lane) read the row's
//     256 codes into registers, widen them to fp16 (exact) and store them into
//     a TMEM stage with tcgen05.st, then free the weight slot: the MMA takes
//     its A operand from TMEM, so the widened weights never travel through
//     shared memory;
//   * one thread issues 16 tcgen05.mma kind::f16 [d], [a_tmem], b_desc (fp32
//     accumulation) once the activation slot and the TMEM stage are full, and
//     frees both with a single commit.  The issuing thread's fixed cost per
//     wait/commit is what bounds a 128-deep pipeline at decode sizes, hence
//     the 256-deep stages.
//
// Exactness.  Every product is an integer of magnitude <= 128^2 and the MMA
// accumulates in fp32, which is exact while every partial sum is an integer of
// magnitude <= 2^24.  For token t and the k range of a K split, |partial| <=
// 128 * S_t with S_t = sum over the range of |x_tk|, which the kernel that
// writes the fp16 codes also writes.  A unit whose tokens all have S_t <=
// 2^24 / 128 is accumulated over its k range in one pass ("fast" unit -- for
// LLM activations S_t is far below the limit).  Otherwise the unit falls back
// to 1024-deep chunks (|partial| <= 1024 * 128^2 = 2^24), each drained by the
// epilogue into an int32 running sum in TMEM.  Both are exact.
//
// TMEM: two fp32 accumulators of BN columns (at least 32), alternated between
// accumulation passes -- a fast unit is one pass, a chunked unit one pass per
// 1024-deep chunk, so the MMA fills one buffer while the epilogue drains the
// other and adds a chunk into the unit's int32 running sum (kept in a scratch
// region of the workspace, one per CTA) -- then NS stages of 128 columns (256
// fp16 per lane) of widened weights.
#include "fused_quant.cuh"
#include "gemm.cuh"

namespace qurl {

// Largest S_t = sum over a k range of |x_tk| for which one fp32 pass is exact.
constexpr int kFastSumMax = (1 << 24) / 128;
// A CTA's scratch for the running sum of a chunked unit: 128 columns x 128 rows.
constexpr int kI8tScratchInts = 128 * 128;
// Saturation of the S_t computed by the activation kernels (> kFastSumMax).
constexpr int kSumCap = 1 << 24;

template <int BN>
struct I8tCfg {
  static constexpr int BM = 128;
  static constexpr int BK = 256;                          // k per stage
  static constexpr int W_BOX = BM * 128;                  // a 128-byte-wide swizzled box of codes
  static constexpr int W_STAGE = 2 * W_BOX;               // 32 KB
  static constexpr int X_BOX = BN * 128;                  // BN rows x 64 fp16
  static constexpr int X_STAGE = 4 * X_BOX;
  static constexpr int NS = BN >= 128 ? 2 : 3;            // TMEM A stages = activation slots
  static constexpr int ACC_COLS = BN < 32 ? 32 : BN;      // an epilogue access spans 32 columns
  static constexpr int A_COLS = BK / 2;                   // 256 fp16 per lane
  static constexpr int A_BASE = 2 * ACC_COLS;
  static constexpr int TMEM_USED = A_BASE + NS * A_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int DYN_LIMIT = 227 * 1024 - 1024;     // leaves room for the static barrier block
  static constexpr int WST_FIT = (DYN_LIMIT - 1024 - NS * X_STAGE) / W_STAGE;
  static constexpr int WST = WST_FIT < 6 ? WST_FIT : 6;   // weight slots
  static constexpr int SMEM_BYTES = WST * W_STAGE + NS * X_STAGE + 1024;
  static constexpr int NUM_THREADS = 512;  // W TMA, MMA, X TMA, mode, 4 epilogue, 8 converter warps
  static constexpr int CHUNK = 1024 / BK;                 // stages per exact chunk
  static constexpr uint32_t IDESC = umma_idesc_f32acc(0, 0, BM, BN);  // f16 x f16 -> f32
  static_assert(TMEM_USED <= 512, "TMEM has 512 columns");
  static_assert(WST >= 3, "weight ring depth");
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

constexpr int kModeWords = 4;  // accumulation modes of a CTA's first 128 units (the rest: chunks)

template <int WST, int NS>
struct I8tBarriers {
  uint64_t wfull[WST];    // TMA -> converters: weight codes landed
  uint64_t wempty[WST];   // converters (128) -> weight producer: codes are in registers
  uint64_t xfull[NS];     // TMA -> MMA: fp16 activation codes landed
  uint64_t afull[NS];     // converters (128) -> MMA: A stage in TMEM
  uint64_t consumed[NS];  // MMA commit -> converters, activation producer: stage read
  uint64_t pfull[2];      // MMA commit -> epilogue: accumulator ready
  uint64_t pempty[2];     // epilogue (128) -> MMA: accumulator drained
  uint64_t done;          // MMA drain on the error path
  uint32_t fast_bits[kModeWords];  // bit j set: the CTA's j-th unit takes one pass over its k range
  uint32_t mode_count;    // mode warp -> MMA, epilogue: bits of units < mode_count are written
  uint32_t tmem_base;
};

// Slot index and phase parity of a ring with N slots.
template <int N>
struct Ring {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++idx == N) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Sum of |c| over 16 int8 codes (|-128| counts 128).
__device__ __forceinline__ int abs_sum16(const uint4 v) {
  unsigned s = 0;
  s = __dp4a(__vabs4(v.x), 0x01010101u, s);
  s = __dp4a(__vabs4(v.y), 0x01010101u, s);
  s = __dp4a(__vabs4(v.z), 0x01010101u, s);
  s = __dp4a(__vabs4(v.w), 0x01010101u, s);
  return static_cast<int>(s);
}

// Sum of c^2 over 16 int8 codes (at most 16 x 128^2).
__device__ __forceinline__ unsigned sq_sum16(const uint4 v) {
  int s = 0;
  s = __dp4a(static_cast<int>(v.x), static_cast<int>(v.x), s);
  s = __dp4a(static_cast<int>(v.y), static_cast<int>(v.y), s);
  s = __dp4a(static_cast<int>(v.z), static_cast<int>(v.z), s);
  s = __dp4a(static_cast<int>(v.w), static_cast<int>(v.w), s);
  return static_cast<unsigned>(s);
}

template <int BN>
__global__ void __launch_bounds__(512, 1)
    w8a8_gemm_i8t_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX16,
                         const GemmArgs args) {
  using C = I8tCfg<BN>;
  constexpr int WST = C::WST;
  constexpr int NS = C::NS;
  __shared__ I8tBarriers<WST, NS> bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stW = smem;                       // [WST][W_STAGE]
  uint8_t* stX = stW + WST * C::W_STAGE;     // [NS][X_STAGE]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const UnitRange R = unit_range(args);
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < WST; ++s) {
      mbar_init(&bars.wfull[s], 1);
      mbar_init(&bars.wempty[s], 128);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars.xfull[s], 1);
      mbar_init(&bars.afull[s], 128);
      mbar_init(&bars.consumed[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.pfull[b], 1);
      mbar_init(&bars.pempty[b], 128);
    }
    bars.mode_count = 0;
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
  const bool fused = args.fq.kind != kFuseNone;
  if (warp != 0 || fused) griddep_wait();

  // j: the unit's position in this CTA's list (call after wait_count(.., j, ..))
  auto is_fast = [&](int j) {
    return j < 32 * kModeWords && ((bars.fast_bits[j >> 5] >> (j & 31)) & 1u) != 0;
  };
  constexpr int kModeUnits = 32 * kModeWords;

  const uint64_t wpol = l2_policy_evict_first();
  auto wload = [&](int slot, const Unit& w, int it) {
    mbar_arrive_expect_tx(&bars.wfull[slot], C::W_STAGE);
    const int k0 = (w.kb0 + it) * C::BK;
    uint8_t* dst = stW + slot * C::W_STAGE;
    tma_load_2d(dst, &tmW, k0, w.a0, &bars.wfull[slot], wpol);
    tma_load_2d(dst + C::W_BOX, &tmW, k0 + 128, w.a0, &bars.wfull[slot], wpol);
  };
  // The first weight slots stream in while the previous kernel (which, per
  // w_prefetch, does not write Wq) is finishing, or, in a fused call, while
  // this kernel quantizes its input rows (after its own grid-dependency wait).
  int npre = 0;  // meaningful in the producer thread
  if (warp == 0 && lane == 0 && (args.w_prefetch || fused) && !args.fault && R.u < R.end) {
    const Unit w = unit_of<true, BN>(args, R.u);
    npre = min(WST, w.nkb);
    for (int it = 0; it < npre; ++it) wload(it, w, it);
  }
  bool run = true;
  if (fused)  // the activation ring is free until the handoff: it holds the rows' reduction scratch
    run = fused_quant_prologue<1>(args.fq, args.fsums, args.M, args.K, kQInt8,
                                  *reinterpret_cast<rq::RowScratch*>(stX), status, args.fault);

  if (!run) {
    // the handoff ran out (the timeout is latched): no role runs; the weight
    // copies already issued land before the CTA leaves
    if (warp == 0 && lane == 0)
      for (int j = 0; j < npre; ++j) mbar_wait_drain(&bars.wfull[j], 0, status);
  } else if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      if (!fused) griddep_wait();
      Ring<WST> r;
      int g = 0;
      bool ok = true;
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<true, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g, r.next()) {
          if (args.fault && g == 0) continue;  // injected fault: this slot never fills
          if (g < npre) continue;
          if (!mbar_wait(&bars.wempty[r.idx], r.phase ^ 1u, status)) {
            ok = false;
            break;
          }
          wload(r.idx, w, it);
        }
      }
      if (!ok) {
        for (int j = max(0, g - WST); j < g; ++j) mbar_wait_drain(&bars.wfull[j % WST], (j / WST) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      Ring<NS> r;
      int nb[2] = {0, 0};  // accumulator fills committed per buffer
      int nextbuf = 0;     // passes (a fast unit, or one chunk of a chunked unit) alternate the buffers
      for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
        const Unit w = unit_of<true, BN>(args, u);
        if (j < kModeUnits && !wait_count(&bars.mode_count, j, status)) {
          ok = false;
          break;
        }
        const bool fast = is_fast(j);
        int b = 0;
        uint32_t d = tmem;
        for (int it = 0; it < w.nkb; ++it, r.next()) {
          const int kin = fast ? it : it % C::CHUNK;  // stage within the accumulation pass
          if (kin == 0) {
            b = nextbuf;
            nextbuf ^= 1;
            if (nb[b] > 0 && !mbar_wait(&bars.pempty[b], (nb[b] - 1) & 1, status)) {
              ok = false;
              break;
            }
            d = tmem + b * C::ACC_COLS;
          }
          if (!mbar_wait(&bars.xfull[r.idx], r.phase, status) || !mbar_wait(&bars.afull[r.idx], r.phase, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_t = tmem + C::A_BASE + r.idx * C::A_COLS;
          const uint32_t xs = smem_addr(stX + r.idx * C::X_STAGE);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint32_t b_addr = xs + (kk >> 2) * C::X_BOX + (kk & 3) * 32;
            umma_f16_tmem_a(d, a_t + kk * 8, umma_desc_sw128(b_addr), C::IDESC, (kin | kk) != 0);
          }
          umma_commit(&bars.consumed[r.idx]);
          const bool pass_end = (it == w.nkb - 1) || (!fast && kin == C::CHUNK - 1);
          if (pass_end) {
            umma_commit(&bars.pfull[b]);
            ++nb[b];
          }
        }
      }
      if (!ok) {
        umma_commit(&bars.done);
        mbar_wait_drain(&bars.done, 0, status);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ activation producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      Ring<NS> r;
      int g = 0;
      bool ok = true;
      for (int u = R.u; u < R.end && ok; u += R.stride) {
        const Unit w = unit_of<true, BN>(args, u);
        for (int it = 0; it < w.nkb; ++it, ++g, r.next()) {
          if (!mbar_wait(&bars.consumed[r.idx], r.phase ^ 1u, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.xfull[r.idx], C::X_STAGE);
          uint8_t* xs = stX + r.idx * C::X_STAGE;
          const int c0 = (w.kb0 + it) * C::BK * 2;  // byte column of the fp16 copy
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_load_2d(xs + j * C::X_BOX, &tmX16, c0 + j * 128, w.b0, &bars.xfull[r.idx], pol);
        }
      }
      if (!ok) {
        for (int j = max(0, g - NS); j < g; ++j) mbar_wait_drain(&bars.xfull[j % NS], (j / NS) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ accumulation mode of each unit
    // Published unit by unit (mode_count), so the MMA starts on the first
    // unit while the modes of later ones are still being read.
    if (lane < kModeWords) bars.fast_bits[lane] = 0;
    __syncwarp();
    if (args.asum != nullptr) {
      for (int u = R.u, j = 0; u < R.end && j < kModeUnits; u += R.stride, ++j) {
        const int t = u % args.tiles_tok;
        const int sp = u / (args.tiles_tok * args.tiles_ch);
        int mx = 0;
#pragma unroll  // the tile's loads all in flight before the first is used
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int m = t * BN + c0 + lane;
          if (c0 + lane < BN && m < args.M)
            mx = max(mx, __ldcg(args.asum + static_cast<size_t>(m) * args.splits + sp));
        }
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        if (lane == 0) {
          if (mx <= kFastSumMax) bars.fast_bits[j >> 5] |= 1u << (j & 31);
          st_release_cta(&bars.mode_count, static_cast<uint32_t>(j + 1));
        }
        __syncwarp();
      }
    }
    if (lane == 0) st_release_cta(&bars.mode_count, 0xFFFFFFFFu);  // all published (the rest: chunks)
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int i = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    // the int32 running sum of a chunked unit: this CTA's scratch region, [column][row]
    int* scr = args.scratch + static_cast<size_t>(blockIdx.x) * kI8tScratchInts + i;
    const int emode = args.mode;
    bool ok = true;
    int nb[2] = {0, 0};
    int nextbuf = 0;
    for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
      const Unit w = unit_of<true, BN>(args, u);
      if (j < kModeUnits && !__all_sync(0xFFFFFFFFu, wait_count(&bars.mode_count, j, status))) {
        ok = false;
        break;
      }
      const bool fast = is_fast(j);
      const int npass = fast ? 1 : (w.nkb + C::CHUNK - 1) / C::CHUNK;
      // scales of this lane's channel and of its token in the first 32-token
      // block, loaded while the accumulator is being filled
      const float sw_lane = channel_scale(args, emode, w.a0 + i);
      const float sx_first = token_scale(args, emode, w.b0 + lane);
      for (int c = 0; c < npass; ++c) {
        const int b = nextbuf;
        nextbuf ^= 1;
        if (!warp_wait(&bars.pfull[b], nb[b] & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool last = (c == npass - 1);
        float sx_lane = sx_first;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          // the next block's token scale, in flight while this block is written
          const float sx_next = (last && c0 + 32 < BN) ? token_scale(args, emode, w.b0 + c0 + 32 + lane) : 0.0f;
          int* sc = scr + static_cast<size_t>(c0) * 128;
          // the running sum is loaded before the accumulator, so both reads are in flight together
          int prev[32];
          if (c > 0) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) prev[jj] = __ldcg(sc + jj * 128);
          }
          uint32_t p[32];
          tmem_ld32(lane_base + b * C::ACC_COLS + c0, p);
          if (npass == 1 && emode == kModeBf16) {
            // a single pass: the fp32 accumulator already holds the exact
            // integer, so it is scaled as it is (no int32 round trip, whose
            // two conversions per element bound this epilogue)
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(p[j]);
            emit32_swap<BN, float>(args, emode, w.a0, w.b0, w.split, i, c0, f, sx_lane, sw_lane);
            sx_lane = sx_next;
            continue;
          }
          int v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float2int_rn(__uint_as_float(p[j]));
          if (c > 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += prev[j];
          }
          if (!last) {
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(sc + j * 128, v[j]);
          } else {
            emit32_swap<BN, int>(args, emode, w.a0, w.b0, w.split, i, c0, v, sx_lane, sw_lane);
          }
          sx_lane = sx_next;
        }
        tc_fence_before();
        mbar_arrive(&bars.pempty[b]);
        ++nb[b];
      }
    }
  } else {
    // ------------------------------------------------------------ converters: weights -> fp16 in TMEM
    // Two groups of four warps (one per TMEM lane quadrant, one weight row per
    // lane) take alternate stages.
    const int q = warp & 3;
    const int grp = (warp - 8) >> 2;
    const int i = q * 32 + lane;  // weight row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int row_off = (i >> 3) * 1024 + (i & 7) * 128;
    Ring<WST> rw;
    Ring<NS> ra;
    int g = 0;
    bool ok = true;
    for (int u = R.u; u < R.end && ok; u += R.stride) {
      const Unit w = unit_of<true, BN>(args, u);
      for (int it = 0; it < w.nkb; ++it, ++g, rw.next(), ra.next()) {
        if ((g & 1) != grp) continue;
        if (!warp_wait(&bars.wfull[rw.idx], rw.phase, status)) {
          ok = false;
          break;
        }
        const uint8_t* wrow = stW + rw.idx * C::W_STAGE + row_off;
        uint4 raw[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)  // 16-byte chunk j = k 16j .. 16j+15, swizzled within its box
          raw[j] = *reinterpret_cast<const uint4*>(wrow + (j >> 3) * C::W_BOX + (((j & 7) ^ (i & 7)) << 4));
        if (!warp_wait(&bars.consumed[ra.idx], ra.phase ^ 1u, status)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the stores below come after the MMAs that read this stage
        const uint32_t a_t = lane_base + C::A_BASE + ra.idx * C::A_COLS;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t v[32];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint4 lo, hi;
            i8x16_to_f16x16(raw[4 * h + jj], lo, hi);
            v[8 * jj + 0] = lo.x; v[8 * jj + 1] = lo.y; v[8 * jj + 2] = lo.z; v[8 * jj + 3] = lo.w;
            v[8 * jj + 4] = hi.x; v[8 * jj + 5] = hi.y; v[8 * jj + 6] = hi.z; v[8 * jj + 7] = hi.w;
          }
          tmem_st32(a_t + h * 32, v);
        }
        // the weight slot is released only once every code read from it has
        // been used (widened into the stores above)
        mbar_arrive(&bars.wempty[rw.idx]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars.afull[ra.idx]);
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

// ---------------------------------------------------------------- CTA pairs, 256 x 256 tiles
//
// Token tiles above 128 run on CTA pairs: the two CTAs of a cluster share
// every MMA (tcgen05.mma.cta_group::2 kind::f16, M = 256 channels -- 128
// widened weight rows in each CTA's TMEM -- by N = 256 tokens), so one
// issued MMA does twice the work of the single-CTA kernel's and one stage of
// 16 MMAs lasts ~1 us: the on-chip refill loop of the widened weights (MMA
// done -> both CTAs widen the next rows -> rank 0 learns of it) has that long
// to close, and the bytes staged per SM buy twice the MMA work.  Each CTA
// stages 128 of the 256 tokens as two 64-row groups (tokens 64 r .. and
// 128 + 64 r .., r = cluster rank); the pair MMA maps CTA r's rows to
// accumulator columns 128 r .., and the epilogue maps the columns back.
//
// TMEM: one 256-column fp32 accumulator (no second buffer: the epilogue of a
// tile and the first MMAs of the next do not overlap) and two 128-column A
// stages.  A unit that needs chunked accumulation runs as two N = 128
// half-passes (one 64-row group of each CTA per half), each in 1024-deep
// chunks drained into an int32 running sum kept in the accumulator's upper
// 128 columns.  Both CTAs' activation loads complete on rank 0's barrier,
// rank 1's converter warps arrive on rank 0's A-stage barrier, and one
// multicast commit releases a stage in both CTAs.
struct I8pCfg {
  static constexpr int BM = 128;                     // weight rows per CTA
  static constexpr int BN = 256;                     // tokens per unit (MMA N of a full pass)
  static constexpr int BK = 256;                     // k per stage
  static constexpr int W_BOX = BM * 128;
  static constexpr int W_STAGE = 2 * W_BOX;          // 32 KB
  static constexpr int XG = 64;                      // token rows of one group
  static constexpr int X_BOX = 2 * XG * 128;         // one 128-byte k column of both groups: 16 KB
  static constexpr int X_STAGE = 4 * X_BOX;          // 64 KB
  static constexpr int NS = 2;                       // activation slots = TMEM A stages
  static constexpr int ACC_COLS = 256;
  static constexpr int A_COLS = BK / 2;
  static constexpr int A_BASE = ACC_COLS;
  static constexpr int TMEM_COLS = 512;
  static constexpr int WST = 3;
  static constexpr int SMEM_BYTES = WST * W_STAGE + NS * X_STAGE + 1024;
  static constexpr int NUM_THREADS = 512;
  static constexpr int CHUNK = 1024 / BK;
  static constexpr uint32_t IDESC_FULL = umma_idesc_f32acc(0, 0, 2 * BM, BN);
  static constexpr uint32_t IDESC_HALF = umma_idesc_f32acc(0, 0, 2 * BM, BN / 2);
  static constexpr int AFULL_ARRIVALS = 128 + 4;     // rank 0's converters, and rank 1's four warps
  static_assert(A_BASE + NS * A_COLS <= TMEM_COLS, "TMEM has 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024 - 1024, "shared memory per CTA");
};

struct I8pBarriers {
  uint64_t wfull[I8pCfg::WST];
  uint64_t wempty[I8pCfg::WST];
  uint64_t xfull[I8pCfg::NS];     // rank 0: both CTAs' activation bytes of a stage
  uint64_t afull[I8pCfg::NS];     // rank 0: both CTAs' converters
  uint64_t consumed[I8pCfg::NS];  // MMA commit (multicast): stage read
  uint64_t pfull;                 // MMA commit (multicast): accumulator (or chunk) ready
  uint64_t pempty;                // rank 0: epilogue warps of both CTAs (8): accumulator drained
  uint64_t done;
  uint32_t fast_bits[kModeWords];
  uint32_t mode_count;
  uint32_t tmem_base;
};

__device__ __forceinline__ void umma_f16_tmem_a_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Unit u of the pair grid: a0 = this CTA's 128 weight rows, b0 = the first of
// the unit's 256 tokens.
__device__ __forceinline__ Unit unit_i8p(const GemmArgs& a, int u, uint32_t rank) {
  const int tok = u % a.tiles_tok;
  const int rest = u / a.tiles_tok;
  const int ch = rest % a.tiles_ch;
  const int sp = rest / a.tiles_ch;
  Unit w;
  w.a0 = ch * 256 + static_cast<int>(rank) * 128;
  w.b0 = tok * 256;
  w.kb0 = sp * a.kb_per_split;
  w.nkb = min(a.num_kb - w.kb0, a.kb_per_split);
  w.split = sp;
  return w;
}

// First token of accumulator columns c0 .. c0 + 31 (c0 a multiple of 32):
// full pass -- column c comes from CTA c / 128, row c % 128 of its two
// 64-token groups; half pass h -- column c from CTA c / 64, row c % 64 of
// its group h.
__device__ __forceinline__ int i8p_token(int b0, int c0, int h, bool full) {
  if (full) {
    const int r = c0 >> 7, j = c0 & 127;
    return b0 + 64 * r + (j & 63) + ((j >> 6) << 7);
  }
  return b0 + 128 * h + 64 * (c0 >> 6) + (c0 & 63);
}

__global__ void __launch_bounds__(512, 1)
    w8a8_gemm_i8p_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX16,
                         const GemmArgs args) {
  using C = I8pCfg;
  constexpr int WST = C::WST;
  constexpr int NS = C::NS;
  __shared__ I8pBarriers bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stW = smem;                       // [WST][W_STAGE]
  uint8_t* stX = stW + WST * C::W_STAGE;     // [NS][X_STAGE]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const UnitRange R{static_cast<int>(blockIdx.x >> 1), static_cast<int>(gridDim.x >> 1),
                    args.tiles_tok * args.tiles_ch * args.splits};
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < WST; ++s) {
      mbar_init(&bars.wfull[s], 1);
      mbar_init(&bars.wempty[s], 128);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars.xfull[s], 1);
      mbar_init(&bars.afull[s], C::AFULL_ARRIVALS);
      mbar_init(&bars.consumed[s], 1);
    }
    mbar_init(&bars.pfull, 1);
    mbar_init(&bars.pempty, 8);
    bars.mode_count = 0;
    mbar_init(&bars.done, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX16);
  }
  if (warp == 1) {
    tmem_alloc<2>(&bars.tmem_base, C::TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any signal reaches them
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  griddep_launch_dependents();
  if (warp != 0) griddep_wait();

  constexpr int kModeUnits = 32 * kModeWords;
  auto is_fast = [&](int j) {
    return j < kModeUnits && ((bars.fast_bits[j >> 5] >> (j & 31)) & 1u) != 0;
  };
  // passes over the unit's k range: one (fast) or two halves (chunked)
  auto passes_of = [&](int j, bool& ok) {
    if (j < kModeUnits && !wait_count(&bars.mode_count, j, status)) ok = false;
    return is_fast(j) ? 1 : 2;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto load = [&](int slot, const Unit& w, int it) {
        mbar_arrive_expect_tx(&bars.wfull[slot], C::W_STAGE);
        const int k0 = (w.kb0 + it) * C::BK;
        uint8_t* dst = stW + slot * C::W_STAGE;
        tma_load_2d(dst, &tmW, k0, w.a0, &bars.wfull[slot], pol);
        tma_load_2d(dst + C::W_BOX, &tmW, k0 + 128, w.a0, &bars.wfull[slot], pol);
      };
      // the first pass's first stages are the same in either mode
      int npre = 0;
      if (args.w_prefetch && !args.fault && R.u < R.end) {
        const Unit w = unit_i8p(args, R.u, rank);
        npre = min(WST, w.nkb);
        for (int it = 0; it < npre; ++it) load(it, w, it);
      }
      griddep_wait();
      Ring<WST> r;
      int g = 0;
      bool ok = true;
      for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
        const Unit w = unit_i8p(args, u, rank);
        const int np = passes_of(j, ok);
        for (int h = 0; h < np && ok; ++h)
          for (int it = 0; it < w.nkb; ++it, ++g, r.next()) {
            if (args.fault && g == 0) continue;  // injected fault: this slot never fills
            if (g < npre) continue;
            if (!mbar_wait(&bars.wempty[r.idx], r.phase ^ 1u, status)) {
              ok = false;
              break;
            }
            load(r.idx, w, it);
          }
      }
      if (!ok) {
        for (int jj = max(0, g - WST); jj < g; ++jj) mbar_wait_drain(&bars.wfull[jj % WST], (jj / WST) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0 && lane == 0) {
      bool ok = true;
      Ring<NS> r;
      int nd = 0;  // accumulator fills committed (epilogue drains to wait for)
      for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
        const Unit w = unit_i8p(args, u, rank);
        const int np = passes_of(j, ok);
        const bool full = (np == 1);
        for (int h = 0; h < np && ok; ++h) {
          for (int it = 0; it < w.nkb; ++it, r.next()) {
            const int kin = full ? it : it % C::CHUNK;  // stage within the accumulation pass
            if (kin == 0 && nd > 0 && !mbar_wait_cluster(&bars.pempty, (nd - 1) & 1, status)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&bars.xfull[r.idx], r.phase, status) ||
                !mbar_wait_cluster(&bars.afull[r.idx], r.phase, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_t = tmem + C::A_BASE + r.idx * C::A_COLS;
            // half pass h: each CTA's 64-row group h
            const uint32_t xs = smem_addr(stX + r.idx * C::X_STAGE) + (full ? 0u : static_cast<uint32_t>(h * C::XG * 128));
            const uint32_t idesc = full ? C::IDESC_FULL : C::IDESC_HALF;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const uint32_t b_addr = xs + (kk >> 2) * C::X_BOX + (kk & 3) * 32;
              umma_f16_tmem_a_pair(tmem, a_t + kk * 8, umma_desc_sw128(b_addr), idesc, (kin | kk) != 0);
            }
            umma_commit_pair(&bars.consumed[r.idx], 0x3);
            if (it == w.nkb - 1 || (!full && kin == C::CHUNK - 1)) {
              umma_commit_pair(&bars.pfull, 0x3);
              ++nd;
            }
          }
        }
      }
      if (!ok) {
        umma_commit_pair(&bars.done, 0x1);
        mbar_wait_drain(&bars.done, 0, status);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ activation producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      const uint32_t xfull0 = cluster_map(&bars.xfull[0], 0);
      Ring<NS> r;
      int g = 0;
      bool ok = true;
      for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
        const Unit w = unit_i8p(args, u, rank);
        const int np = passes_of(j, ok);
        for (int h = 0; h < np && ok; ++h)
          for (int it = 0; it < w.nkb; ++it, ++g, r.next()) {
            if (!mbar_wait(&bars.consumed[r.idx], r.phase ^ 1u, status)) {
              ok = false;
              break;
            }
            if (rank == 0) mbar_arrive_expect_tx(&bars.xfull[r.idx], 2 * C::X_STAGE);
            uint8_t* xs = stX + r.idx * C::X_STAGE;
            const int c0 = (w.kb0 + it) * C::BK * 2;  // byte column of the fp16 copy
#pragma unroll
            for (int kc = 0; kc < 4; ++kc)
#pragma unroll
              for (int grp = 0; grp < 2; ++grp)
                tma_load_2d_pair(xs + kc * C::X_BOX + grp * C::XG * 128, &tmX16, c0 + kc * 128,
                                 w.b0 + grp * 128 + static_cast<int>(rank) * C::XG, xfull0 + r.idx * 8, pol);
          }
      }
      if (!ok && rank == 0) {
        // rank 0's barriers count both CTAs' bytes; rank 1 leaves only after
        // the closing cluster barrier, which rank 0 reaches after this
        for (int jj = max(0, g - NS); jj < g; ++jj) mbar_wait_drain(&bars.xfull[jj % NS], (jj / NS) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ accumulation mode of each unit
    if (lane < kModeWords) bars.fast_bits[lane] = 0;
    __syncwarp();
    if (args.asum != nullptr) {
      for (int u = R.u, j = 0; u < R.end && j < kModeUnits; u += R.stride, ++j) {
        const int t = u % args.tiles_tok;
        const int sp = u / (args.tiles_tok * args.tiles_ch);
        int mx = 0;
#pragma unroll  // the tile's loads all in flight before the first is used
        for (int c0 = 0; c0 < C::BN; c0 += 32) {
          const int m = t * C::BN + c0 + lane;
          if (c0 + lane < C::BN && m < args.M)
            mx = max(mx, __ldg(args.asum + static_cast<size_t>(m) * args.splits + sp));
        }
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        if (lane == 0) {
          if (mx <= kFastSumMax) bars.fast_bits[j >> 5] |= 1u << (j & 31);
          st_release_cta(&bars.mode_count, static_cast<uint32_t>(j + 1));
        }
        __syncwarp();
      }
    }
    if (lane == 0) st_release_cta(&bars.mode_count, 0xFFFFFFFFu);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int i = q * 32 + lane;  // weight row of this CTA's tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tR = lane_base + 128;  // running sum of a chunked half pass
    const uint32_t pempty0 = cluster_map(&bars.pempty, 0);
    const int emode = args.mode;
    bool ok = true;
    int nd = 0;
    auto drained = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(pempty0);  // rank 0's next MMA writes both CTAs' TMEM
      ++nd;
    };
    for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
      const Unit w = unit_i8p(args, u, rank);
      if (j < kModeUnits && !__all_sync(0xFFFFFFFFu, wait_count(&bars.mode_count, j, status))) {
        ok = false;
        break;
      }
      const bool full = is_fast(j);
      const float sw_lane = channel_scale(args, emode, w.a0 + i);
      if (full) {
        float sx_lane = token_scale(args, emode, i8p_token(w.b0, 0, 0, true) + lane);
        if (!warp_wait(&bars.pfull, nd & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < C::BN; c0 += 32) {
          const int tb = i8p_token(w.b0, c0, 0, true);
          const float sx_next =
              c0 + 32 < C::BN ? token_scale(args, emode, i8p_token(w.b0, c0 + 32, 0, true) + lane) : 0.0f;
          uint32_t p[32];
          tmem_ld32(lane_base + c0, p);
          if (emode == kModeBf16) {
            float f[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) f[jj] = __uint_as_float(p[jj]);
            emit32_swap<C::BN, float>(args, emode, w.a0, tb - c0, w.split, i, c0, f, sx_lane, sw_lane);
          } else {
            int v[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] = __float2int_rn(__uint_as_float(p[jj]));
            emit32_swap<C::BN, int>(args, emode, w.a0, tb - c0, w.split, i, c0, v, sx_lane, sw_lane);
          }
          sx_lane = sx_next;
        }
        drained();
      } else {
        const int npass = (w.nkb + C::CHUNK - 1) / C::CHUNK;
        for (int h = 0; h < 2 && ok; ++h) {
          for (int c = 0; c < npass; ++c) {
            if (!warp_wait(&bars.pfull, nd & 1, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool last = (c == npass - 1);
#pragma unroll 1
            for (int c0 = 0; c0 < C::BN / 2; c0 += 32) {
              const int tb = i8p_token(w.b0, c0, h, false);
              const float sx_lane = last ? token_scale(args, emode, tb + lane) : 0.0f;
              uint32_t p[32];
              tmem_ld32(lane_base + c0, p);
              int v[32];
              if (c > 0) {
                uint32_t rs[32];
                tmem_ld32(tR + c0, rs);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) v[jj] = static_cast<int>(rs[jj]) + __float2int_rn(__uint_as_float(p[jj]));
              } else {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) v[jj] = __float2int_rn(__uint_as_float(p[jj]));
              }
              if (!last) {
                uint32_t wv[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) wv[jj] = static_cast<uint32_t>(v[jj]);
                tmem_st32(tR + c0, wv);
              } else {
                emit32_swap<C::BN, int>(args, emode, w.a0, tb - c0, w.split, i, c0, v, sx_lane, sw_lane);
              }
            }
            if (!last) tmem_wait_st();
            drained();
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ converters (both CTAs)
    const int q = warp & 3;
    const int grp = (warp - 8) >> 2;
    const int i = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int row_off = (i >> 3) * 1024 + (i & 7) * 128;
    const uint32_t afull0 = cluster_map(&bars.afull[0], 0);
    Ring<WST> rw;
    Ring<NS> ra;
    int g = 0;
    bool ok = true;
    for (int u = R.u, j = 0; u < R.end && ok; u += R.stride, ++j) {
      const Unit w = unit_i8p(args, u, rank);
      bool mok = true;
      const int np = __all_sync(0xFFFFFFFFu, j >= kModeUnits || wait_count(&bars.mode_count, j, status))
                         ? (is_fast(j) ? 1 : 2)
                         : (mok = false, 2);
      if (!mok) {
        ok = false;
        break;
      }
      for (int h = 0; h < np && ok; ++h)
        for (int it = 0; it < w.nkb; ++it, ++g, rw.next(), ra.next()) {
          if ((g & 1) != grp) continue;
          if (!warp_wait(&bars.wfull[rw.idx], rw.phase, status)) {
            ok = false;
            break;
          }
          const uint8_t* wrow = stW + rw.idx * C::W_STAGE + row_off;
          uint4 raw[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            raw[jj] = *reinterpret_cast<const uint4*>(wrow + (jj >> 3) * C::W_BOX + (((jj & 7) ^ (i & 7)) << 4));
          if (!warp_wait(&bars.consumed[ra.idx], ra.phase ^ 1u, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_t = lane_base + C::A_BASE + ra.idx * C::A_COLS;
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            uint32_t v[32];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              uint4 lo, hi;
              i8x16_to_f16x16(raw[4 * hh + jj], lo, hi);
              v[8 * jj + 0] = lo.x; v[8 * jj + 1] = lo.y; v[8 * jj + 2] = lo.z; v[8 * jj + 3] = lo.w;
              v[8 * jj + 4] = hi.x; v[8 * jj + 5] = hi.y; v[8 * jj + 6] = hi.z; v[8 * jj + 7] = hi.w;
            }
            tmem_st32(a_t + hh * 32, v);
          }
          mbar_arrive(&bars.wempty[rw.idx]);
          tmem_wait_st();
          tc_fence_before();
          if (rank == 0) {
            mbar_arrive(&bars.afull[ra.idx]);
          } else {
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(afull0 + ra.idx * 8);
          }
        }
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA frees its TMEM or exits while rank 0's MMAs, commits or the
  // peer's copies and arrivals may still reach it
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<2>(tmem, C::TMEM_COLS);
  }
}

// One block per row: int8 codes -> fp16 (exact), [M, K] dense -> [M, K]
// dense, and the row's sums of |code| (saturated at kSumCap) and, when wanted,
// of code^2 over the ranges of `sums`, for the GEMM's accumulation mode.
__global__ void __launch_bounds__(256) i8_to_f16_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                        int K, const CodeSums sums) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ unsigned long long cnt[2 * kMaxSums];
  for (int j = threadIdx.x; j < sums.nsum; j += blockDim.x) cnt[j] = cnt[kMaxSums + j] = 0;
  __syncthreads();
  const int m = blockIdx.x;
  const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<size_t>(m) * K);
  uint4* d = reinterpret_cast<uint4*>(dst + static_cast<size_t>(m) * K * 2);
  const int nvec = K >> 4;
  const int lane = threadIdx.x & 31;
  // warp-uniform steps over 32 consecutive vectors; ranges are multiples of
  // 16 vectors, so a step's vectors lie in at most two (r0, r0 + 1)
  for (int v0 = threadIdx.x & ~31; v0 < nvec; v0 += blockDim.x) {
    const int v = v0 + lane;
    unsigned a = 0, q = 0;
    if (v < nvec) {
      const uint4 raw = __ldg(s + v);
      uint4 lo, hi;
      i8x16_to_f16x16(raw, lo, hi);
      d[2 * v] = lo;
      d[2 * v + 1] = hi;
      a = static_cast<unsigned>(abs_sum16(raw));
      q = sq_sum16(raw);
    }
    const int r0 = (v0 * 16) / sums.sum_len;
    const bool first = (v < nvec ? (v * 16) / sums.sum_len : r0) == r0;
    const unsigned s0 = __reduce_add_sync(0xFFFFFFFFu, first ? a : 0u);
    const unsigned s1 = __reduce_add_sync(0xFFFFFFFFu, first ? 0u : a);
    const unsigned q0 = __reduce_add_sync(0xFFFFFFFFu, first ? q : 0u);
    const unsigned q1 = __reduce_add_sync(0xFFFFFFFFu, first ? 0u : q);
    if (lane == 0) {
      if (s0 != 0) atomicAdd(&cnt[r0], static_cast<unsigned long long>(s0));
      if (s1 != 0) atomicAdd(&cnt[r0 + 1], static_cast<unsigned long long>(s1));
      if (q0 != 0) atomicAdd(&cnt[kMaxSums + r0], static_cast<unsigned long long>(q0));
      if (q1 != 0) atomicAdd(&cnt[kMaxSums + r0 + 1], static_cast<unsigned long long>(q1));
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < sums.nsum; j += blockDim.x) {
    sums.asum[static_cast<size_t>(m) * sums.nsum + j] =
        static_cast<int>(cnt[j] < static_cast<unsigned long long>(kSumCap) ? cnt[j] : kSumCap);
    if (sums.qsum)
      sums.qsum[static_cast<size_t>(m) * sums.nsum + j] =
          static_cast<unsigned>(cnt[kMaxSums + j] < 0xFFFFFFFFull ? cnt[kMaxSums + j] : 0xFFFFFFFFull);
  }
}

template <int BN>
cudaError_t launch_i8t_inst(const CUtensorMap& tw, const CUtensorMap& tx, const GemmArgs& args, dim3 grid,
                            cudaStream_t stream) {
  using C = I8tCfg<BN>;
  static bool attr_done[64] = {};
  return launch_persistent(w8a8_gemm_i8t_kernel<BN>, C::NUM_THREADS, C::SMEM_BYTES, tw, tx, args, grid, stream,
                           attr_done);
}

cudaError_t launch_gemm_i8t(int bn, const CUtensorMap& tw, const CUtensorMap& tx16, const GemmArgs& a, dim3 grid,
                            cudaStream_t st) {
  switch (bn) {
    case 16: return launch_i8t_inst<16>(tw, tx16, a, grid, st);
    case 32: return launch_i8t_inst<32>(tw, tx16, a, grid, st);
    case 64: return launch_i8t_inst<64>(tw, tx16, a, grid, st);
    case 128: return launch_i8t_inst<128>(tw, tx16, a, grid, st);
    default: break;
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_i8p(const CUtensorMap& tw, const CUtensorMap& tx16, const GemmArgs& args_in, dim3 grid,
                            cudaStream_t stream) {
  using C = I8pCfg;
  auto kern = w8a8_gemm_i8p_kernel;
  static bool attr_done[64] = {};
  static int max_pairs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (max_pairs[dev] <= 0) {
    // one cluster of two CTAs per pair of SMs, as many as can be resident
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(C::NUM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorLaunchOutOfResources;
    max_pairs[dev] = n;
  }
  GemmArgs args = args_in;
  args.tiles_tok = grid.x;
  args.tiles_ch = grid.y;
  args.splits = grid.z;
  const long long units = static_cast<long long>(args.tiles_tok) * args.tiles_ch * args.splits;
  const int pairs = static_cast<int>(std::max<long long>(1, std::min<long long>(units, max_pairs[dev])));
  return launch_pdl_pair(kern, dim3(static_cast<unsigned>(2 * pairs)), dim3(C::NUM_THREADS), C::SMEM_BYTES, stream,
                         tw, tx16, args);
}

cudaError_t launch_i8_to_f16(const void* src, void* dst, int M, int K, CodeSums sums, cudaStream_t st) {
  return launch_pdl(i8_to_f16_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0, st,
                    reinterpret_cast<const uint8_t*>(src), reinterpret_cast<uint8_t*>(dst), K, sums);
}

}  // namespace qurl
