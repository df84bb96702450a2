// gemm_i8w.cu -- the INT8 W8A8 GEMM for prefill on CTA pairs, with both
// operands widened to fp16 in the workspace.
//
// The codes are widened exactly (every integer of magnitude <= 128 is an fp16)
// once per call: the activation codes by the quantizer that writes them (or a
// row kernel), the weight codes by widen_weights_kernel below.  The GEMM is
// then the plain fp16 x fp16 -> fp32 product on the 5th-generation tensor
// cores, laid out like the FP8 pair kernel: the two CTAs of a cluster share
// every MMA (tcgen05.mma.cta_group::2 kind::f16, M = 256 tokens, N = 256
// channels, K = 16), each CTA stages 128 token rows and 128 channel rows of a
// 64-deep k-block (32 KB, six stages), both CTAs' TMA loads complete on rank
// 0's barrier and one multicast commit releases a stage in both CTAs.  Per
// k-block an SM takes in the same bytes for the same MMA time as the FP8 pair
// kernel; the widening costs 3 N K bytes of HBM traffic per call, a few per
// cent of a prefill GEMM's time.
//
// Exactness.  Every product is an integer of magnitude <= 128^2; the fp32
// accumulator holds the exact integer while every partial sum of the k order
// stays within 2^24.  For token t and channel n, over any part of a k range,
// |partial| <= sum |x_tk| |w_nk| <= min(128 S_t, sqrt(Q_t Q_n)) with S_t the
// sum of |x_tk| and Q_t, Q_n the sums of squares over the range (Cauchy-
// Schwarz).  A unit (256 tokens x 256 channels x a K split) whose tokens all
// have S_t <= 2^17, or with max_t Q_t x max_n Q_n <= 2^48, is accumulated in
// one pass ("fast"; the second test is what LLM activations after a norm pass
// -- their sums of |code| exceed 2^17 at K >= 5120).  Any other unit is
// accumulated in 1024-deep chunks (1024 x 128^2 = 2^24), the two accumulator
// buffers alternating between chunks as between units, so the MMA does not
// wait for a chunk to be drained; the epilogue adds the chunks in int32 into
// a running sum kept in a per-CTA scratch region of the workspace.
//
// TMEM: two 256-column fp32 accumulators (512 columns).
#include <algorithm>

#include "gemm.cuh"

namespace qurl {
namespace {

constexpr int kI8wModeWords = 16;                  // accumulation modes of a CTA's first 512 units
constexpr int kI8wModeUnits = 32 * kI8wModeWords;  // (later units: chunks, exact either way)
constexpr int kFastAbsSum = (1 << 24) / 128;       // S_t bound of a one-pass unit
constexpr unsigned long long kFastSqProd = 1ull << 48;  // Q_t x Q_n bound of a one-pass unit

struct I8wCfg {
  static constexpr int BM = 128;             // token rows per CTA (MMA M = 256 per pair)
  static constexpr int BN = 256;             // channels per pair (MMA N)
  static constexpr int BNH = 128;            // channel rows this CTA stages
  static constexpr int BK = 64;              // k per k-block: 128 bytes of fp16 per row
  static constexpr int A_STAGE = BM * 128;   // 16 KB
  static constexpr int B_STAGE = BNH * 128;  // 16 KB
  static constexpr int STAGES = 7;
  static constexpr int PAIR_TX = 2 * (A_STAGE + B_STAGE);  // bytes rank 0's barrier counts per stage
  static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) + 1024;
  static constexpr int NUM_THREADS = 352;    // producer, MMA, mode, 8 epilogue warps
  static constexpr int EPI_WARPS = 8;        // two per TMEM lane quadrant, 128 columns each
  static constexpr int TMEM_COLS = 512;      // two 256-column fp32 accumulators
  static constexpr int CHUNK_KB = 1024 / BK; // k-blocks of one exact chunk
  static constexpr int MMAS_PER_KB = 4;      // K = 16 (32 bytes of fp16) per MMA
  static constexpr int SCRATCH_INTS = BN * BM;  // a CTA's running sums: [256 columns][128 rows]
  static constexpr uint32_t IDESC = umma_idesc_f32acc(0, 0, 2 * BM, BN);  // f16 x f16 -> f32
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

struct I8wBarriers {
  uint64_t full[I8wCfg::STAGES];   // rank 0: both CTAs' TMA bytes of a stage
  uint64_t empty[I8wCfg::STAGES];  // MMA commit (multicast) -> producers: stage read
  uint64_t pfull[2];               // MMA commit (multicast) -> epilogues: accumulator (or chunk) ready
  uint64_t pempty[2];              // rank 0: epilogue warps of both CTAs (16) -> MMA: drained
  uint64_t done;                   // MMA drain on the error path
  uint32_t fast_bits[kI8wModeWords];
  uint32_t mode_count;             // mode warp -> MMA, epilogue: modes of units < mode_count are set
  uint32_t tmem_base;
};

// Unit u: the first whole_units units are tiles 0 .. whole_units - 1 over all
// of K (sp = -1); the remaining tiles are split `splits` ways, split slowest
// (so the pieces of one tile run on different pairs at the same time).  With
// whole_units = 0 every tile is split.
struct UnitCoords {
  int tok, ch, sp;
};
__device__ __forceinline__ UnitCoords i8w_coords(const GemmArgs& a, int u) {
  UnitCoords c;
  int v;
  if (u < a.whole_units) {
    v = u;
    c.sp = -1;
  } else {
    const int tail = a.tiles_tok * a.tiles_ch - a.whole_units;
    const int w = u - a.whole_units;
    c.sp = w / tail;
    v = a.whole_units + (w - c.sp * tail);
  }
  group_tile(a.tiles_tok, a.tiles_ch, kWideTokGroup, v, c.tok, c.ch);
  return c;
}

__device__ __forceinline__ int i8w_units(const GemmArgs& a) {
  return a.whole_units + (a.tiles_tok * a.tiles_ch - a.whole_units) * a.splits;
}

// This CTA's part of unit u: token rows a0 .. a0 + 127, output channels
// b0 .. b0 + 255 of which it stages b0 + 128 rank ...
__device__ __forceinline__ Unit i8w_unit(const GemmArgs& a, int u, uint32_t rank) {
  const UnitCoords c = i8w_coords(a, u);
  Unit w;
  w.a0 = c.tok * 256 + static_cast<int>(rank) * 128;
  w.b0 = c.ch * 256;
  w.kb0 = c.sp < 0 ? 0 : c.sp * a.kb_per_split;
  w.nkb = c.sp < 0 ? a.num_kb : min(a.num_kb - w.kb0, a.kb_per_split);
  w.split = c.sp;
  return w;
}

__global__ void __launch_bounds__(I8wCfg::NUM_THREADS, 1)
    w8a8_gemm_i8w_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                         const GemmArgs args) {
  using C = I8wCfg;
  __shared__ I8wBarriers bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stA = smem;                       // [STAGES][A_STAGE]: fp16 activation codes
  uint8_t* stB = stA + C::STAGES * C::A_STAGE;  // [STAGES][B_STAGE]: fp16 weight codes

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  // the two CTAs of a cluster walk the same units
  const int u_begin = static_cast<int>(blockIdx.x >> 1), u_stride = static_cast<int>(gridDim.x >> 1);
  const int u_end = i8w_units(args);
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.pfull[b], 1);
      mbar_init(&bars.pempty[b], 2 * C::EPI_WARPS);
    }
    mbar_init(&bars.done, 1);
    bars.mode_count = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc<2>(&bars.tmem_base, C::TMEM_COLS);
    tmem_relinquish<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any load or commit reaches them
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  griddep_launch_dependents();
  griddep_wait();

  auto is_fast = [&](int j) {
    return j < kI8wModeUnits && ((bars.fast_bits[j >> 5] >> (j & 31)) & 1u) != 0;
  };
  // accumulation passes over a unit's k-blocks: one, or one per 1024-deep chunk
  auto passes = [&](int j, int nkb) {
    return (args.float_acc || is_fast(j)) ? 1 : (nkb + C::CHUNK_KB - 1) / C::CHUNK_KB;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t polA = l2_policy_evict_last();   // activations: reused by every channel tile
      const uint64_t polB = l2_policy_evict_normal();
      const uint32_t full0 = cluster_map(&bars.full[0], 0);
      int g = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; u += u_stride) {
        const Unit w = i8w_unit(args, u, rank);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          const int s = g % C::STAGES;
          if (args.fault && g == 0) continue;  // injected fault: this stage never fills
          if (!mbar_wait(&bars.empty[s], ((g / C::STAGES) & 1) ^ 1, status)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&bars.full[s], C::PAIR_TX);
          const int kc = (w.kb0 + it) * 128;  // byte column of the fp16 copies
          tma_load_2d_pair(stA + s * C::A_STAGE, &tmX, kc, w.a0, full0 + s * 8, polA);
          tma_load_2d_pair(stB + s * C::B_STAGE, &tmW, kc, w.b0 + static_cast<int>(rank) * C::BNH, full0 + s * 8,
                           polB);
        }
      }
      if (!ok && rank == 0) {
        // rank 0's barriers count both CTAs' bytes: once they complete, no copy
        // of either CTA is in flight (rank 1 leaves only after the closing
        // cluster barrier, which rank 0 reaches after this)
        for (int j = max(0, g - C::STAGES); j < g; ++j)
          mbar_wait_drain(&bars.full[j % C::STAGES], (j / C::STAGES) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0 && lane == 0) {
      bool ok = true;
      int g = 0;                   // k-blocks consumed
      int nb[2] = {0, 0};          // fills committed per accumulator buffer
      int nextbuf = 0;
      for (int u = u_begin, j = 0; u < u_end && ok; u += u_stride, ++j) {
        const Unit w = i8w_unit(args, u, rank);
        if (j < kI8wModeUnits && !wait_count(&bars.mode_count, j, status)) {
          ok = false;
          break;
        }
        const int np = passes(j, w.nkb);
        int it = 0;
        for (int p = 0; p < np && ok; ++p) {
          const int b = nextbuf;
          nextbuf ^= 1;
          // the epilogues of both CTAs must have drained this buffer's previous fill
          if (nb[b] > 0 && !mbar_wait_cluster(&bars.pempty[b], (nb[b] - 1) & 1, status)) {
            ok = false;
            break;
          }
          const uint32_t d = tmem + b * C::BN;
          const int kend = (np == 1) ? w.nkb : min(w.nkb, (p + 1) * C::CHUNK_KB);
          for (int kin = 0; it < kend; ++it, ++g, ++kin) {
            const int s = g % C::STAGES;
            if (!mbar_wait(&bars.full[s], (g / C::STAGES) & 1, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_addr(stA + s * C::A_STAGE);
            const uint32_t sb = smem_addr(stB + s * C::B_STAGE);
#pragma unroll
            for (int kk = 0; kk < C::MMAS_PER_KB; ++kk)
              umma_f16<2>(d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), C::IDESC,
                          (kin | kk) != 0);
            umma_commit_pair(&bars.empty[s], 0x3);
          }
          if (!ok) break;
          umma_commit_pair(&bars.pfull[b], 0x3);
          ++nb[b];
        }
      }
      if (!ok) {  // no MMA may still be writing TMEM when it is released
        umma_commit_pair(&bars.done, 0x1);
        mbar_wait_drain(&bars.done, 0, status);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ accumulation mode of each unit (both CTAs)
    // Published unit by unit (mode_count), so the MMA starts on the first unit
    // while the modes of later ones are still being read.
    if (lane < kI8wModeWords) bars.fast_bits[lane] = 0;
    __syncwarp();
    if (args.asum != nullptr) {
      for (int u = u_begin, j = 0; u < u_end && j < kI8wModeUnits; u += u_stride, ++j) {
        const UnitCoords uc = i8w_coords(args, u);
        const int t = uc.tok, ch = uc.ch, sp = uc.sp;
        // a whole-K unit's sums are those of all the split ranges added (exact
        // integers; a capped range makes the total exceed the bounds either way)
        const int s0 = sp < 0 ? 0 : sp, s1 = sp < 0 ? args.splits : sp + 1;
        // eight token rows and eight channels a lane
        unsigned long long smax = 0, qmax = 0;
        unsigned nmax = 0;
        if (s1 - s0 == 1) {
          // one split range (every unit of an unsplit call): all sixteen or
          // twenty-four loads are issued before any is used, so the first
          // unit's mode, which the MMA waits for, costs one load latency
          unsigned long long sa[8], qa[8];
          unsigned nq[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int m = t * 256 + lane + 32 * r;
            const int n = ch * 256 + lane + 32 * r;
            const size_t at = static_cast<size_t>(m) * args.splits + s0;
            sa[r] = m < args.M ? static_cast<unsigned long long>(__ldg(args.asum + at)) : 0ull;
            qa[r] = (args.qsum && m < args.M) ? __ldg(args.qsum + at) : 0ull;
            nq[r] = (args.qn && n < args.N) ? __ldg(args.qn + n) : 0u;
          }
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            smax = max(smax, sa[r]);
            qmax = max(qmax, qa[r]);
            nmax = max(nmax, nq[r]);
          }
        } else {
          // a whole-K unit of a call with a split tail: its row sums add all
          // the split ranges, row by row (batching four ranges of the eight
          // rows measured slower at eighteen ranges: 32B down, M = 1024)
          for (int c = lane; c < 256; c += 32) {
            const int m = t * 256 + c;
            if (m < args.M) {
              unsigned long long sa = 0, qa = 0;
              for (int k = s0; k < s1; ++k) {
                const size_t at = static_cast<size_t>(m) * args.splits + k;
                sa += static_cast<unsigned long long>(__ldg(args.asum + at));
                if (args.qsum) qa += __ldg(args.qsum + at);
              }
              smax = max(smax, sa);
              qmax = max(qmax, qa);
            }
            const int n = ch * 256 + c;
            if (args.qn && n < args.N) nmax = max(nmax, __ldg(args.qn + n));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          smax = max(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, o));
          qmax = max(qmax, __shfl_xor_sync(0xFFFFFFFFu, qmax, o));
        }
        nmax = __reduce_max_sync(0xFFFFFFFFu, nmax);
        // Q_t x Q_n <= 2^48, in exact 128-bit arithmetic
        const unsigned long long lo = qmax * static_cast<unsigned long long>(nmax);
        const unsigned long long hi = __umul64hi(qmax, static_cast<unsigned long long>(nmax));
        const bool fast = smax <= static_cast<unsigned long long>(kFastAbsSum) ||
                          (args.qsum && args.qn && hi == 0 && lo <= kFastSqProd);
        if (lane == 0) {
          if (fast) bars.fast_bits[j >> 5] |= 1u << (j & 31);
          st_release_cta(&bars.mode_count, static_cast<uint32_t>(j + 1));
        }
        __syncwarp();
      }
    }
    if (lane == 0) st_release_cta(&bars.mode_count, 0xFFFFFFFFu);  // all published (the rest: chunks)
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs, warps 3-10)
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int i = q * 32 + lane;          // token row of this CTA's tile = TMEM lane
    const int cbeg = ((warp - 3) >> 2) * (C::BN / 2);  // this warp's 128 of the 256 columns
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t pempty0 = cluster_map(&bars.pempty[0], 0);
    int* scr = args.scratch + static_cast<size_t>(blockIdx.x) * C::SCRATCH_INTS + i;  // [column][row]
    int nb[2] = {0, 0};
    int nextbuf = 0;
    bool ok = true;
    for (int u = u_begin, j = 0; u < u_end && ok; u += u_stride, ++j) {
      const Unit w = i8w_unit(args, u, rank);
      if (j < kI8wModeUnits && !__all_sync(0xFFFFFFFFu, wait_count(&bars.mode_count, j, status))) {
        ok = false;
        break;
      }
      // a whole-K unit of a call with a split tail writes its result itself:
      // scaled to Y, or as raw sums straight into the accumulator output
      const bool whole = (w.split < 0);
      const int emode = whole ? (args.Y ? kModeBf16 : kModeAcc) : args.mode;
      const int esplit = whole ? 0 : w.split;
      void* ebase = (whole && !args.Y) ? args.acc_out : nullptr;
      const int np = passes(j, w.nkb);
      // the dequantizing epilogue's scales, loaded while the accumulator fills:
      // this lane's token row and its channel in each of the warp's 32-column
      // groups
      float sxm = 0.0f, swr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (emode == kModeBf16) {
        const int m = w.a0 + i;
        sxm = m < args.M ? __ldg(args.sx + m) : 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int n = w.b0 + cbeg + 32 * k + lane;
          swr[k] = n < args.N ? __ldg(args.sw + n) : 0.0f;
        }
      }
      for (int p = 0; p < np; ++p) {
        const int b = nextbuf;
        nextbuf ^= 1;
        if (!warp_wait(&bars.pfull[b], nb[b] & 1, status)) {
          ok = false;
          break;
        }
        ++nb[b];
        tc_fence_after();
        const bool last = (p == np - 1);
#pragma unroll 1
        for (int c0 = cbeg; c0 < cbeg + C::BN / 2; c0 += 32) {
          int* sc = scr + static_cast<size_t>(c0) * C::BM;
          // the running sum of a chunked unit is loaded before the accumulator, so
          // both reads are in flight together
          int prev[32];
          if (np > 1 && p > 0) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) prev[jj] = __ldcg(sc + jj * C::BM);
          }
          uint32_t r[32];
          tmem_ld32(lane_base + b * C::BN + c0, r);
          if (np == 1 && (emode == kModeBf16 || args.float_acc)) {
            // one pass: the fp32 accumulator holds the exact integer (or, for fp16 operands that
            // are not integers, the fp32 sum itself); scale it, or write it as an fp32 partial
            float f[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) f[jj] = __uint_as_float(r[jj]);
            if (emode == kModeBf16) {
              const int k = (c0 - cbeg) >> 5;
              const float swk = k == 0 ? swr[0] : (k == 1 ? swr[1] : (k == 2 ? swr[2] : swr[3]));
              emit32_prescaled<float>(args, w.a0 + i, w.b0 + c0, f, sxm, swk);
            } else {
              emit32<C::BN, float>(args, emode, w.a0, w.b0, esplit, i, c0, f, ebase);
            }
            continue;
          }
          int v[32];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) v[jj] = __float2int_rn(__uint_as_float(r[jj]));
          if (np > 1) {
            if (p > 0) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) v[jj] += prev[jj];
            }
            if (!last) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) __stcg(sc + jj * C::BM, v[jj]);
              continue;
            }
          }
          if (emode == kModeBf16) {
            const int k = (c0 - cbeg) >> 5;
            const float swk = k == 0 ? swr[0] : (k == 1 ? swr[1] : (k == 2 ? swr[2] : swr[3]));
            emit32_prescaled<int>(args, w.a0 + i, w.b0 + c0, v, sxm, swk);
          } else {
            emit32<C::BN, int>(args, emode, w.a0, w.b0, esplit, i, c0, v, ebase);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(pempty0 + b * 8);  // rank 0's MMA writes both CTAs' TMEM
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

// One warp per weight row: int8 codes [N, K] -> fp16 [N, K] (exact), and the
// row's sum of code^2 (saturated at 2^32 - 1) for the GEMM's accumulation mode.
__global__ void __launch_bounds__(256) widen_weights_kernel(const uint8_t* __restrict__ Wq, int N, int K,
                                                            uint8_t* __restrict__ w16, unsigned* __restrict__ qn) {
  griddep_wait();
  griddep_launch_dependents();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= N) return;
  const uint4* s = reinterpret_cast<const uint4*>(Wq + static_cast<size_t>(row) * K);
  uint4* d = reinterpret_cast<uint4*>(w16 + static_cast<size_t>(row) * K * 2);
  const int nvec = K >> 4;
  unsigned long long q = 0;
  for (int v = lane; v < nvec; v += 32) {
    const uint4 raw = __ldg(s + v);
    uint4 lo, hi;
    i8x16_to_f16x16(raw, lo, hi);
    d[2 * v] = lo;
    d[2 * v + 1] = hi;
    int t = 0;
    t = __dp4a(static_cast<int>(raw.x), static_cast<int>(raw.x), t);
    t = __dp4a(static_cast<int>(raw.y), static_cast<int>(raw.y), t);
    t = __dp4a(static_cast<int>(raw.z), static_cast<int>(raw.z), t);
    t = __dp4a(static_cast<int>(raw.w), static_cast<int>(raw.w), t);
    q += static_cast<unsigned long long>(t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xFFFFFFFFu, q, o);
  if (lane == 0) qn[row] = static_cast<unsigned>(q < 0xFFFFFFFFull ? q : 0xFFFFFFFFull);
}

// The split tail of a hybrid plan: one CTA per 4 rows of a tail tile, 64
// threads a row, 4 adjacent columns a thread (one 16-byte load per split when
// N is a multiple of 4).  Each output is the sum of its `splits` partials in
// split order (int32: exact in any order; fp32: a fixed order), then the
// epilogue y = bf16((fp32(sum) * sx[m]) * sw[n]), or the raw sum into acc_out.
__device__ __forceinline__ void add_bits(int& s, uint32_t b) { s += static_cast<int>(b); }
__device__ __forceinline__ void add_bits(float& s, uint32_t b) { s += __uint_as_float(b); }

template <typename T>
__global__ void __launch_bounds__(256) tail_reduce_kernel(const T* __restrict__ part, int splits, int M, int N,
                                                          int tiles_tok, int tiles_ch, int whole_units,
                                                          int tok_group, const float* __restrict__ sx,
                                                          const float* __restrict__ sw,
                                                          __nv_bfloat16* __restrict__ Y, long long ldy,
                                                          T* __restrict__ acc_out) {
  griddep_wait();
  griddep_launch_dependents();
  const int v = whole_units + static_cast<int>(blockIdx.x >> 6);  // the tail tile
  int tok, ch;
  group_tile(tiles_tok, tiles_ch, tok_group, v, tok, ch);
  const int m = tok * 256 + static_cast<int>(blockIdx.x & 63) * 4 + static_cast<int>(threadIdx.x >> 6);
  const int n = ch * 256 + static_cast<int>(threadIdx.x & 63) * 4;
  if (m >= M || n >= N) return;
  const int nc = min(4, N - n);
  const size_t plane = static_cast<size_t>(M) * N;
  const size_t at = static_cast<size_t>(m) * N + n;
  T sum[4] = {T(0), T(0), T(0), T(0)};
  if (nc == 4 && (N & 3) == 0) {
#pragma unroll 4
    for (int z = 0; z < splits; ++z) {
      const uint4 w = __ldcg(reinterpret_cast<const uint4*>(part + z * plane + at));
      const uint32_t e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) add_bits(sum[c], e[c]);
    }
  } else {
    for (int z = 0; z < splits; ++z)
      for (int c = 0; c < nc; ++c) sum[c] += __ldcg(part + z * plane + at + c);
  }
  if (Y) {
    const float sxm = __ldg(sx + m);
    for (int c = 0; c < nc; ++c)
      Y[static_cast<size_t>(m) * ldy + n + c] =
          __float2bfloat16_rn(__fmul_rn(__fmul_rn(static_cast<float>(sum[c]), sxm), __ldg(sw + n + c)));
  } else {
    for (int c = 0; c < nc; ++c) acc_out[at + c] = sum[c];
  }
}

}  // namespace

int i8w_max_ctas(int num_sms) { return num_sms > 0 ? num_sms : 1; }

cudaError_t launch_widen_weights(const void* Wq, int N, int K, void* w16, unsigned* qn, int num_sms,
                                 cudaStream_t st) {
  (void)num_sms;
  return launch_pdl(widen_weights_kernel, dim3(static_cast<unsigned>((N + 7) / 8)), dim3(256), 0, st,
                    reinterpret_cast<const uint8_t*>(Wq), N, K, reinterpret_cast<uint8_t*>(w16), qn);
}

cudaError_t launch_gemm_i8w(const CUtensorMap& tx16, const CUtensorMap& tw16, const GemmArgs& args_in, dim3 grid,
                            cudaStream_t stream) {
  using C = I8wCfg;
  auto kern = w8a8_gemm_i8w_kernel;
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
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(args.tiles_tok) * args.tiles_ch;
  const long long units = args.whole_units + (tiles - args.whole_units) * args.splits;
  // the scratch holds one region per CTA, sized for one CTA per SM
  const int pairs = static_cast<int>(
      std::max<long long>(1, std::min<long long>(std::min<long long>(units, max_pairs[dev]), sms / 2)));
  return launch_pdl_pair(kern, dim3(static_cast<unsigned>(2 * pairs)), dim3(C::NUM_THREADS), C::SMEM_BYTES, stream,
                         tx16, tw16, args);
}

cudaError_t launch_tail_reduce(bool int_partials, int tok_group, const GemmArgs& a, cudaStream_t st) {
  const long long tail = static_cast<long long>(a.tiles_tok) * a.tiles_ch - a.whole_units;
  if (tail <= 0) return cudaSuccess;
  if (tok_group <= 0) tok_group = a.tiles_tok;
  const dim3 grid(static_cast<unsigned>(tail * 64));
  if (int_partials)
    return launch_pdl(tail_reduce_kernel<int>, grid, dim3(256), 0, st, reinterpret_cast<const int*>(a.part), a.splits,
                      a.M, a.N, a.tiles_tok, a.tiles_ch, a.whole_units, tok_group, a.sx, a.sw, a.Y, a.ldy,
                      reinterpret_cast<int*>(a.acc_out));
  return launch_pdl(tail_reduce_kernel<float>, grid, dim3(256), 0, st, reinterpret_cast<const float*>(a.part),
                    a.splits, a.M, a.N, a.tiles_tok, a.tiles_ch, a.whole_units, tok_group, a.sx, a.sw, a.Y, a.ldy,
                    reinterpret_cast<float*>(a.acc_out));
}

}  // namespace qurl
