// gemm_fp8p.cu -- the FP8-E4M3 W8A8 GEMM on CTA pairs.
//
// The two CTAs of a cluster share every MMA (tcgen05.mma.cta_group::2
// kind::f8f6f4, M = 256, N = BN, K = 32): each CTA stages 128 rows of the A
// operand and BN / 2 rows of the B operand of a k-block, the pair's MMA reads
// both CTAs' tiles, and each CTA's TMEM receives its 128 A rows x BN columns
// of the accumulator.  Prefill: A = 128 token rows, B = 256 channels (per
// k-block an SM takes in 32 KB for 128 x 256 x 128 multiply-adds instead of
// 48 KB).  Decode (SWAP): A = 128 weight rows, B = the BN tokens (the weight
// stream per SM is unchanged, the token bytes halve, and more weight stages
// fit in shared memory).  The operand bytes a CTA keeps in flight over the
// load latency are what bounds the single-CTA kernels.
//
// Synchronisation without thread-level traffic between the CTAs on the
// k-block path: both CTAs' TMA loads complete on rank 0's "full" barrier
// (the pair form of the load, which counts the bytes on the peer CTA's
// mbarrier), rank 0's producer alone arms it with both CTAs' bytes, and
// rank 0's MMA thread releases each stage in both CTAs with one multicast
// commit.  Only the epilogue's "accumulator drained" signal crosses CTAs by
// thread arrivals (once per tile).
#include "fused_quant.cuh"
#include "gemm.cuh"

namespace qurl {

template <int BN_, int STAGES>
struct Fp8PairCfg {
  static constexpr int BM = 128;             // A rows per CTA (MMA M = 256 per pair)
  static constexpr int BN = BN_;             // MMA N (B rows of the pair)
  static constexpr int BNH = BN / 2;         // B rows this CTA stages
  static constexpr int BK = 128;             // k (bytes of e4m3 codes) per k-block
  static constexpr int A_STAGE = BM * BK;    // 16 KB
  static constexpr int B_STAGE = BNH * BK;
  static constexpr int PAIR_TX = 2 * (A_STAGE + B_STAGE);  // bytes rank 0's barrier counts per stage
  static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) + 1024;
  static constexpr int NUM_THREADS = 192;    // producer, MMA, 4 epilogue warps
  static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : 2 * BN;  // two BN-column fp32 accumulators
  static constexpr int MMA_K_BYTES = 32;
  static constexpr int MMAS_PER_KB = BK / MMA_K_BYTES;
  static constexpr uint32_t IDESC = umma_idesc_f32acc(0, 0, 2 * BM, BN);  // e4m3 x e4m3 -> f32
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "pair MMA N");
  static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation: a power of two");
};

template <int STAGES>
struct Fp8PairBarriers {
  uint64_t full[STAGES];   // rank 0: both CTAs' TMA bytes of a stage (rank 1's copy unused)
  uint64_t empty[STAGES];  // MMA commit (multicast) -> producer: stage read
  uint64_t pfull[2];       // MMA commit (multicast) -> epilogue: accumulator ready
  uint64_t pempty[2];      // rank 0: epilogue warps of both CTAs (8) -> MMA: accumulator drained
  uint64_t done;           // MMA drain on the error path
  uint32_t tmem_base;
};

// This CTA's part of unit u: A rows a0 .. a0 + 127 (rank r takes the r-th
// half of the pair's 256), B columns b0 .. b0 + BN - 1 of the output, of which
// it stages rows b0 + r BN / 2 ...  Prefill: A = tokens, B = channels;
// SWAP: A = channels, B = tokens.  Tiles are numbered token tile fastest
// (prefill: within groups of tok_group token tiles, group_tile); the first
// whole_units units (prefill only) are tiles 0 .. whole_units - 1 over all of
// K (split -1), the remaining tiles are split `splits` ways, split slowest
// (with whole_units = 0 every tile is split).
struct PairUnit {
  int a0, b0, kb0, nkb, split;
};

template <bool SWAP, int BN>
__device__ __forceinline__ PairUnit pair_unit(const GemmArgs& a, int u, uint32_t rank) {
  int v, sp;
  if (u < a.whole_units) {
    v = u;
    sp = -1;
  } else {
    const int tail = a.tiles_tok * a.tiles_ch - a.whole_units;
    const int w = u - a.whole_units;
    sp = w / tail;
    v = a.whole_units + (w - sp * tail);
  }
  int tok, ch;
  if (SWAP) {
    tok = v % a.tiles_tok;
    ch = v / a.tiles_tok;
  } else {
    group_tile(a.tiles_tok, a.tiles_ch, a.tok_group > 0 ? a.tok_group : a.tiles_tok, v, tok, ch);
  }
  PairUnit w;
  w.a0 = (SWAP ? ch : tok) * 256 + static_cast<int>(rank) * 128;
  w.b0 = (SWAP ? tok : ch) * BN;
  w.kb0 = sp < 0 ? 0 : sp * a.kb_per_split;
  w.nkb = sp < 0 ? a.num_kb : min(a.num_kb - w.kb0, a.kb_per_split);
  w.split = sp;
  return w;
}

template <bool SWAP, int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
    w8a8_gemm_fp8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                              const GemmArgs args) {
  using C = Fp8PairCfg<BN, STAGES>;
  __shared__ Fp8PairBarriers<STAGES> bars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stA = smem;                       // [STAGES][A_STAGE]
  uint8_t* stB = stA + STAGES * C::A_STAGE;  // [STAGES][B_STAGE]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  // the two CTAs of a cluster walk the same units
  const int u_begin = static_cast<int>(blockIdx.x >> 1), u_stride = static_cast<int>(gridDim.x >> 1);
  const int tiles = args.tiles_tok * args.tiles_ch;
  const int u_end = args.whole_units + (tiles - args.whole_units) * args.splits;  // as the launch counts them
  int* status = args.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.pfull[b], 1);
      mbar_init(&bars.pempty[b], 8);
    }
    mbar_init(&bars.done, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
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

  // the operand read once (weights, decode) streams through L2 first
  const uint64_t polA = SWAP ? l2_policy_evict_first() : l2_policy_evict_last();
  const uint64_t polB = SWAP ? l2_policy_evict_last() : l2_policy_evict_normal();
  const uint32_t full0 = cluster_map(&bars.full[0], 0);
  // A fused call (decode) quantizes its input rows first; meanwhile the weight
  // halves of the first stages stream in (their barriers on rank 0 are armed
  // with both CTAs' full stage bytes, the token halves follow the handoff).
  const bool fused = SWAP && args.fq.kind != kFuseNone;
  int npre = 0;  // meaningful in the producer thread
  if (fused && warp == 0 && lane == 0 && !args.fault && u_begin < u_end) {
    const PairUnit w = pair_unit<SWAP, BN>(args, u_begin, rank);
    npre = min(STAGES, w.nkb);
    for (int it = 0; it < npre; ++it) {
      if (rank == 0) mbar_arrive_expect_tx(&bars.full[it], C::PAIR_TX);
      tma_load_2d_pair(stA + it * C::A_STAGE, &tmA, (w.kb0 + it) * C::BK, w.a0, full0 + it * 8, polA);
    }
  }
  bool run = true;
  if constexpr (SWAP) {
    if (fused)  // the token stages are free until the handoff: they hold the rows' reduction scratch
      run = fused_quant_prologue<4>(args.fq, args.fsums, args.M, args.K, kQFp8,
                                    *reinterpret_cast<rq::RowScratch*>(stB), status, args.fault);
  }

  if (!run) {
    // the handoff ran out (the timeout is latched): no role runs.  Rank 0's
    // barriers of the stages issued count both CTAs' weight halves (and the
    // token halves never issued: bounded waits), so once they are done no copy
    // of either CTA is in flight; rank 1 leaves after the closing cluster
    // barrier, which rank 0 reaches after this.
    if (warp == 0 && lane == 0 && rank == 0)
      for (int j = 0; j < npre; ++j) mbar_wait_drain(&bars.full[j], 0, status);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; u += u_stride) {
        const PairUnit w = pair_unit<SWAP, BN>(args, u, rank);
        for (int it = 0; it < w.nkb; ++it, ++g) {
          const int s = g % STAGES;
          if (args.fault && g == 0) continue;  // injected fault: this stage never fills
          if (g < npre) {  // the weight half is in flight; add the token half
            tma_load_2d_pair(stB + s * C::B_STAGE, &tmB, (w.kb0 + it) * C::BK, w.b0 + static_cast<int>(rank) * C::BNH,
                             full0 + s * 8, polB);
            continue;
          }
          if (!mbar_wait(&bars.empty[s], ((g / STAGES) & 1) ^ 1, status)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&bars.full[s], C::PAIR_TX);
          const int kc = (w.kb0 + it) * C::BK;
          tma_load_2d_pair(stA + s * C::A_STAGE, &tmA, kc, w.a0, full0 + s * 8, polA);
          tma_load_2d_pair(stB + s * C::B_STAGE, &tmB, kc, w.b0 + static_cast<int>(rank) * C::BNH, full0 + s * 8,
                           polB);
        }
      }
      if (!ok && rank == 0) {
        // rank 0's barriers count both CTAs' bytes: once they complete, no
        // copy of either CTA is in flight (rank 1 leaves only after the
        // cluster barrier below, which rank 0 reaches after this)
        for (int j = max(0, g - STAGES); j < g; ++j) mbar_wait_drain(&bars.full[j % STAGES], (j / STAGES) & 1, status);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0 && lane == 0) {
      bool ok = true;
      int g = 0;   // k-blocks consumed
      int cg = 0;  // accumulators filled (buffer cg & 1)
      for (int u = u_begin; u < u_end && ok; u += u_stride) {
        const PairUnit w = pair_unit<SWAP, BN>(args, u, rank);
        const int buf = cg & 1;
        // the epilogues of both CTAs must have drained this buffer's previous tile
        if (cg >= 2 && !mbar_wait_cluster(&bars.pempty[buf], ((cg >> 1) - 1) & 1, status)) {
          ok = false;
          break;
        }
        const uint32_t d = tmem + buf * C::BN;
        for (int it = 0; it < w.nkb; ++it, ++g) {
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
            umma_f8f6f4<2>(d, umma_desc_sw128(sa + kk * C::MMA_K_BYTES), umma_desc_sw128(sb + kk * C::MMA_K_BYTES),
                           C::IDESC, (it | kk) != 0);
          umma_commit_pair(&bars.empty[s], 0x3);
        }
        if (!ok) break;
        umma_commit_pair(&bars.pfull[buf], 0x3);
        ++cg;
      }
      if (!ok) {  // no MMA may still be writing TMEM when it is released
        umma_commit_pair(&bars.done, 0x1);
        mbar_wait_drain(&bars.done, 0, status);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int i = q * 32 + lane;          // token row of this CTA's tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t pempty0 = cluster_map(&bars.pempty[0], 0);
    const int emode = args.mode;
    int cg = 0;
    for (int u = u_begin; u < u_end; u += u_stride, ++cg) {
      const PairUnit w = pair_unit<SWAP, BN>(args, u, rank);
      const int buf = cg & 1;
      // swap: scales of this lane's channel and of its token in the first
      // 32-token block, loaded while the accumulator is being filled
      const float sw_lane = SWAP ? channel_scale(args, emode, w.a0 + i) : 0.0f;
      const float sx_first = SWAP ? token_scale(args, emode, w.b0 + lane) : 0.0f;
      // prefill: the unit's mode, and for the dequantizing epilogue this lane's
      // token scale and its channel's scale in the first 32-column group,
      // loaded while the accumulator fills
      const bool whole = !SWAP && w.split < 0;
      const int umode = whole ? (args.Y ? kModeBf16 : kModeAcc) : emode;
      const float sxm = (!SWAP && umode == kModeBf16 && w.a0 + i < args.M) ? __ldg(args.sx + w.a0 + i) : 0.0f;
      float swc = (!SWAP && umode == kModeBf16) ? channel_scale(args, kModeBf16, w.b0 + lane) : 0.0f;
      if (!warp_wait(&bars.pfull[buf], (cg >> 1) & 1, status)) break;
      tc_fence_after();
      float sx_lane = sx_first;
#pragma unroll 1
      for (int c0 = 0; c0 < C::BN; c0 += 32) {
        const float sx_next = (SWAP && c0 + 32 < C::BN) ? token_scale(args, emode, w.b0 + c0 + 32 + lane) : 0.0f;
        const float sw_next =
            (!SWAP && umode == kModeBf16 && c0 + 32 < C::BN) ? channel_scale(args, kModeBf16, w.b0 + c0 + 32 + lane)
                                                              : 0.0f;
        uint32_t p[32];
        tmem_ld32(lane_base + buf * C::BN + c0, p);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(p[j]);
        if constexpr (SWAP) {
          emit32_swap<BN, float>(args, emode, w.a0, w.b0, w.split, i, c0, v, sx_lane, sw_lane);
        } else if (umode == kModeBf16) {
          emit32_prescaled<float>(args, w.a0 + i, w.b0 + c0, v, sxm, swc);
        } else {
          // a whole-K unit of a call with a split tail writes its raw sums
          // straight into the accumulator output
          emit32<BN, float>(args, umode, w.a0, w.b0, whole ? 0 : w.split, i, c0, v,
                            (whole && !args.Y) ? args.acc_out : nullptr);
        }
        sx_lane = sx_next;
        swc = sw_next;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(pempty0 + buf * 8);  // rank 0's MMA writes both CTAs' TMEM
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

template <bool SWAP, int BN, int STAGES>
cudaError_t launch_pair_inst(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args_in, dim3 grid,
                             cudaStream_t stream) {
  using C = Fp8PairCfg<BN, STAGES>;
  auto kern = w8a8_gemm_fp8_pair_kernel<SWAP, BN, STAGES>;
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
  const long long tiles = static_cast<long long>(args.tiles_tok) * args.tiles_ch;
  const long long units = args.whole_units + (tiles - args.whole_units) * args.splits;
  const int pairs = static_cast<int>(std::max<long long>(1, std::min<long long>(units, max_pairs[dev])));
  return launch_pdl_pair(kern, dim3(static_cast<unsigned>(2 * pairs)), dim3(C::NUM_THREADS), C::SMEM_BYTES, stream,
                         ta, tb, args);
}

// Stage counts fill ~192-200 KB of shared memory: (128 + BN / 2) x 128 B per stage.
cudaError_t launch_gemm_fp8_pair(bool swap, int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                                 dim3 grid, cudaStream_t st) {
  if (!swap) return bn == 256 ? launch_pair_inst<false, 256, 6>(ta, tb, a, grid, st) : cudaErrorInvalidValue;
  switch (bn) {
    case 64: return launch_pair_inst<true, 64, 9>(ta, tb, a, grid, st);
    case 128: return launch_pair_inst<true, 128, 8>(ta, tb, a, grid, st);
    case 256: return launch_pair_inst<true, 256, 6>(ta, tb, a, grid, st);
    default: break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace qurl
