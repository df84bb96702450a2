// fused_quant.cuh -- the quantizer of a fused entry point (RMSNorm -> quant,
// quant with the UAQ pre-scale, SiLU * up -> quant) run inside the decode GEMM
// kernel that consumes its codes, so a fused decode call is one kernel (plus
// the split-K reduction where K is split) instead of a quantizer kernel and a
// GEMM kernel.
//
// Every CTA of the persistent grid quantizes the rows blockIdx.x,
// blockIdx.x + gridDim.x, ... (a decode batch of M <= 256 tokens spreads over
// the SMs one or two rows each), with the same row arithmetic as the
// standalone quantizers (rowquant.cuh), then the CTAs hand over: each
// publishes its rows (a release fence for the generic proxy and one for the
// async proxy, whose TMA loads read the codes next) and waits until all
// gridDim.x CTAs have, through a counter in the caller's workspace.  The
// persistent grids have at most one CTA per SM, so every CTA becomes resident
// once whatever ran before it on the SMs has drained; the wait is bounded all
// the same (the kernel latches QURL_ERR_TIMEOUT and skips its main loop, and
// the counters are left as they were: the caller zeroes them again).  The
// last CTA to leave resets the counters, so every call leaves them zero.
#pragma once

#include "ptx.cuh"
#include "rowquant.cuh"

namespace qurl {

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Quantize this CTA's rows of the fused activation, then wait (bounded) until
// every CTA of the grid has.  Every thread of the block calls it; sh is
// shared-memory scratch no copy lands in before the call returns.  Returns
// false when the wait ran out.
// fault (test hook): CTA 0 does not arrive, so every CTA's wait runs out.
template <int NC>
__device__ __forceinline__ bool fused_quant_prologue(const FusedQuant& fq, const CodeSums& sums, int M, int K,
                                                     int qt, rq::RowScratch& sh, int* status, int fault) {
  const auto* X = reinterpret_cast<const __nv_bfloat16*>(fq.X);
  auto* Xq = reinterpret_cast<uint8_t*>(fq.Xq);
  auto* x16 = reinterpret_cast<uint8_t*>(fq.x16);
  for (int m = blockIdx.x; m < M; m += gridDim.x) {
    if (fq.kind == kFuseRmsNorm)
      rq::rmsnorm_quant_row<NC>(m, X, K, fq.ldx, fq.gamma, fq.eps, qt, Xq, fq.sx, nullptr, x16, sums, sh);
    else if (fq.kind == kFuseQuant)
      rq::quant_act_row<NC>(m, X, K, fq.ldx, fq.pre, qt, Xq, fq.sx, x16, sums, sh);
    else
      rq::silu_mul_quant_row<NC>(m, X, K, fq.ldx, fq.pre, qt, Xq, fq.sx, nullptr, x16, sums, sh);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    fence_proxy_async_global();  // this CTA's rows, for the TMA loads of every CTA
    if (!(fault && blockIdx.x == 0)) atomicAdd(&fq.sync[0], 1u);
    bool ok = ld_acquire_gpu(&fq.sync[0]) >= gridDim.x;
    const uint64_t t0 = globaltimer_ns();
    while (!ok) {
      __nanosleep(128);
      if (ld_acquire_gpu(&fq.sync[0]) >= gridDim.x) {
        ok = true;
      } else if (*reinterpret_cast<volatile int*>(status) != kDevOk) {
        break;
      } else if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(status, kDevOk, kDevTimeout);
        break;
      }
    }
    if (ok) {
      fence_proxy_async_global();
      // every CTA has seen all arrivals before it counts its departure, so the
      // last to depart may reset both counters for the next call
      if (atomicAdd(&fq.sync[1], 1u) == gridDim.x - 1) {
        atomicExch(&fq.sync[0], 0u);
        atomicExch(&fq.sync[1], 0u);
      }
    }
    sh.red[0] = ok ? 1.0f : 0.0f;
  }
  __syncthreads();
  const bool ok = sh.red[0] != 0.0f;
  __syncthreads();
  return ok;
}

}  // namespace qurl
