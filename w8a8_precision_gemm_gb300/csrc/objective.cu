// objective.cu -- the ACR token objective of a quantized rollout: decoupled PPO
// with the truncated importance weight of TIS and ACR's adaptive clipping range.
//
// Method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
// Quantized Rollout", section "方法详解 > 关键设计 > 自适应裁剪范围 (ACR)":
//   J = E~[ min(pi_prox / pi_behav, C) * min(R A, clip(R, 1 - eps, (1 + eps) / r) A) ]
// with r the truncated weight itself and R = pi_theta / pi_prox; section
// "损失函数 / 训练策略": the GRPO/DAPO decoupled variant, a token-level mean.
//
// HBM-bound streaming: per token slot 4 fp32 inputs + 1 mask byte in, the fp32
// derivative (and optionally the term) out.  One kernel: CTAs (four per SM)
// stride over groups of 4 consecutive tokens with 16-byte loads, reduce their
// sums (fp32 per thread, fp64 across warps) to one row of partials, and the
// last CTA to finish (a ticket on a counter in the workspace) adds the rows in
// a fixed order -- so a call is deterministic run to run -- and resets the
// counter.  (A 4-stage cp.async ring in shared memory per thread measured
// slower than the plain loads: 26.5 vs 17 us on 4.2 M slots.)
#include <cstdint>

#include "internal.h"
#include "objective.h"
#include "ptx.cuh"

namespace qurl {
namespace {

constexpr int kObjThreads = 256;
constexpr int kObjWarps = kObjThreads / 32;
constexpr int kObjCtasPerSm = 4;
constexpr int kObjPartial = 8;  // doubles per CTA row (6 used)

struct ObjAcc {
  float term = 0.f, w = 0.f, kl = 0.f;
  int n = 0, clipped = 0, capped = 0;
};

// One token.  Everything is a product or a min/max, except the two
// log-ratio differences and the bounds 1 -+ eps: no contraction into FMAs.
__device__ __forceinline__ void acr_token(float lp, float lpp, float lpb, float A, bool valid, float eps, float C,
                                          bool adaptive, float& term, float& dterm, ObjAcc& acc) {
  term = 0.f;
  dterm = 0.f;
  if (!valid) return;  // padding: its values (even NaN) are never used
  const float ratio_pb = expf(__fsub_rn(lpp, lpb));  // pi_prox / pi_behav
  const float w = fminf(ratio_pb, C);                 // truncated importance weight (= r)
  const float R = expf(__fsub_rn(lp, lpp));           // pi_theta / pi_prox
  const float lower = 1.f - eps;
  const float upper = adaptive ? __fdiv_rn(1.f + eps, w) : 1.f + eps;
  const float c = fminf(fmaxf(R, lower), upper);  // clip(R, lower, upper); upper wins when below lower
  const float u = __fmul_rn(R, A), v = __fmul_rn(c, A);
  if (u <= v) {
    term = __fmul_rn(w, u);
    dterm = __fmul_rn(__fmul_rn(w, A), R);
  } else {
    term = __fmul_rn(w, v);
    ++acc.clipped;
  }
  ++acc.n;
  acc.term = __fadd_rn(acc.term, term);
  acc.w = __fadd_rn(acc.w, w);
  acc.capped += ratio_pb > C;
  acc.kl = __fadd_rn(acc.kl, __fsub_rn(lpb, lpp));
}

__global__ void __launch_bounds__(kObjThreads, kObjCtasPerSm)
    acr_objective_kernel(const float* __restrict__ lp, const float* __restrict__ lpp, const float* __restrict__ lpb,
                         const float* __restrict__ adv, const uint8_t* __restrict__ mask, long long T, float eps,
                         float C, int adaptive, float* __restrict__ term_out, float* __restrict__ dterm_out,
                         double* __restrict__ partials, unsigned int* __restrict__ ticket, double* __restrict__ stats) {
  griddep_wait();
  griddep_launch_dependents();
  const bool ad = adaptive != 0;
  const int tid = threadIdx.x;
  ObjAcc acc;
  const long long T4 = T >> 2;
  const float4* lp4 = reinterpret_cast<const float4*>(lp);
  const float4* lpp4 = reinterpret_cast<const float4*>(lpp);
  const float4* lpb4 = reinterpret_cast<const float4*>(lpb);
  const float4* a4 = reinterpret_cast<const float4*>(adv);
  const uint32_t* m4 = reinterpret_cast<const uint32_t*>(mask);
  const long long stride = static_cast<long long>(gridDim.x) * kObjThreads;
  for (long long g = static_cast<long long>(blockIdx.x) * kObjThreads + tid; g < T4; g += stride) {
    const float4 x = __ldcs(lp4 + g), p = __ldcs(lpp4 + g), b = __ldcs(lpb4 + g), a = __ldcs(a4 + g);
    const uint32_t m = __ldcs(m4 + g);
    float4 t, d;
    acr_token(x.x, p.x, b.x, a.x, (m & 0xFFu) != 0, eps, C, ad, t.x, d.x, acc);
    acr_token(x.y, p.y, b.y, a.y, (m & 0xFF00u) != 0, eps, C, ad, t.y, d.y, acc);
    acr_token(x.z, p.z, b.z, a.z, (m & 0xFF0000u) != 0, eps, C, ad, t.z, d.z, acc);
    acr_token(x.w, p.w, b.w, a.w, (m & 0xFF000000u) != 0, eps, C, ad, t.w, d.w, acc);
    if (dterm_out) __stcs(reinterpret_cast<float4*>(dterm_out) + g, d);
    if (term_out) __stcs(reinterpret_cast<float4*>(term_out) + g, t);
  }
  // the last T mod 4 slots
  if (blockIdx.x == 0 && tid < (T & 3)) {
    const long long k = (T4 << 2) + tid;
    float t, d;
    acr_token(lp[k], lpp[k], lpb[k], adv[k], mask[k] != 0, eps, C, ad, t, d, acc);
    if (dterm_out) dterm_out[k] = d;
    if (term_out) term_out[k] = t;
  }
  // CTA reduction: fixed shuffle pattern within warps, then the warps in order in fp64
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc.term = __fadd_rn(acc.term, __shfl_xor_sync(0xFFFFFFFFu, acc.term, o));
    acc.w = __fadd_rn(acc.w, __shfl_xor_sync(0xFFFFFFFFu, acc.w, o));
    acc.kl = __fadd_rn(acc.kl, __shfl_xor_sync(0xFFFFFFFFu, acc.kl, o));
    acc.n += __shfl_xor_sync(0xFFFFFFFFu, acc.n, o);
    acc.clipped += __shfl_xor_sync(0xFFFFFFFFu, acc.clipped, o);
    acc.capped += __shfl_xor_sync(0xFFFFFFFFu, acc.capped, o);
  }
  __shared__ double warp_sums[kObjWarps][6];
  __shared__ unsigned int last;
  const int warp = tid >> 5;
  if ((tid & 31) == 0) {
    warp_sums[warp][0] = acc.term;
    warp_sums[warp][1] = acc.n;
    warp_sums[warp][2] = acc.clipped;
    warp_sums[warp][3] = acc.w;
    warp_sums[warp][4] = acc.capped;
    warp_sums[warp][5] = acc.kl;
  }
  __syncthreads();
  if (tid < 6) {
    double s = 0.0;
    for (int j = 0; j < kObjWarps; ++j) s += warp_sums[j][tid];
    partials[static_cast<size_t>(blockIdx.x) * kObjPartial + tid] = s;
    __threadfence();  // the row is visible device-wide before this CTA takes its ticket
  }
  __syncthreads();
  if (tid == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  // the last CTA: every row is written; warp k adds statistic k over the rows
  // in a fixed order (lane l takes rows l, l + 32, ..., then a fixed shuffle tree)
  __threadfence();
  const int lane = tid & 31;
  if (warp < 6) {
    double t = 0.0;
    for (int r = lane; r < static_cast<int>(gridDim.x); r += 32)
      t += __ldcg(partials + static_cast<size_t>(r) * kObjPartial + warp);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if (lane == 0) warp_sums[0][warp] = t;  // the per-warp sums above are no longer needed
  }
  __syncthreads();
  if (tid == 0) {
    const double* tot = warp_sums[0];
    const double n = tot[1];
    const bool any = n > 0.0;
    stats[0] = any ? tot[0] / n : 0.0;  // the objective: mean term over the valid tokens
    stats[1] = n;
    stats[2] = any ? tot[2] / n : 0.0;  // clipped fraction
    stats[3] = any ? tot[3] / n : 0.0;  // mean truncated weight
    stats[4] = any ? tot[4] / n : 0.0;  // fraction with pi_prox / pi_behav > C
    stats[5] = any ? tot[5] / n : 0.0;  // mean logp_behav - logp_prox (KL(behav || prox))
    *ticket = 0;                        // ready for the next call on this workspace
  }
}

}  // namespace

int acr_grid(long long T, int num_sms) {
  const long long want = ((T >> 2) + kObjThreads - 1) / kObjThreads;
  const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * kObjCtasPerSm;
  long long g = want < cap ? want : cap;
  if (g > kAcrMaxCtas) g = kAcrMaxCtas;
  return g < 1 ? 1 : static_cast<int>(g);
}

cudaError_t launch_acr_objective(const float* lp, const float* lpp, const float* lpb, const float* adv,
                                 const uint8_t* mask, long long T, float eps, float C, int adaptive, float* term,
                                 float* dterm, double* stats, void* workspace, int num_sms, cudaStream_t st) {
  const int grid = acr_grid(T, num_sms);
  double* partials = reinterpret_cast<double*>(workspace);
  unsigned int* ticket = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + kAcrTicketOffset);
  return launch_pdl(acr_objective_kernel, dim3(grid), dim3(kObjThreads), 0, st, lp, lpp, lpb, adv, mask, T,
                    eps, C, adaptive, term, dterm, partials, ticket, stats);
}

}  // namespace qurl
