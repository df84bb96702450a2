// internal.h -- declarations shared by the translation units of libqurl
// (not part of the public ABI; the public header is include/qurl.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

namespace qurl {

// Status codes written by kernels into the per-device status word.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 6;  // QURL_ERR_TIMEOUT
constexpr int kDevBadIndex = 1;  // QURL_ERR_INVALID_ARG: an index read on the device was out of range

constexpr int kQInt8 = 0;  // QURL_INT8
constexpr int kQFp8 = 1;   // QURL_FP8_E4M3

// Token tiles per group of the INT8 CTA-pair prefill kernel's tile order.
constexpr int kWideTokGroup = 16;
constexpr int kModeBf16 = 0;  // GEMM epilogue dequantizes and writes Y
constexpr int kModeAcc = 1;   // GEMM writes the raw accumulator of its split to part

// Per-token sums of |code| over consecutive ranges of sum_len codes (the K
// splits of the INT8 decode GEMM): asum[m * nsum + j], j < nsum.  Written by
// the kernel that writes the fp16 copy of the codes; asum null: not wanted.
constexpr int kMaxSums = 128;
struct CodeSums {
  int* asum;
  int sum_len;     // a multiple of 256
  int nsum;        // <= kMaxSums
  unsigned* qsum;  // the sums of code^2 over the same ranges (saturated at 2^32 - 1), or null
};

// The quantizer of a fused entry point, run by the decode GEMM kernel itself
// before its main loop (kind 0: none -- the activation codes are an input).
// Every CTA quantizes rows blockIdx.x, blockIdx.x + gridDim.x, ... < M and the
// CTAs then hand over through two counters in the caller's workspace.
constexpr int kFuseNone = 0;
constexpr int kFuseRmsNorm = 1;  // RMSNorm with the folded gain -> quant
constexpr int kFuseQuant = 2;    // quant with the UAQ pre-scale
constexpr int kFuseSiluMul = 3;  // SiLU(gate) * up -> quant (pre-scale)
struct FusedQuant {
  int kind;
  const void* X;       // bf16 [M, ldx] (kFuseSiluMul: [M, 2K], gate | up)
  long long ldx;
  const float* gamma;  // kFuseRmsNorm: folded gain [K]
  float eps, pre;
  void* Xq;            // codes [M, K]
  float* sx;           // scales [M]
  void* x16;           // INT8 decode: the fp16 copy of the codes (and `sums`), else null
  unsigned* sync;      // two handoff counters, zero between calls
};

struct GemmArgs {
  int M, N, K;       // tokens, output channels, depth
  int num_kb;        // k-blocks covering K
  int kb_per_split;  // k-blocks per split
  int tiles_tok;     // work units = tiles_tok x tiles_ch x splits, token tile fastest;
  int tiles_ch;      // a persistent CTA takes units blockIdx.x, blockIdx.x + gridDim.x, ...
  int splits;
  int mode;
  const float* sx;   // [M]
  const float* sw;   // [N]
  __nv_bfloat16* Y;  // [M, ldy]
  long long ldy;
  void* part;        // [splits][M][N] int32 (INT8) or fp32 (FP8), mode kModeAcc
  int* status;       // device status word
  int w_prefetch;    // the previous kernel in the stream does not write Wq and triggers
                     // its dependents only after its own wait (so every earlier kernel has
                     // completed): the first stages may be loaded before waiting for it
  void* acc_out;       // raw-accumulator output [M, N] (unused by the kernels; kept with the call)
  int fault;           // test hook: 1 = the producer skips its first k-block, so the consumer's
                       // bounded wait runs out and the kernel latches a timeout
  const int* asum;     // INT8 decode: [M][splits] sums of |Xq[m,k]| over each split's k range
                       // (null: every unit accumulates in chunks)
  const unsigned* qsum;  // INT8 on pairs with widened weights: [M][splits] sums of Xq[m,k]^2 over
                         // each split's k range, and
  const unsigned* qn;    // [N] sums of Wq[n,k]^2 over all of K (null: not available)
  int* scratch;          // INT8: per CTA, the int32 running sum of a unit accumulated in chunks
  FusedQuant fq;         // decode fused entries: the quantizer this kernel runs first
  CodeSums fsums;        // ... and where it writes the code sums (INT8 decode)
  int float_acc;         // fp16 operands that are not integers (the 4-bit variant): every unit in
                         // one fp32 pass, fp32 partials
  int whole_units;       // CTA-pair prefill kernels: the first whole_units tiles (in their unit order) run
                         // over all of K as single units, only the rest are split `splits` ways (0: all)
  int tok_group;         // FP8 CTA-pair prefill: token tiles per group of its tile order (group_tile)
};

// Number of kernels this library has launched in the process (api.cu).
extern std::atomic<unsigned long long> g_kernel_launches;

// Launch a kernel with programmatic stream serialization: it may start while
// the previous kernel in the stream finishes; every kernel of this library
// calls griddepcontrol.wait before it reads anything the previous kernel may
// have written (weights excepted where the caller says they are not written
// there, see GemmArgs::w_prefetch).
//
// Who may start early.  The GEMMs allow their dependents to launch right after
// their prologue.  Every other kernel (quantizers, widening, reductions, weight
// preparation, the objective) allows it only after its own griddepcontrol.wait
// has returned, i.e. once the kernel before it has completed.  A GEMM that
// loads weight tiles before its own wait (w_prefetch) follows one of those
// kernels, so its launch implies that every kernel two or more places earlier
// in the stream -- e.g. a qurl_prepare_weights that rewrote Wq -- has completed
// and its writes are visible.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// launch_pdl for a kernel whose CTAs work in clusters of two (grid.x even).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_pair(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// quant.cu.  x16 (may be null): also write the INT8 codes as fp16 [M, K]
// (the operand the INT8 decode GEMM reads), saving it a widening pass, and,
// when sums.asum is not null, the code sums the GEMM reads with it.
cudaError_t launch_quant_act(const void* X, int M, int K, long long ldx, float pre, int qt, void* Xq, float* sx,
                             void* x16, CodeSums sums, cudaStream_t st);
cudaError_t launch_rmsnorm_quant(const void* X, int M, int K, long long ldx, const float* gamma, float eps,
                                 int qt, void* Xq, float* sx, float* ms_out, void* x16, CodeSums sums,
                                 cudaStream_t st);
// status: the device status word, where the streaming SiLU kernel latches a
// timed-out row copy (null: the row kernels, which wait on nothing, only).
cudaError_t launch_silu_mul_quant(const void* GU, int M, int I, long long ldgu, float pre, int qt, void* Xq,
                                  float* sx, float* h_out, void* x16, CodeSums sums, int* status, cudaStream_t st);
cudaError_t launch_prepare_weights(const void* W, bool w_f32, int N, int K, long long ldw, const float* gamma,
                                   float s, int qt, void* Wq, float* sw, float* gamma_folded, float* W_scaled,
                                   cudaStream_t st);
cudaError_t launch_count_diff(const void* a, const void* b, size_t n, unsigned long long* count, int num_sms,
                              cudaStream_t st);
// quant.cu: FP8 key/value cache quantization into slots, and its read-back (status: the device status word)
cudaError_t launch_kv_cache_quant(const void* QKV, int M, long long ldq, int q_dim, int kv_heads, int head_dim,
                                  const long long* slots, long long num_slots, void* kc, float* ks, void* vc,
                                  float* vs, int* status, cudaStream_t st);
cudaError_t launch_kv_cache_dequant(const void* cache, const float* scale, const long long* slots, int n,
                                    int kv_heads, int head_dim, long long num_slots, void* out, int* status,
                                    cudaStream_t st);

// How one GEMM call is cut into CTAs.
struct GemmPlan {
  bool swap;         // weights on the MMA M side (decode)
  bool tmem_a;       // INT8 decode: weights widened into TMEM, fp16 activation copy in the workspace
  bool pair;         // CTA pairs: 256-row A tiles per pair (FP8 prefill: tokens; FP8 swap and the INT8
                     // TMEM-operand kernel: channels), each CTA staging half of the bn B rows
  size_t x16_bytes;  // bytes at the start of the workspace for that fp16 copy and, after it
                     // (at asum_off), the per-token sums of |code| (256-aligned pieces)
  size_t asum_off;
  int bn;            // MMA N (tile width on the B side)
  int bk;            // k per k-block (per stage: 256 for the TMEM-operand INT8 kernel)
  int tiles_tok;     // grid.x
  int tiles_ch;      // grid.y
  int splits;        // grid.z
  int num_kb;
  int kb_per_split;
  size_t part_bytes;  // split-K partials (after the fp16 copy)
  size_t ws_bytes;    // total workspace: fp16 activation copy + split-K partials
  // INT8 on CTA pairs with both operands widened to fp16 in the workspace (prefill):
  bool wide;
  size_t qsum_off;     // per-token sums of code^2 (after the sums of |code|)
  size_t w16_off;      // fp16 copy of the weight codes [N, K]
  size_t qn_off;       // per-channel sums of code^2 [N]
  size_t scratch_off;  // running sums of chunked units, one region per CTA
  int whole_units;     // tiles that run unsplit before the split tail (GemmArgs::whole_units)
};

// gemm_common.cu.  ws_bytes of a plan includes kSyncBytes at the end of the
// workspace: the two handoff counters of the fused entry points live in the
// last kSyncBytes of the caller's workspace.
constexpr size_t kSyncBytes = 256;
GemmPlan plan_gemm(int M, int N, int K, int qt, int num_sms, size_t ws_avail);
// The 4-bit variant's plan: the CTA-pair layout of the INT8 prefill (both operands widened to fp16
// in the workspace), for every M; false when ws_avail is short.
bool plan_nvfp4(GemmPlan& p, int M, int N, int K, int num_sms, size_t ws_avail, bool w_attached = false);
// INT8 with the weights' fp16 copy attached by the caller (no weight region in the workspace):
// the CTA-pair plan for batches above 256 tokens; false otherwise or when ws_avail is short.
bool plan_attached(GemmPlan& p, int M, int N, int K, int num_sms, size_t ws_avail);
// api.cu: the workspace the shape's plan asks for on the current device when no fp16 weight copy is
// attached (0 for invalid arguments).
size_t plain_workspace_bytes(int M, int N, int K, int qt);

// gemm_fp8.cu / gemm_i8.cu / gemm_i8t.cu: launch the instantiation matching
// (swap, bn) as a persistent grid.  grid = (token tiles, channel tiles, K
// splits); with K split, each split writes its raw partial (mode kModeAcc) and
// launch_splitk_reduce sums them.
cudaError_t launch_gemm_fp8(bool swap, int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                            dim3 grid, cudaStream_t st);
cudaError_t launch_gemm_i8(bool swap, int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                           dim3 grid, cudaStream_t st);
// gemm_fp8p.cu: FP8 on CTA pairs, 256-row A tiles per pair (grid = token tiles, channel tiles,
// K splits; prefill: 256 tokens x 256 channels, swap: 256 channels x bn tokens, bn in {64, 128, 256}).
cudaError_t launch_gemm_fp8_pair(bool swap, int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                                 dim3 grid, cudaStream_t st);
// gemm_i8t.cu: the INT8 decode GEMM with the weight operand in TMEM, and the
// int8 -> fp16 widening of the activation codes it reads.
cudaError_t launch_gemm_i8t(int bn, const CUtensorMap& tw, const CUtensorMap& tx16, const GemmArgs& a, dim3 grid,
                            cudaStream_t st);
// gemm_i8t.cu: the same on CTA pairs, 256 channels x 256 tokens per pair (grid = 256-token tiles,
// 256-channel tiles, K splits; the fp16 codes' tensor map has 64-row boxes).
cudaError_t launch_gemm_i8p(const CUtensorMap& tw, const CUtensorMap& tx16, const GemmArgs& a, dim3 grid,
                            cudaStream_t st);
// int8 codes [M, K] -> fp16 [M, K] in dst, and the sums of |code| (saturated at 2^24).
cudaError_t launch_i8_to_f16(const void* src, void* dst, int M, int K, CodeSums sums, cudaStream_t st);
// gemm_i8w.cu: the INT8 GEMM on CTA pairs with both operands widened to fp16 (grid = 256-token tiles,
// 256-channel tiles, K splits), and the widening of the weight codes with their sums of code^2.
cudaError_t launch_gemm_i8w(const CUtensorMap& tx16, const CUtensorMap& tw16, const GemmArgs& a, dim3 grid,
                            cudaStream_t st);
// The reduction of a hybrid plan's split tail: the tiles after the first whole_units (in the CTA-pair
// kernels' tile order, groups of tok_group token tiles: group_tile in gemm.cuh) sum their s partials
// in split order and apply the epilogue (or write acc_out).
cudaError_t launch_tail_reduce(bool int_partials, int tok_group, const GemmArgs& a, cudaStream_t st);
cudaError_t launch_widen_weights(const void* Wq, int N, int K, void* w16, unsigned* qn, int num_sms,
                                 cudaStream_t st);
// the CTAs an i8w launch of this plan runs (one per SM of the resident pairs), for sizing its scratch
int i8w_max_ctas(int num_sms);

// nvfp4.cu: the 4-bit variant's row quantizer (bf16 rows times pre, or fp32 rows) and the exact
// widening of its rows to fp16.
cudaError_t launch_nvfp4_quant(const void* X, bool x_f32, int R, int K, long long ldx, float pre, void* q4,
                               void* sblk, float* g, cudaStream_t st);
cudaError_t launch_nvfp4_widen(const void* q4, const void* sblk, int R, int K, void* out16, int num_sms,
                               cudaStream_t st);
// split-K reduction in split order: T = int (INT8) or float (FP8)
cudaError_t launch_splitk_reduce(int qt, const void* part, int splits, int M, int N, const float* sx,
                                 const float* sw, void* Y, long long ldy, void* acc_out, int num_sms,
                                 cudaStream_t st);
// probe.cu: tensor-rate probes (route 0: mma.sync s8; 1: tcgen05 kind::f16 from shared memory; 2: the
// same with A in TMEM; 3: tcgen05 kind::f8f6f4), and the multiply-add operations x 2 of a launch.
cudaError_t launch_probe(int route, int ctas, int iters, int* status, cudaStream_t st);
double probe_ops(int route, int ctas, int iters);
}  // namespace qurl
