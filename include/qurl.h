/*
 * qurl.h -- C ABI of libqurl, the W8A8 linear layer of QuRL's quantized
 * rollout actor on one NVIDIA GB300 (sm_103a).
 *
 * Source of the method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement
 * Learning with Quantized Rollout":
 *   [UAQ]   section "方法详解 > 关键设计 > 更新感知量化 (UAQ)": W X = (W/s)(sX);
 *           s is applied column-wise to W and row-wise to the preceding
 *           activation, and can be folded into the preceding norm gain.
 *   [LOSS]  section "损失函数 / 训练策略": per-channel (output channel) weight
 *           quantization and per-token activation quantization, INT8 or FP8;
 *           UAQ factor s = 1.5.
 *   [SYS]   section "系统集成与工程实现": UAQ is a one-time preprocessing of
 *           the weights; the rollout runs INT8/FP8 matrix-multiply kernels.
 *   [FRAME] section "方法详解 > 整体框架": every RL step quantizes the current
 *           weights theta_old for the rollout.
 *   [ACR]   section "方法详解 > 关键设计 > 自适应裁剪范围 (ACR)": the decoupled
 *           PPO objective with the truncated weight min(pi_prox / pi_behav, C)
 *           and the clipping range [1 - eps, (1 + eps) / r].
 *   [OBJ]   section "损失函数 / 训练策略": the GRPO/DAPO decoupled variant, a
 *           token-level mean.
 *   [LIMITS] section "局限与展望": FP8 KV-cache quantization is not yet
 *           optimized in the rollout engine (page 5's FP8-RL entry quantizes
 *           the KV cache to FP8); 4-bit quantization would speed the rollout
 *           up further but was not explored (page 5's QeRL entry uses NVFP4).
 *
 * Conventions (all entry points):
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *     allocates no device memory on any of these calls and keeps no pointer
 *     after a call returns.
 *   - Row-major layouts.  M = tokens, K = in-features, N = out-features.
 *     X: [M, K] bf16 with row stride ldx (elements).  W / Wq: [N, K] (the
 *     torch Linear layout, K contiguous).  Y: [M, N] bf16 with row stride ldy.
 *     Codes (Xq, Wq) are one byte each: int8 two's complement (QURL_INT8) or
 *     OCP FP8 E4M3 "e4m3fn" (QURL_FP8_E4M3), densely packed with stride K.
 *     Scales (sx [M], sw [N]) are fp32.
 *   - Quantization is symmetric absmax per row: scale = absmax / qmax (IEEE
 *     fp32 division, qmax = 127 for INT8, 448 for FP8), code = v / scale
 *     (IEEE division) rounded to nearest even and clamped to [-127, 127]
 *     (INT8) or converted with round-to-nearest-even and saturation to
 *     +-448 (FP8).  An all-zero row has scale 1 and zero codes.  NaN inputs
 *     are outside the domain.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and may be captured in a CUDA graph.  They validate
 *     their arguments on the host BEFORE any launch and return QURL_OK or an
 *     error code; nothing is launched when an error is returned.  They never
 *     throw and never abort.
 *   - Device-side failures (a bounded wait inside a kernel that ran out, ~1 s)
 *     are latched in a per-device status word; qurl_check_device_status()
 *     synchronises the stream and returns (and clears) it.
 *   - Alignment: every pointer passed as a tensor must be 16-byte aligned and
 *     every row stride must be a multiple of 16 bytes; K must be a multiple
 *     of 16.  Violations return QURL_ERR_ALIGNMENT / QURL_ERR_UNSUPPORTED.
 *   - Sizes: M, N, K in [1, 2^31); M*K, N*K, M*N below 2^40.
 */
#ifndef QURL_H_
#define QURL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QURL_OK = 0,
    QURL_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, unknown enum, bad stride */
    QURL_ERR_UNSUPPORTED = 2, /* shape the kernels do not cover (e.g. K % 16 != 0) */
    QURL_ERR_ALIGNMENT = 3,   /* pointer or row stride not 16-byte aligned */
    QURL_ERR_WORKSPACE = 4,   /* scratch too small: the workspace given to qurl_acr_objective, or the
                                 buffer built into qurl_w8a8_linear_static_scratch for this shape */
    QURL_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed */
    QURL_ERR_TIMEOUT = 6      /* a device-side bounded wait ran out */
} qurl_status;

typedef enum { QURL_INT8 = 0, QURL_FP8_E4M3 = 1 } qurl_qtype;
typedef enum { QURL_BF16 = 0, QURL_FP32 = 1 } qurl_ftype;

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* qurl_stream_t;

/*
 * UAQ weight preparation + per-output-channel weight quantization
 * ([UAQ], [LOSS], [SYS], [FRAME]).
 *
 *   W'[n,k]     = W[n,k] / s          (IEEE fp32 division; the same scalar s
 *                                      on every input column)
 *   gamma'[k]   = gamma[k] * s        (the preceding RMSNorm gain, fp32)
 *   sw[n]       = max_k |W'[n,k]| / qmax
 *   Wq[n,k]     = quantize(W'[n,k] / sw[n])
 *
 * Called once with s = 1.5 at set-up (the fold), then every RL step with the
 * trained W' and s = 1 (re-quantization of the current weights).
 *
 *   W            [N, K] bf16 or fp32 (w_type), row stride ldw elements.
 *   gamma        [K] fp32 or NULL (no norm to fold into).
 *   s            > 0, finite.
 *   Wq           [N, K] codes (out).        sw [N] fp32 (out).
 *   gamma_folded [K] fp32 (out) or NULL; required when gamma is given.
 *   W_scaled     [N, K] fp32 (out) or NULL: W', the new training master.
 *                May alias W when w_type == QURL_FP32 and ldw == K.
 */
qurl_status qurl_prepare_weights(const void* W, qurl_ftype w_type, int N, int K, int ldw, const float* gamma,
                                 float s, qurl_qtype qt, void* Wq, float* sw, float* gamma_folded,
                                 float* W_scaled, qurl_stream_t stream);

/*
 * Per-token dynamic activation quantization ([LOSS]).
 *   v[m,k] = fp32(X[m,k]) * pre_scale;  sx[m] = max_k |v| / qmax;
 *   Xq[m,k] = quantize(v[m,k] / sx[m]).
 * pre_scale carries the UAQ factor s into an activation that has no norm to
 * fold it into ([UAQ]: "row-wise on the preceding activation"); pass 1.0f
 * otherwise.  X [M, K] bf16 with row stride ldx; Xq [M, K] (stride K); sx [M].
 */
qurl_status qurl_quant_act(const void* X, int M, int K, int ldx, float pre_scale, qurl_qtype qt, void* Xq,
                           float* sx, qurl_stream_t stream);

/*
 * RMSNorm with the folded gain gamma' = gamma * s, then per-token quantization
 * ([UAQ] fold into the norm, [LOSS]).
 *   ms[m] = (sum_k x^2) / K: each x^2 is exact in fp32 and the sum is kept
 *           as an error-free compensated pair, divided by K in fp64 and
 *           rounded to fp32 -- the correctly rounded mean unless it lies
 *           within ~2^-44 (relative) of an fp32 rounding midpoint;
 *   r = 1 / sqrt(ms + eps) (correctly rounded fp32 sqrt and division);
 *   v[m,k] = (x * r) * gamma'[k] (two fp32 products); then as qurl_quant_act.
 * ms_out [M] fp32 or NULL receives ms (lets a checker reproduce the codes).
 */
qurl_status qurl_rmsnorm_quant(const void* X, int M, int K, int ldx, const float* gamma_folded, float eps,
                               qurl_qtype qt, void* Xq, float* sx, float* ms_out, qurl_stream_t stream);

/*
 * SiLU(gate) * up, then per-token quantization: the MLP activation between
 * the fused gate_up and the down projection.  GU [M, 2I] bf16, row stride
 * ldgu; columns [0, I) are the gate g, [I, 2I) the up projection u.
 *   h = (g / (1 + exp(-g))) * u (fp32);  v = h * pre_scale;  quantize rows.
 * Xq [M, I] (stride I), sx [M]; h_out [M, I] fp32 or NULL receives h.
 * I must be a multiple of 16.
 */
qurl_status qurl_silu_mul_quant(const void* GU, int M, int I, int ldgu, float pre_scale, qurl_qtype qt,
                                void* Xq, float* sx, float* h_out, qurl_stream_t stream);

/*
 * Bytes of workspace the linear entry points (qurl_w8a8_linear,
 * qurl_w8a8_gemm_acc and the fused *_linear entries) use for this shape at
 * full speed: split-K partial sums and, for INT8, an fp16 copy of the
 * activation codes (2 M K bytes) with per-token sums of |code| over each K
 * split, the int32 running sums of units accumulated in chunks (one region
 * per SM), and from 2048 tokens on an fp16 copy of the weight codes (2 N K
 * bytes) with their per-channel sums of squares; above 256 tokens (and from
 * 129 tokens for weights of 2^26 codes or more) also enough for the plan that
 * reads an attached fp16 weight copy (qurl_widen_weights) instead.  The last
 * 256 bytes of any
 * workspace hold two counters through which the CTAs of a fused decode call
 * hand over (see the fused entries): they must be zero before the
 * workspace's first use by a fused entry, and every call leaves them zero.
 * A smaller workspace (or none) is accepted: the kernels then split K into
 * fewer parts and INT8, without room for the fp16 copies, keeps the weights
 * in TMEM or widens both operands in shared memory instead (slower, same
 * result); a fused entry then runs its quantizer as a separate kernel.
 */
size_t qurl_workspace_size(int M, int N, int K, qurl_qtype qt);

/*
 * The W8A8 linear layer ([SYS], [LOSS]):
 *   acc[m,n] = sum_k Xq[m,k] * Wq[n,k]   (INT8: exact int32; FP8: fp32)
 *   Y[m,n]   = bf16_RNE( (fp32(acc) * sx[m]) * sw[n] )
 * Xq [M, K], Wq [N, K] codes; sx [M], sw [N] fp32; Y [M, N] bf16, row stride
 * ldy.  workspace: device scratch of ws_bytes (may be NULL / 0).
 * INT8 runs on the fp16 tensor path: the codes are widened to fp16 (exact)
 * and accumulated in fp32, which is exact while every partial sum is an
 * integer of magnitude <= 2^24: a tile is accumulated in one pass when its
 * tokens have sum |x| <= 2^24 / 128 over the k range, or (on the CTA-pair
 * kernel) when max over its tokens of sum x^2 times max over its channels of
 * sum w^2 is <= 2^48 (Cauchy-Schwarz bounds every partial sum by 2^24), and
 * in 1024-deep chunks (1024 * 128^2 = 2^24) added in int32 otherwise.  The
 * int32 accumulator and the bf16 Y are therefore exact for any codes.
 */
qurl_status qurl_w8a8_linear(const void* Xq, const float* sx, const void* Wq, const float* sw, int M, int N,
                             int K, qurl_qtype qt, void* Y, int ldy, void* workspace, size_t ws_bytes,
                             qurl_stream_t stream);

/*
 * qurl_w8a8_linear without a caller-provided workspace and without allocating:
 * the same computation and the same results as qurl_w8a8_linear given a
 * workspace (of the size the shape's plan asks for when no fp16 weight copy
 * is attached, qurl_widen_weights), but its scratch is a
 * 32 MiB buffer compiled into the library (a file-scope device array), so
 * neither the caller nor the library has to allocate device memory for it.
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate: an engine that has already reserved all of
 * HBM for its own pools (KV caches sized to fill the device), code paths that
 * must not risk an allocation failure or the device-wide synchronisation a
 * cudaMalloc / cudaFree can bring in the middle of a decode loop, and foreign
 * callers that have no handle on the application's allocator.
 *
 *   - Limit: a shape whose plan needs more than 32 MiB (33,554,432 bytes)
 *     returns QURL_ERR_WORKSPACE and launches nothing.  Every 7B-class
 *     decode projection up to M = 256 fits, and every 32B-class one but the
 *     INT8 down projection (K = 27648) at M = 256.
 *   - The buffer lives in a CUDA module of its own.  Under the CUDA runtime's
 *     default lazy module loading, a device commits its 32 MiB on the first
 *     call of this entry point made with that device current (the call looks
 *     the buffer's device address up with cudaGetSymbolAddress, which loads
 *     the module) and holds them until the process exits; devices on which
 *     only other entry points are called do not hold it.  Under
 *     CUDA_MODULE_LOADING=EAGER the module is loaded, on every device the
 *     library is used on, when the library's first call binds that device's
 *     context.  A caller that reserves the rest of HBM for its own pools
 *     should therefore make one call of this entry point on each device
 *     before reserving, and make that first call before any stream capture.
 *   - All calls on a device share the buffer, and it keeps what the last call
 *     left there (nothing in it needs to start at zero).  Calls whose kernels
 *     overlap on the GPU -- e.g. issued on two streams without ordering between
 *     them -- race on it; serialise them (one stream, or events).
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 */
qurl_status qurl_w8a8_linear_static_scratch(const void* Xq, const float* sx, const void* Wq, const float* sw,
                                            int M, int N, int K, qurl_qtype qt, void* Y, int ldy,
                                            qurl_stream_t stream);

/*
 * The raw accumulator of the 8-bit GEMM, acc [M, N] (stride N): int32 for
 * INT8 (exact), fp32 for FP8.  For checking the GEMM on its own.
 */
qurl_status qurl_w8a8_gemm_acc(const void* Xq, const void* Wq, int M, int N, int K, qurl_qtype qt, void* acc,
                               void* workspace, size_t ws_bytes, qurl_stream_t stream);

/*
 * Fused entry: RMSNorm(gamma') -> per-token quantization -> W8A8 linear
 * ([UAQ]: s lives in gamma', so Y = W (RMSNorm_gamma(X)) up to quantization).
 * Xq_scratch [M, K] codes and sx_scratch [M] fp32 are caller-provided
 * intermediate buffers (they hold the quantized activation afterwards).
 *
 * The fused entries (this one and the two below) compute exactly what their
 * quantizer followed by qurl_w8a8_linear computes.  For decode batches (M <=
 * 256) with a full workspace they are ONE kernel (plus the split-K reduction
 * where K is split): the GEMM's CTAs first quantize the input rows between
 * them, hand over through the two counters in the workspace's last 256 bytes
 * (zero before the first use, left zero by every call), then run the product.
 * Calls sharing a workspace must not overlap on the GPU.  If that handoff
 * times out (qurl_check_device_status returns QURL_ERR_TIMEOUT) the counters
 * are left set: zero the workspace's last 256 bytes before its next use.
 * Otherwise (prefill, or a smaller workspace) the quantizer is a separate
 * kernel launched before the GEMM.
 */
qurl_status qurl_rmsnorm_quant_linear(const void* X, int ldx, const float* gamma_folded, float eps,
                                      const void* Wq, const float* sw, int M, int N, int K, qurl_qtype qt,
                                      void* Y, int ldy, void* Xq_scratch, float* sx_scratch, void* workspace,
                                      size_t ws_bytes, qurl_stream_t stream);

/*
 * Fused entry: per-token quantization (with the UAQ pre-scale) -> W8A8 linear,
 * for a projection with no norm in front of it (o_proj: s moves to the
 * activation, [UAQ]).  Same arguments and scratch buffers as above.
 */
qurl_status qurl_quant_act_linear(const void* X, int ldx, float pre_scale, const void* Wq, const float* sw, int M,
                                  int N, int K, qurl_qtype qt, void* Y, int ldy, void* Xq_scratch, float* sx_scratch,
                                  void* workspace, size_t ws_bytes, qurl_stream_t stream);

/*
 * Fused entry: SiLU(gate) * up -> per-token quantization (pre-scale) -> W8A8
 * linear (the down projection; K = I).  GU [M, 2I] bf16, row stride ldgu.
 */
qurl_status qurl_silu_mul_quant_linear(const void* GU, int ldgu, float pre_scale, const void* Wq, const float* sw,
                                       int M, int N, int I, qurl_qtype qt, void* Y, int ldy, void* Xq_scratch,
                                       float* sx_scratch, void* workspace, size_t ws_bytes, qurl_stream_t stream);

/*
 * Weight-update probe ([UAQ]: the quantization error shrinks by s while the
 * update grows by s): *count (device, uint64) = number of byte positions where
 * the code buffers a and b (n bytes each) differ.  *count is overwritten.
 */
qurl_status qurl_count_diff(const void* a, const void* b, size_t n, unsigned long long* count,
                            qurl_stream_t stream);

/*
 * A persistent fp16 copy of an INT8 weight matrix for the prefill GEMM.  INT8
 * products run on the fp16 tensor cores (the codes are exact in fp16); for
 * large batches (the plan reported as kernel 4 by qurl_debug_plan) the GEMM
 * reads an fp16 copy of Wq and the per-channel sums of code^2, which a linear
 * call otherwise writes into its workspace every time (2 N K + 4 N bytes
 * written, N K read).  qurl_widen_weights writes that copy into the caller's
 * buffer `wide` (qurl_wide_weights_size(N, K) bytes, 16-byte aligned, owned by
 * the caller) and attaches it to Wq: later linear calls on this Wq with the
 * same N, K read it instead.  qurl_prepare_weights into an attached Wq (the
 * per-RL-step re-quantization) refreshes the copy on the same stream; codes
 * written into Wq by any other means require calling qurl_widen_weights
 * again before the next linear call, or the copy is stale.
 * qurl_detach_wide_weights(Wq) forgets the attachment; call it before
 * freeing Wq or `wide` (the table is keyed by Wq's address and shape, so a
 * later matrix allocated at that address would otherwise inherit the copy).
 * Up to 1024 matrices are attached at a time (more: the call returns
 * QURL_ERR_UNSUPPORTED).  With a copy attached, INT8 calls above 256 tokens,
 * and from 129 tokens on weights of 2^26 codes or more, run on the CTA-pair
 * kernel that reads it (qurl_workspace_size covers that plan); outputs are
 * bit-identical either way.  Attaching or detaching must
 * not run concurrently with calls on the same Wq.
 * Errors: INVALID_ARG (NULL, a non-positive size), UNSUPPORTED (K % 16, table
 * full), ALIGNMENT.  One kernel launch.
 */
size_t qurl_wide_weights_size(int N, int K);
qurl_status qurl_widen_weights(const void* Wq, int N, int K, void* wide, qurl_stream_t stream);
qurl_status qurl_detach_wide_weights(const void* Wq);

/*
 * 4-bit variant (W4A4, NVFP4) of the linear layer ([LIMITS]: 4-bit named as
 * the next speedup; the format itself is a reading, the pages do not define
 * it).  A row (an output channel of W, a token of X) of K values, K a multiple
 * of 16, is stored as
 *   q4   [K/2] bytes: E2M1 codes (sign bit 3; magnitudes 0, 0.5, 1, 1.5, 2,
 *        3, 4, 6 for codes 0..7), value 2j in the low nibble of byte j;
 *   sblk [K/16] bytes: one OCP E4M3 scale per 16 consecutive values;
 *   g    fp32: the row's second-level scale;
 * and a value is dec(code) * dec(sblk) * g.  Quantization of a row v (IEEE
 * fp32 throughout): A = max|v|; g = A / 2688 (6 * 448), 1 for an all-zero
 * row; per block s = e4m3_RNE_satfinite(max|v_block| / fl(6 g)); step e =
 * fl(dec(s) * g); code = e2m1_RNE_satfinite(v / e) with the sign of v kept
 * (also on zero), and every code 0 where e = 0.
 *
 * qurl_nvfp4_quant: R rows of X ([R, ldx], bf16 with v = x * pre_scale, or
 * fp32 with v = x -- the UAQ-folded master weights W' of qurl_prepare_weights)
 * -> q4 [R, K/2], sblk [R, K/16], g [R], densely packed.  R = 0 is valid.
 * One kernel launch.  Errors: INVALID_ARG (NULL, K <= 0, R < 0, ldx < K,
 * non-finite pre_scale, unknown x_type), UNSUPPORTED (K % 16), ALIGNMENT (X,
 * q4 not 16-byte aligned, ldx * element size not a multiple of 16).
 *
 * qurl_nvfp4_linear: Y [M, N] (bf16, row stride ldy) =
 *   bf16_RNE(fl(fl(fp32(acc[m, n]) * gx[m]) * gw[n])),
 *   acc[m, n] = sum_k dec(x code) dec(x block scale) dec(w code) dec(w block scale),
 * accumulated in fp32 on the tensor cores (the products are exact; the
 * order of the sum is the kernel's, like the FP8 GEMM's).  Both operands
 * are widened to fp16 in the workspace (ws_bytes >= qurl_nvfp4_workspace_size
 * (M, N, K), 16-byte aligned, contents undefined between calls), then one
 * CTA-pair GEMM runs; K split (where the tiles leave SMs idle) adds a
 * reduction kernel.  3-4 kernel launches.  qurl_nvfp4_gemm_acc writes the fp32
 * sums acc [M, N] themselves (for tests).  Errors: INVALID_ARG (NULL, a
 * non-positive size, ldy < N), UNSUPPORTED (K % 16), ALIGNMENT (q4x, q4w, Y,
 * acc or the workspace not 16-byte aligned, ldy * 2 not a multiple of 16),
 * WORKSPACE (ws_bytes too small).
 */
qurl_status qurl_nvfp4_quant(const void* X, qurl_ftype x_type, int R, int K, int ldx, float pre_scale, void* q4,
                             void* sblk, float* g, qurl_stream_t stream);
size_t qurl_nvfp4_workspace_size(int M, int N, int K);
qurl_status qurl_nvfp4_linear(const void* q4x, const void* sbx, const float* gx, const void* q4w, const void* sbw,
                              const float* gw, int M, int N, int K, void* Y, int ldy, void* workspace,
                              size_t ws_bytes, qurl_stream_t stream);
qurl_status qurl_nvfp4_gemm_acc(const void* q4x, const void* sbx, const void* q4w, const void* sbw, int M, int N,
                                int K, float* acc, void* workspace, size_t ws_bytes, qurl_stream_t stream);

/* As qurl_widen_weights for 4-bit weight rows: writes their fp16 values
 * dec(code) * dec(block scale) [N, K] (2 N K bytes, 16-byte aligned, caller
 * owned) into `wide` and attaches it to q4; qurl_nvfp4_linear / _gemm_acc on
 * those weights then read it instead of widening them every call, and
 * qurl_nvfp4_quant into attached rows refreshes it.  Detach with
 * qurl_detach_wide_weights(q4) before freeing q4 or `wide`.  Errors and
 * limits as for qurl_widen_weights.  One kernel launch. */
qurl_status qurl_nvfp4_widen_weights(const void* q4, const void* sblk, int N, int K, void* wide,
                                     qurl_stream_t stream);

/*
 * FP8 key/value cache quantization ([LIMITS]: section "局限与展望" names FP8
 * KV-cache quantization as not yet optimized in the rollout engine; page 5's
 * FP8-RL entry quantizes the KV cache to FP8 beside its W8A8 layers).  The
 * granularity is this library's reading: the per-token rule applied to each
 * attention head.  For token m and KV head h of the fused qkv output
 *   key   = qkv[m, q_dim + h hd .. + hd),   value = qkv[m, q_dim + kv hd + h hd .. + hd)
 * (hd = head_dim, kv = kv_heads), each vector is quantized as one row:
 *   scale = max|x| / 448 (1 for an all-zero vector), code = e4m3_RNE_satfinite(x / scale)
 * and stored in slot s = slot_mapping[m] of the caches:
 *   k_cache[s][h][0 .. hd) bytes, k_scale[s][h] fp32 (likewise v_cache, v_scale).
 * Slots are the flattened (block, offset) positions of a paged cache, so the
 * caches are [num_slots, kv_heads, head_dim] bytes and [num_slots, kv_heads]
 * fp32.  A negative slot (a padding token) writes nothing.  Slots are read on
 * the device: one >= num_slots writes nothing and latches QURL_ERR_INVALID_ARG
 * in the device status word (qurl_check_device_status).
 *   qkv [M, ldq] bf16 (ldq >= q_dim + 2 kv hd, a multiple of 8); slot_mapping
 *   [M] int64; head_dim a multiple of 16, at most 256; q_dim a multiple of 8.
 * M = 0 is valid (nothing launched).  One kernel launch.
 */
qurl_status qurl_kv_cache_quant(const void* qkv, int M, int ldq, int q_dim, int kv_heads, int head_dim,
                                const int64_t* slot_mapping, long long num_slots, void* k_cache, float* k_scale,
                                void* v_cache, float* v_scale, qurl_stream_t stream);

/*
 * Read-back of an FP8 cache (the values an attention kernel consumes):
 *   out[i][h hd + d] = bf16_RNE(fp32(e4m3 value of cache[slots[i]][h][d]) * scale[slots[i]][h])
 * out [n, kv_heads * head_dim] bf16.  A slot outside [0, num_slots) writes
 * nothing for that row and latches QURL_ERR_INVALID_ARG in the device status
 * word.  n = 0 is valid.
 */
qurl_status qurl_kv_cache_dequant(const void* cache, const float* scale, const int64_t* slots, int n, int kv_heads,
                                  int head_dim, long long num_slots, void* out, qurl_stream_t stream);

/*
 * ACR token objective of a quantized rollout ([ACR], [OBJ]): the decoupled-PPO
 * objective with the truncated importance weight of TIS and ACR's adaptive
 * clipping range, over T token slots (the responses of a mini-batch, padded
 * slots masked out).  Per valid slot t (mask[t] != 0):
 *   w     = min(exp(logp_prox - logp_behav), C)    truncated weight pi_prox / pi_behav (= r)
 *   R     = exp(logp - logp_prox)                  pi_theta / pi_prox
 *   upper = (1 + eps) / w  if adaptive,  1 + eps otherwise (plain TIS)
 *   c     = min(max(R, 1 - eps), upper)            (the upper bound wins when below the lower)
 *   term  = w * min(R adv, c adv)
 *   dterm = d term / d logp = w adv R where R adv <= c adv, else 0 (clipped)
 * fp32 arithmetic, expf, no fused multiply-adds; padded slots give 0 and their
 * values (even NaN) are never used.  The objective is the mean term over the
 * valid slots, so its gradient with respect to logp[t] is dterm[t] / n.
 *
 *   logp, logp_prox, logp_behav  [T] fp32 log-probabilities of the sampled
 *       tokens under the policy being trained, the full-precision old actor and
 *       the quantized actor that generated them; finite, with |differences|
 *       below 80 (fp32 exp range).
 *   adv   [T] fp32 advantages (a response's advantage repeated over its tokens).
 *   mask  [T] bytes, nonzero = valid token.
 *   eps in (0, 1); C > 0; adaptive 1 (ACR) or 0 (plain TIS clipping).
 *   term, dterm  [T] fp32 (out) or NULL.
 *   stats  [QURL_ACR_NSTATS] fp64 device array (out): [0] objective (0 when no
 *       slot is valid), [1] n valid, [2] clipped fraction (R adv > c adv),
 *       [3] mean w, [4] fraction with pi_prox / pi_behav > C, [5] mean of
 *       logp_behav - logp_prox (the sample estimate of KL(pi_behav || pi_prox)).
 *       Sums: fp32 per thread, fp64 across threads in a fixed order, so the
 *       results are identical run to run.  Each thread sums about
 *       T / (4 x 256 x SMs) slots, so the sums carry a relative error of up to
 *       that many fp32 roundings of their magnitude: ~2e-6 at 4 M slots on
 *       152 SMs, ~4e-5 at 100 M.
 *   workspace  qurl_acr_workspace_size() bytes of device scratch, 16-byte
 *       aligned, ZERO-FILLED before its first use: its last 256 bytes hold a
 *       counter the call's CTAs take tickets from; the last CTA resets it, so
 *       every call leaves the workspace ready for the next one.  Calls that may
 *       run at the same time need separate workspaces.
 * Every pointer 16-byte aligned except stats (8).  T = 0 is valid (all stats 0;
 * the token pointers may then be NULL).  Errors: QURL_ERR_INVALID_ARG (NULL
 * pointer, T < 0 or >= 2^40, eps or C out of range, adaptive not 0/1),
 * QURL_ERR_WORKSPACE (ws_bytes too small), QURL_ERR_ALIGNMENT.
 * One kernel launch on `stream`.
 */
#define QURL_ACR_NSTATS 6
size_t qurl_acr_workspace_size(void);
qurl_status qurl_acr_objective(const float* logp, const float* logp_prox, const float* logp_behav, const float* adv,
                               const uint8_t* mask, long long T, float eps, float C, int adaptive, float* term,
                               float* dterm, double* stats, void* workspace, size_t ws_bytes, qurl_stream_t stream);

/* Synchronise `stream`, then return and clear the device status word of the
 * current device (QURL_OK, QURL_ERR_TIMEOUT from a kernel's bounded wait, or
 * QURL_ERR_INVALID_ARG from an index a kernel found out of range), or
 * QURL_ERR_CUDA if the synchronisation itself failed. */
qurl_status qurl_check_device_status(qurl_stream_t stream);

/* Fault injection, for testing the failure path: the next GEMM this process
 * launches (any linear / gemm_acc entry) skips the first k-block load of each
 * CTA, so a shared-memory stage is never filled -- or, in a fused decode call,
 * its first CTA does not arrive at the handoff; the waits run out after ~1 s,
 * the kernel latches QURL_ERR_TIMEOUT in the device status word, lets its own
 * copies land, frees its tensor memory and exits.  Its outputs are then
 * undefined; qurl_check_device_status() returns QURL_ERR_TIMEOUT and clears
 * the word, and later calls run normally (after a fused call, once the
 * workspace's last 256 bytes are zeroed again).  One-shot; always QURL_OK. */
qurl_status qurl_debug_inject_timeout(void);

/* Where a fused quantize -> linear entry (qurl_rmsnorm_quant_linear,
 * qurl_quant_act_linear, qurl_silu_mul_quant_linear) runs its quantizer for a
 * decode batch (M <= 256, on the plans whose GEMM kernel can take it): inside
 * the GEMM kernel (one launch: the GEMM's CTAs quantize the rows between them,
 * then meet at a grid-wide handoff) or as its own kernel just before the GEMM
 * (two launches: the GEMM starts early under programmatic dependent launch and
 * reads its weights while the quantizer runs).
 *   on = 0: always its own kernel;
 *   on = 1 (the default): inside the GEMM where that measured faster on GB300
 *     -- RMSNorm rows for INT8, and for FP8 at M <= 64; per-token rows for
 *     INT8 at M <= 64; never SiLU * up rows;
 *   on = 2: inside the GEMM wherever the plan allows.
 * All three give bit-identical outputs.  Process-wide, for calls made after it
 * returns; the previous setting goes to *previous when that is not NULL.
 * QURL_ERR_INVALID_ARG unless on is 0, 1 or 2. */
qurl_status qurl_set_fused_decode(int on, int* previous);

/* The GEMM plan the library takes for an M x N x K product of `qt` codes on a
 * GPU with `num_sms` SMs and `ws_bytes` of workspace (SIZE_MAX: as much as
 * qurl_workspace_size asks for).  Host-side only; no device is needed.  Not
 * a computation of the method: a window on the tiling, for tests and tuning.
 * The plan is the one for weights without an attached fp16 copy.
 * out[0..7]: kernel (0 = operands staged in shared memory, INT8 widened
 * there; 1 = INT8 with the widened weights in TMEM; 2 = the same on CTA
 * pairs, 256 x 256 tiles; 3 = FP8 on CTA pairs; 4 = INT8 on CTA pairs with
 * both operands widened to fp16 in the workspace), weights on the MMA M side
 * (1) or tokens (0), token tile width, token tiles, channel tiles, K splits,
 * k-blocks per split, workspace bytes the plan uses.  QURL_ERR_INVALID_ARG
 * for a null `out`, a non-positive size or SM count, or an unknown qt. */
qurl_status qurl_debug_plan(int M, int N, int K, qurl_qtype qt, int num_sms, size_t ws_bytes, long long* out);

/* The same window with the plan's schedule of units and, with `attached`
 * nonzero, the INT8 plan a call takes when the weights carry an fp16 copy
 * (qurl_widen_weights).  out[0..7] as qurl_debug_plan; out[8]: whole-K units
 * -- with K splits > 1, the first out[8] tiles (in the kernel's unit order)
 * run over all of K and write their own results, and only the remaining
 * tiles are split out[5] ways and reduced (0: every tile is split, or none
 * when out[5] = 1).  Host-side only; errors as qurl_debug_plan. */
qurl_status qurl_debug_plan_ex(int M, int N, int K, qurl_qtype qt, int num_sms, size_t ws_bytes, int attached,
                               long long* out);

/* Tensor-rate probe (not a computation of the method: it measures the
 * denominators of the roofline).  Launches, asynchronously on `stream`, a
 * kernel that issues `iters` multiply-accumulate instructions of one kind on
 * zero operands and nothing else; *ops receives the operations (2 x
 * multiply-adds) the launch performs, so that timing the launch with CUDA
 * events gives the instruction's rate on this GPU.
 *   route 0: mma.sync.m16n8k32 s8 x s8 -> s32 (warp-level integer MMA), 8 warps
 *            per CTA, four independent accumulator chains per warp;
 *   route 1: tcgen05.mma kind::f16 (fp16 x fp16 -> fp32, M 128, N 256, K 16),
 *            operands in shared memory -- the INT8 GEMMs' route, codes widened
 *            to fp16;
 *   route 2: the same with the A operand in tensor memory;
 *   route 3: tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> fp32, M 128, N 256, K 32).
 * ctas in [1, 4096] (routes 1-3: at most the SM count, one CTA per SM), iters
 * in [1, 2^24].  QURL_ERR_INVALID_ARG otherwise. */
qurl_status qurl_debug_mma_probe(int route, int ctas, int iters, double* ops, qurl_stream_t stream);

/* Static, human-readable name of a status code. */
const char* qurl_status_string(qurl_status s);

/* ABI version of this header (major * 100 + minor). */
int qurl_version(void);

/* Number of CUDA kernels this library has launched (or recorded into a graph
 * under stream capture) in this process: lets a caller count the kernels one
 * call, or one captured step, consists of.  Host-side counter; no device work. */
unsigned long long qurl_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* QURL_H_ */
