/*
 * qurl_oracle.c -- plain, slow CPU oracle of the W8A8 quantized-rollout linear
 * layer (QuRL).  TEST INFRASTRUCTURE ONLY: nothing on the product path links,
 * loads or calls this file.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark use it.
 *
 * It shares no code, header, table or helper with the CUDA library.  Every
 * function states the passage of the source pages it restates:
 *
 *   [NOTES]  Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning
 *            with Quantized Rollout".
 *     [NOTES/UAQ]   section "方法详解 > 关键设计 > 更新感知量化 (UAQ)":
 *                   W X = (W/s)(s X); s applied column-wise to W and row-wise
 *                   to the preceding activation, foldable into the norm gain.
 *     [NOTES/LOSS]  section "损失函数 / 训练策略": per-channel weight
 *                   quantization + per-token activation quantization, INT8 or
 *                   FP8, UAQ factor s = 1.5.
 *     [NOTES/SYS]   section "系统集成与工程实现": UAQ is a one-time weight
 *                   preprocessing; the rollout runs INT8/FP8 matmul kernels.
 *     [NOTES/FRAME] section "方法详解 > 整体框架": step (1) quantizes theta_old
 *                   for every rollout.
 *     [NOTES/LIMITS] section "局限与展望": FP8 KV-cache quantization is named
 *                   as not yet optimized in the rollout engine (with page 5's
 *                   FP8-RL entry, which quantizes the KV cache to FP8).
 *     [NOTES/LIMITS/4BIT] the same section: 4-bit quantization would speed
 *                   the rollout up further but was not explored; page 5 (the
 *                   fugumt summary of the QuRL paper, related-papers list,
 *                   QeRL entry) pairs RL rollout with NVFP4 quantization.
 *     [NOTES/ACR]   section "方法详解 > 关键设计 > 自适应裁剪范围 (ACR)": the
 *                   decoupled-PPO objective of the quantized rollout, with the
 *                   truncated importance weight min(pi_prox / pi_behav, C) and
 *                   the clipping range [1 - eps, (1 + eps) / r]; section
 *                   "损失函数 / 训练策略": the GRPO/DAPO decoupled variant.
 *
 * Readings where the pages are silent (symmetric absmax scaling, round to
 * nearest even, IEEE division, saturating clamp, zero rows, RMSNorm epsilon,
 * epilogue order) are listed in the design notes of the repository; each is
 * restated where it is used below.
 *
 * Precision: every decision that produces an integer code is taken in fp32,
 * the precision the quantized model stores its scales in; GEMM accumulations
 * are exact (int64 for INT8, fp64 for FP8 -- every e4m3 x e4m3 product is a
 * multiple of 2^-18 below 2^18, so a sum of up to 2^33 / 2^18 terms is exact in
 * the 53-bit fp64 significand); the RMSNorm mean of squares is fp64.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread (no
 * fast-math; no contraction, so x86-64 and aarch64 give identical bits).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_INT8 0
#define ORC_FP8_E4M3 1

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_OVERFLOW 2

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float v) {
    uint32_t b;
    memcpy(&b, &v, 4);
    return b;
}

static float f32_from_bits(uint32_t b) {
    float v;
    memcpy(&v, &b, 4);
    return v;
}

/* Round a double to the nearest integer, ties to even (the IEEE default
 * rounding direction), written out rather than taken from the C library. */
static double round_half_even(double r) {
    double fl = floor(r);
    double diff = r - fl; /* exact: r and fl share the binade or fl == 0 */
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    /* a tie: pick the even neighbour */
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/*
 * OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, so the largest finite magnitude is
 * S.1111.110 = 1.75 * 2^8 = 448.  Exponent field 0 holds subnormals m/8 * 2^-6.
 *
 * Encode: round |v| to the nearest value of that grid, ties to even, keep the
 * sign (also of zero), and saturate every magnitude >= 448 to 448 ("satfinite":
 * the next grid point above 448 would be 480, and the midpoint 464 ties to the
 * even mantissa 110, i.e. 448, so every finite |v| >= 448 ends at 448).
 */
uint8_t orc_e4m3_encode(float v) {
    uint32_t b = f32_bits(v);
    uint8_t sign = (uint8_t)((b >> 24) & 0x80u);
    uint32_t mag = b & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return (uint8_t)(sign | 0x7F); /* NaN */
    double a = (double)f32_from_bits(mag);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* spacing of the e4m3 grid around a */
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9); /* subnormal spacing */
    } else {
        int ex;
        frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
        quantum = ldexp(1.0, (ex - 1) - 3);
    }
    double n = round_half_even(a / quantum); /* a / quantum is exact */
    double r = n * quantum;                  /* the rounded magnitude, <= 448 */
    uint8_t code;
    if (r < ldexp(1.0, -6)) {
        code = (uint8_t)n; /* subnormal: exponent field 0, mantissa n in 0..7 */
    } else {
        int ex;
        double f = frexp(r, &ex); /* r = f * 2^ex, f in [0.5, 1) */
        int e = ex - 1;           /* r = (2f) * 2^e, 2f in [1, 2) */
        int m = (int)((2.0 * f - 1.0) * 8.0);
        code = (uint8_t)(((e + 7) << 3) | m);
    }
    return (uint8_t)(sign | code);
}

/* Exact value of an e4m3 code (NaN for S.1111.111). */
double orc_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * bfloat16 = the upper 16 bits of an fp32.  Round to nearest even on the 16
 * discarded bits; a carry out of the mantissa moves into the exponent (and
 * from the largest finite value into infinity), as IEEE rounding does.
 */
uint16_t orc_bf16_encode(float v) {
    uint32_t b = f32_bits(v);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((b >> 16) | 0x0040u); /* quiet NaN */
    uint32_t keep = b >> 16;
    uint32_t rest = b & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

float orc_bf16_decode(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

void orc_e4m3_encode_array(const float* v, size_t n, uint8_t* out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_bf16_encode_array(const float* v, size_t n, uint16_t* out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_bf16_encode(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Symmetric absmax quantization of one row [NOTES/LOSS]                     */
/* ------------------------------------------------------------------------ */

/*
 * One row (an output channel of W, or a token of X) is quantized with its own
 * scale:  a = max_k |v_k|;  scale = a / qmax (fp32, IEEE division);
 * code_k = clamp(RNE(v_k / scale), -127, 127) for INT8, or
 * code_k = e4m3_RNE_satfinite(v_k / scale) for FP8 (qmax = 448).
 * A row that is all zero gets scale 1 and all-zero codes.
 */
static void quant_row(const float* v, int K, int qtype, uint8_t* q, float* scale_out) {
    float a = 0.0f;
    for (int k = 0; k < K; ++k) {
        float t = fabsf(v[k]);
        if (t > a) a = t;
    }
    float qmax = (qtype == ORC_INT8) ? 127.0f : 448.0f;
    float scale = (a == 0.0f) ? 1.0f : a / qmax;
    for (int k = 0; k < K; ++k) {
        float r = v[k] / scale;
        if (qtype == ORC_INT8) {
            double n = round_half_even((double)r);
            if (n > 127.0) n = 127.0;
            if (n < -127.0) n = -127.0;
            q[k] = (uint8_t)(int8_t)n;
        } else {
            q[k] = orc_e4m3_encode(r);
        }
    }
    *scale_out = scale;
}

int orc_quant_rows_f32(const float* V, int M, int K, int ldv, int qtype, uint8_t* q, float* scale) {
    if (!V || !q || !scale || M < 0 || K <= 0 || ldv < K) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) quant_row(V + (size_t)m * ldv, K, qtype, q + (size_t)m * K, scale + m);
    return ORC_OK;
}

/*
 * Per-token activation quantization of a bf16 activation X[M, K] (row stride
 * ldx): v = fp32(x) * pre_scale, then quant_row.  pre_scale carries the UAQ
 * factor s into an activation that has no norm to fold it into
 * [NOTES/UAQ: "row-wise on the preceding activation"]; it is 1 otherwise.
 */
int orc_quant_act(const uint16_t* X, int M, int K, int ldx, float pre_scale, int qtype, uint8_t* Xq,
                  float* sx) {
    if (!X || !Xq || !sx || M < 0 || K <= 0 || ldx < K) return ORC_ERR_ARG;
    float* v = (float*)malloc(sizeof(float) * (size_t)K);
    if (!v) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        for (int k = 0; k < K; ++k) v[k] = orc_bf16_decode(X[(size_t)m * ldx + k]) * pre_scale;
        quant_row(v, K, qtype, Xq + (size_t)m * K, sx + m);
    }
    free(v);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* UAQ fold + per-channel weight quantization [NOTES/UAQ, NOTES/LOSS, SYS]    */
/* ------------------------------------------------------------------------ */

/*
 * W[N, K] fp32 (row n = output channel, column k = input channel).
 * W'_{nk} = W_{nk} / s   (the same s on every column: the scalar reading of
 *                         "s applied column-wise to W");
 * gamma'_k = gamma_k * s (s folded into the preceding norm gain; skipped when
 *                         gamma is NULL);
 * then every row of W' is quantized on its own (per-output-channel scale sw_n).
 * With s = 1 this is the per-step re-quantization of the current weights
 * [NOTES/FRAME].  W_scaled (may be NULL) receives W' in fp32.
 */
int orc_prepare_weights(const float* W, int N, int K, int ldw, const float* gamma, float s, int qtype,
                        uint8_t* Wq, float* sw, float* gamma_folded, float* W_scaled) {
    if (!W || !Wq || !sw || N < 0 || K <= 0 || ldw < K || !(s > 0.0f)) return ORC_ERR_ARG;
    float* row = (float*)malloc(sizeof(float) * (size_t)K);
    if (!row) return ORC_ERR_ARG;
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) row[k] = W[(size_t)n * ldw + k] / s;
        if (W_scaled) memcpy(W_scaled + (size_t)n * K, row, sizeof(float) * (size_t)K);
        quant_row(row, K, qtype, Wq + (size_t)n * K, sw + n);
    }
    free(row);
    if (gamma && gamma_folded)
        for (int k = 0; k < K; ++k) gamma_folded[k] = gamma[k] * s;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm (gain already folded) -> per-token quantization                   */
/* ------------------------------------------------------------------------ */

/* Mean of squares of each bf16 row, accumulated in fp64. */
void orc_rms_ms(const uint16_t* X, int M, int K, int ldx, double* ms) {
    for (int m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
            double x = (double)orc_bf16_decode(X[(size_t)m * ldx + k]);
            acc += x * x;
        }
        ms[m] = acc / (double)K;
    }
}

/*
 * RMSNorm with gain gamma' (= gamma * s after the UAQ fold) followed by
 * per-token quantization:
 *   ms = mean_k x_k^2;  r = 1 / sqrt(fp32(ms) + eps)  (fp32, correctly rounded
 *   sqrt and division);  v_k = (x_k * r) * gamma'_k  (two fp32 products);
 *   then quant_row(v).
 * ms_given: NULL -> the oracle's own fp64 mean of squares; otherwise the
 * per-row fp32 values to use (the kernel's reduction order is its own, so the
 * codes are compared given the kernel's mean of squares).
 * v_out (may be NULL) receives v [M, K].
 */
int orc_rmsnorm_quant(const uint16_t* X, int M, int K, int ldx, const float* gamma_folded, float eps,
                      const float* ms_given, int qtype, uint8_t* Xq, float* sx, float* ms_out,
                      float* v_out) {
    if (!X || !gamma_folded || !Xq || !sx || M < 0 || K <= 0 || ldx < K) return ORC_ERR_ARG;
    float* v = (float*)malloc(sizeof(float) * (size_t)K);
    double* ms = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
    if (!v || !ms) {
        free(v);
        free(ms);
        return ORC_ERR_ARG;
    }
    orc_rms_ms(X, M, K, ldx, ms);
    for (int m = 0; m < M; ++m) {
        float msf = ms_given ? ms_given[m] : (float)ms[m];
        if (ms_out) ms_out[m] = msf;
        float den = sqrtf(msf + eps);
        float r = 1.0f / den;
        for (int k = 0; k < K; ++k) {
            float x = orc_bf16_decode(X[(size_t)m * ldx + k]);
            float xr = x * r;
            v[k] = xr * gamma_folded[k];
        }
        if (v_out) memcpy(v_out + (size_t)m * K, v, sizeof(float) * (size_t)K);
        quant_row(v, K, qtype, Xq + (size_t)m * K, sx + m);
    }
    free(v);
    free(ms);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* SiLU(gate) * up -> per-token quantization (decoder MLP between gate_up    */
/* and down; the pages are silent on it, the projection chain needs it)      */
/* ------------------------------------------------------------------------ */

/*
 * GU[M, 2I] bf16 (row stride ldgu): columns [0, I) are the gate g, [I, 2I)
 * the up projection u.  h = (g / (1 + exp(-g))) * u in fp32 (host expf),
 * v = h * pre_scale, then quant_row(v).  h_given: NULL -> compute h; else use
 * the given fp32 h (the kernel's exp differs from the host's by ulps, so codes
 * are compared given the kernel's h).  h_out may be NULL.
 */
int orc_silu_mul_quant(const uint16_t* GU, int M, int I, int ldgu, float pre_scale, const float* h_given,
                       int qtype, uint8_t* Xq, float* sx, float* h_out) {
    if (!GU || !Xq || !sx || M < 0 || I <= 0 || ldgu < 2 * I) return ORC_ERR_ARG;
    float* v = (float*)malloc(sizeof(float) * (size_t)I);
    if (!v) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        for (int i = 0; i < I; ++i) {
            float h;
            if (h_given) {
                h = h_given[(size_t)m * I + i];
            } else {
                float g = orc_bf16_decode(GU[(size_t)m * ldgu + i]);
                float u = orc_bf16_decode(GU[(size_t)m * ldgu + I + i]);
                float e = expf(-g);
                float sg = g / (1.0f + e);
                h = sg * u;
            }
            if (h_out) h_out[(size_t)m * I + i] = h;
            v[i] = h * pre_scale;
        }
        quant_row(v, I, qtype, Xq + (size_t)m * I, sx + m);
    }
    free(v);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* FP8 key/value cache quantization [NOTES/LIMITS]                           */
/* ------------------------------------------------------------------------ */

/*
 * [NOTES/LIMITS] section "局限与展望" names FP8 quantization of the KV cache
 * as what the rollout engine does not yet do well, and the FP8-RL entry of the
 * related-work list (page 5) quantizes the KV cache to FP8 beside its W8A8
 * layers.  Neither fixes the granularity; the reading taken here is the
 * method's per-token rule applied to each attention head.
 *
 * QKV[M, ldq] bf16 holds, per token, the query (q_dim columns), then the keys
 * and then the values of kv_heads heads of head_dim columns each (the fused
 * qkv projection's output).  For token m and head h, the key vector
 * k = QKV[m, q_dim + h hd .. + hd) is quantized as one row (quant_row, FP8:
 * scale = max|k| / 448, codes e4m3_RNE_satfinite(k / scale)); likewise the
 * value vector at q_dim + kv_heads hd + h hd.  The codes of token m go to slot
 * s = slot_mapping[m] of the caches: kc[s][h][0 .. hd), ks[s][h] (and vc, vs);
 * a negative slot (a padding token) writes nothing.  Slots are the flattened
 * (block, offset) positions of a paged cache.
 */
int orc_kv_cache_quant(const uint16_t* QKV, int M, int ldq, int q_dim, int kv_heads, int head_dim,
                       const int64_t* slot_mapping, uint8_t* kc, float* ks, uint8_t* vc, float* vs) {
    if (!QKV || !slot_mapping || !kc || !ks || !vc || !vs || M < 0 || q_dim < 0 || kv_heads <= 0 ||
        head_dim <= 0 || ldq < q_dim + 2 * kv_heads * head_dim)
        return ORC_ERR_ARG;
    float* v = (float*)malloc(sizeof(float) * (size_t)head_dim);
    if (!v) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        const int64_t slot = slot_mapping[m];
        if (slot < 0) continue;
        for (int part = 0; part < 2; ++part) {
            uint8_t* codes = part == 0 ? kc : vc;
            float* scales = part == 0 ? ks : vs;
            for (int h = 0; h < kv_heads; ++h) {
                const size_t col = (size_t)q_dim + (size_t)part * kv_heads * head_dim + (size_t)h * head_dim;
                for (int d = 0; d < head_dim; ++d) v[d] = orc_bf16_decode(QKV[(size_t)m * ldq + col + d]);
                const size_t at = (size_t)slot * kv_heads + h;
                quant_row(v, head_dim, ORC_FP8_E4M3, codes + at * head_dim, scales + at);
            }
        }
    }
    free(v);
    return ORC_OK;
}

/*
 * The values a cache holds, for the slots a reader gathers: out[n][h hd + d] =
 * bf16_RNE(fp32(e4m3 value of code) * scale) of slot slots[n], head h (the
 * e4m3 value is exact in fp32, so one fp32 rounding and one bf16 rounding).
 */
int orc_kv_cache_dequant(const uint8_t* cache, const float* scale, const int64_t* slots, int n, int kv_heads,
                         int head_dim, uint16_t* out) {
    if (!cache || !scale || !slots || !out || n < 0 || kv_heads <= 0 || head_dim <= 0) return ORC_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        if (slots[i] < 0) return ORC_ERR_ARG;
        for (int h = 0; h < kv_heads; ++h) {
            const size_t at = (size_t)slots[i] * kv_heads + h;
            for (int d = 0; d < head_dim; ++d) {
                const float x = (float)orc_e4m3_decode(cache[at * head_dim + d]) * scale[at];
                out[((size_t)i * kv_heads + h) * head_dim + d] = orc_bf16_encode(x);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* 8-bit GEMM (exact accumulation) and dequantizing epilogue [NOTES/SYS]     */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* Xq;
    const uint8_t* Wq;
    int M, N, K, qtype;
    int m0, m1;
    int32_t* acc_i32;
    double* acc_f64;
    int overflow;
} gemm_job;

static double e4m3_table[256];
static pthread_once_t e4m3_table_once = PTHREAD_ONCE_INIT;
static void e4m3_table_init(void) {
    for (int c = 0; c < 256; ++c) e4m3_table[c] = orc_e4m3_decode((uint8_t)c);
}

/* acc[m, n] = sum_k Xq[m, k] * Wq[n, k] over rows m0..m1 of the job. */
static void* gemm_rows(void* p) {
    gemm_job* j = (gemm_job*)p;
    const int N = j->N, K = j->K;
    for (int m = j->m0; m < j->m1; ++m) {
        const uint8_t* x = j->Xq + (size_t)m * K;
        for (int n = 0; n < N; ++n) {
            const uint8_t* w = j->Wq + (size_t)n * K;
            if (j->qtype == ORC_INT8) {
                int64_t acc = 0;
                for (int k = 0; k < K; ++k) acc += (int64_t)(int8_t)x[k] * (int64_t)(int8_t)w[k];
                if (acc > INT32_MAX || acc < INT32_MIN) j->overflow = 1;
                j->acc_i32[(size_t)m * N + n] = (int32_t)acc;
            } else {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) acc += e4m3_table[x[k]] * e4m3_table[w[k]];
                j->acc_f64[(size_t)m * N + n] = acc;
            }
        }
    }
    return NULL;
}

static int gemm_run(const uint8_t* Xq, const uint8_t* Wq, int M, int N, int K, int qtype, int32_t* acc_i32,
                    double* acc_f64, int nthreads) {
    if (!Xq || !Wq || M < 0 || N < 0 || K <= 0) return ORC_ERR_ARG;
    pthread_once(&e4m3_table_once, e4m3_table_init);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = M > 0 ? M : 1;
    gemm_job* jobs = (gemm_job*)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return ORC_ERR_ARG;
    }
    for (int t = 0; t < nthreads; ++t) {
        gemm_job* j = &jobs[t];
        j->Xq = Xq;
        j->Wq = Wq;
        j->M = M;
        j->N = N;
        j->K = K;
        j->qtype = qtype;
        j->m0 = (int)((int64_t)M * t / nthreads);
        j->m1 = (int)((int64_t)M * (t + 1) / nthreads);
        j->acc_i32 = acc_i32;
        j->acc_f64 = acc_f64;
        j->overflow = 0;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, gemm_rows, &jobs[t]);
    gemm_rows(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    int overflow = 0;
    for (int t = 0; t < nthreads; ++t) overflow |= jobs[t].overflow;
    free(jobs);
    free(th);
    return overflow ? ORC_ERR_OVERFLOW : ORC_OK;
}

/* INT8: acc = sum_k Xq*Wq in int64, stored as int32; ORC_ERR_OVERFLOW if a
 * sum leaves the int32 range. */
int orc_gemm_i8(const int8_t* Xq, const int8_t* Wq, int M, int N, int K, int32_t* acc, int nthreads) {
    if (!acc) return ORC_ERR_ARG;
    return gemm_run((const uint8_t*)Xq, (const uint8_t*)Wq, M, N, K, ORC_INT8, acc, NULL, nthreads);
}

/* FP8: acc = sum_k dec(Xq)*dec(Wq) in fp64 (exact, see the header). */
int orc_gemm_fp8(const uint8_t* Xq, const uint8_t* Wq, int M, int N, int K, double* acc, int nthreads) {
    if (!acc) return ORC_ERR_ARG;
    return gemm_run(Xq, Wq, M, N, K, ORC_FP8_E4M3, NULL, acc, nthreads);
}

/*
 * Dequantizing epilogue: y[m, n] = bf16_RNE( (fp32(acc) * sx[m]) * sw[n] ),
 * fp32 products in that order, the accumulator first rounded to fp32.
 * Y has row stride ldy.
 */
void orc_epilogue_i32(const int32_t* acc, const float* sx, const float* sw, int M, int N, uint16_t* Y, int ldy) {
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            float a = (float)acc[(size_t)m * N + n];
            float t = a * sx[m];
            float y = t * sw[n];
            Y[(size_t)m * ldy + n] = orc_bf16_encode(y);
        }
}

void orc_epilogue_f64(const double* acc, const float* sx, const float* sw, int M, int N, uint16_t* Y, int ldy) {
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            float a = (float)acc[(size_t)m * N + n];
            float t = a * sx[m];
            float y = t * sw[n];
            Y[(size_t)m * ldy + n] = orc_bf16_encode(y);
        }
}

/* ------------------------------------------------------------------------ */
/* 4-bit W4A4 variant: NVFP4 rows [NOTES/LIMITS/4BIT]                        */
/* ------------------------------------------------------------------------ */

/*
 * The pages name 4-bit quantization (NVFP4 through the QeRL entry) without
 * defining it; the reading taken is NVIDIA's published NVFP4 layout with the
 * pages' per-channel / per-token split for its second-level scale:
 *   * element codes E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa
 *     bit 0; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7;
 *   * one E4M3 scale per 16 consecutive values of a row (a block);
 *   * one fp32 scale g per row (an output channel of W, a token of X).
 * A value is dec(code) * dec(block scale) * g.
 *
 * Quantizing a row v[0..K), K a multiple of 16 (every division IEEE fp32):
 *   A = max |v|;  g = A / 2688 (6 * 448: the largest E2M1 magnitude times the
 *   largest E4M3 scale), 1 for an all-zero row;  d6 = fl(6 * g);
 *   block b: a_b = max of its |v|;  s_b = e4m3_RNE_satfinite(a_b / d6);
 *   step e_b = fl(dec(s_b) * g);  code = e2m1_RNE_satfinite(v / e_b), with the
 *   sign of v kept also where the magnitude rounds to 0 (as IEEE rounding
 *   keeps the sign of zero); every code of a block with e_b = 0 is 0.
 */
static const double e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Round to the E2M1 grid: nearest magnitude, ties to the even code (mantissa
 * bit 0), magnitudes >= 6 saturate to 6.  NaN is outside the domain (0). */
uint8_t orc_e2m1_encode(float r) {
    if (r != r) return 0;
    double a = fabs((double)r);
    int code = 7;
    for (int i = 0; i < 7; ++i) {
        double lo = e2m1_mag[i], hi = e2m1_mag[i + 1], mid = 0.5 * (lo + hi);
        if (a < hi) {
            if (a < mid) code = i;
            else if (a > mid) code = i + 1;
            else code = (i % 2 == 0) ? i : i + 1;
            break;
        }
    }
    if (a >= 6.0) code = 7;
    return (uint8_t)((signbit(r) ? 8 : 0) | code);
}

double orc_e2m1_decode(uint8_t c) {
    double m = e2m1_mag[c & 7];
    return (c & 8) ? -m : m;
}

/* One row: q4[K/2] (value 2j in the low nibble of byte j), sblk[K/16], *g. */
static void nvfp4_row(const float* v, int K, uint8_t* q4, uint8_t* sblk, float* g_out) {
    float A = 0.0f;
    for (int k = 0; k < K; ++k) {
        float t = fabsf(v[k]);
        if (t > A) A = t;
    }
    float g = (A == 0.0f) ? 1.0f : A / 2688.0f;
    float d6 = 6.0f * g;
    memset(q4, 0, (size_t)K / 2);
    for (int b = 0; b < K / 16; ++b) {
        const float* vb = v + 16 * b;
        float ab = 0.0f;
        for (int k = 0; k < 16; ++k) {
            float t = fabsf(vb[k]);
            if (t > ab) ab = t;
        }
        uint8_t s = orc_e4m3_encode(ab / d6);
        sblk[b] = s;
        float eb = (float)orc_e4m3_decode(s) * g;
        for (int k = 0; k < 16; ++k) {
            uint8_t c = (eb == 0.0f) ? 0 : orc_e2m1_encode(vb[k] / eb);
            int kk = 16 * b + k;
            q4[kk / 2] |= (uint8_t)((kk & 1) ? (c << 4) : c);
        }
    }
    *g_out = g;
}

/* Rows of fp32 values (weights: the UAQ-folded W'). */
int orc_nvfp4_quant_rows_f32(const float* V, int R, int K, int ldv, uint8_t* q4, uint8_t* sblk, float* g) {
    if (!V || !q4 || !sblk || !g || R < 0 || K <= 0 || K % 16 != 0 || ldv < K) return ORC_ERR_ARG;
    for (int r = 0; r < R; ++r)
        nvfp4_row(V + (size_t)r * ldv, K, q4 + (size_t)r * (K / 2), sblk + (size_t)r * (K / 16), g + r);
    return ORC_OK;
}

/* Rows of bf16 activations with the UAQ pre-scale: v = fl(x * pre_scale). */
int orc_nvfp4_quant_act(const uint16_t* X, int M, int K, int ldx, float pre_scale, uint8_t* q4, uint8_t* sblk,
                        float* g) {
    if (!X || !q4 || !sblk || !g || M < 0 || K <= 0 || K % 16 != 0 || ldx < K) return ORC_ERR_ARG;
    float* v = (float*)malloc(sizeof(float) * (size_t)K);
    if (!v) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        for (int k = 0; k < K; ++k) v[k] = orc_bf16_decode(X[(size_t)m * ldx + k]) * pre_scale;
        nvfp4_row(v, K, q4 + (size_t)m * (K / 2), sblk + (size_t)m * (K / 16), g + m);
    }
    free(v);
    return ORC_OK;
}

/*
 * acc[m, n] = sum_k dec(x code) dec(x block scale) dec(w code) dec(w block
 * scale), exactly: each factor dec(code) * dec(scale) is a multiple of 2^-10
 * (E2M1 values are multiples of 1/2, E4M3 values of 2^-9) of magnitude at
 * most 6 * 448, so each product is an integer multiple of 2^-20 below 2^43
 * in those units, and the sum over K < 2^20 terms fits int64.  The int64 sum
 * is converted to fp64 (exact below 2^53 units).  The row scales gx, gw
 * enter the dequantizing epilogue (orc_epilogue_f64) as sx and sw.
 */
typedef struct {
    const uint8_t *q4x, *sbx;
    const int64_t* wf; /* [N][K] weight factors in units of 2^-10 */
    int M, N, K, m0, m1;
    double* acc;
} nvfp4_job;

static int64_t nvfp4_factor(const uint8_t* q4, const uint8_t* sb, int k) {
    uint8_t c = (uint8_t)((k & 1) ? (q4[k / 2] >> 4) : (q4[k / 2] & 15));
    /* 2 dec(code) and 2^9 dec(scale) are integers */
    int64_t cv = (int64_t)(2.0 * orc_e2m1_decode(c));
    int64_t sv = (int64_t)ldexp(orc_e4m3_decode(sb[k / 16]), 9);
    return cv * sv;
}

static void* nvfp4_rows(void* p) {
    nvfp4_job* j = (nvfp4_job*)p;
    int K = j->K;
    int64_t* xf = (int64_t*)malloc(sizeof(int64_t) * (size_t)K);
    if (!xf) return (void*)1;
    for (int m = j->m0; m < j->m1; ++m) {
        for (int k = 0; k < K; ++k)
            xf[k] = nvfp4_factor(j->q4x + (size_t)m * (K / 2), j->sbx + (size_t)m * (K / 16), k);
        for (int n = 0; n < j->N; ++n) {
            int64_t s = 0;
            const int64_t* w = j->wf + (size_t)n * K;
            for (int k = 0; k < K; ++k) s += xf[k] * w[k];
            j->acc[(size_t)m * j->N + n] = ldexp((double)s, -20);
        }
    }
    free(xf);
    return NULL;
}

int orc_gemm_nvfp4(const uint8_t* q4x, const uint8_t* sbx, const uint8_t* q4w, const uint8_t* sbw, int M, int N,
                   int K, double* acc, int nthreads) {
    if (!q4x || !sbx || !q4w || !sbw || !acc || M < 0 || N < 0 || K <= 0 || K % 16 != 0 || K >= (1 << 20))
        return ORC_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = M > 0 ? M : 1;
    nvfp4_job* jobs = (nvfp4_job*)calloc((size_t)nthreads, sizeof(nvfp4_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    int64_t* wf = (int64_t*)malloc(sizeof(int64_t) * ((size_t)K * N + 1));
    if (!jobs || !th || !wf) {
        free(jobs);
        free(th);
        free(wf);
        return ORC_ERR_ARG;
    }
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            wf[(size_t)n * K + k] = nvfp4_factor(q4w + (size_t)n * (K / 2), sbw + (size_t)n * (K / 16), k);
    int rc = ORC_OK;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (nvfp4_job){q4x, sbx, wf, M, N, K, (int)((long long)M * t / nthreads),
                              (int)((long long)M * (t + 1) / nthreads), acc};
        if (pthread_create(&th[t], NULL, nvfp4_rows, &jobs[t]) != 0) {
            nvfp4_rows(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t) {
        void* r = NULL;
        if (th[t]) pthread_join(th[t], &r);
        if (r) rc = ORC_ERR_ARG;
    }
    free(jobs);
    free(th);
    free(wf);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Weight-update probe [NOTES/UAQ: error ~ |theta|/(s 2^b) shrinks by s,     */
/* update ~ s alpha G grows by s]                                            */
/* ------------------------------------------------------------------------ */

/* Number of positions where two code buffers differ. */
uint64_t orc_count_diff(const uint8_t* a, const uint8_t* b, size_t n) {
    uint64_t c = 0;
    for (size_t i = 0; i < n; ++i) c += (a[i] != b[i]);
    return c;
}

/* ------------------------------------------------------------------------ */
/* ACR token objective [NOTES/ACR]                                           */
/* ------------------------------------------------------------------------ */

#define ORC_ACR_NSTATS 6

/* The decoupled-PPO objective of a quantized rollout over T token slots.
 *
 * Per valid token (mask != 0), with the three log-probabilities of the token
 * the rollout sampled -- logp (the policy being trained, pi_theta), logp_prox
 * (the full-precision old actor, the proximal policy pi_prox) and logp_behav
 * (the quantized old actor that generated it, the behaviour policy) -- and its
 * advantage A:
 *   w     = min(pi_prox / pi_behav, C)       truncated importance weight (TIS);
 *                                            it is the scaling factor r of ACR
 *   R     = pi_theta / pi_prox               the clipping ratio
 *   upper = (1 + eps) / w   (adaptive)  or  1 + eps  (plain TIS)
 *   c     = clip(R, 1 - eps, upper) = min(max(R, 1 - eps), upper)
 *   term  = w * min(R A, c A)
 * and the objective is the token-level mean of term over the valid tokens
 * (the GRPO/DAPO decoupled variant averages over all tokens of the batch).
 *
 * dterm = d term / d logp: w A R where the unclipped product R A is the
 * minimum (dR / dlogp = R), 0 where the clipped constant c A is; the gradient
 * of the objective is dterm / n.  Masked slots: term = dterm = 0.
 *
 * stats[0] objective (0 when n = 0)      stats[3] mean w
 * stats[1] n, the number of valid tokens stats[4] fraction with pi_prox / pi_behav > C
 * stats[2] fraction clipped (R A > c A)  stats[5] mean of logp_behav - logp_prox
 * (the sample estimate of KL(pi_behav || pi_prox), tokens drawn from pi_behav).
 * Everything in fp64 from the fp32 inputs; sums in token order.
 * term, dterm: [T] or NULL. */
int orc_acr_objective(const float* logp, const float* logp_prox, const float* logp_behav, const float* adv,
                      const uint8_t* mask, int64_t T, double eps, double C, int adaptive, double* term,
                      double* dterm, double* stats) {
    if (T < 0 || !(eps > 0.0 && eps < 1.0) || !(C > 0.0) || !stats) return ORC_ERR_ARG;
    double sum_term = 0.0, sum_w = 0.0, sum_kl = 0.0;
    int64_t n = 0, clipped = 0, capped = 0;
    for (int64_t t = 0; t < T; ++t) {
        double tt = 0.0, dt = 0.0;
        if (mask[t]) {
            const double ratio_pb = exp((double)logp_prox[t] - (double)logp_behav[t]);
            const double w = ratio_pb < C ? ratio_pb : C;
            const double R = exp((double)logp[t] - (double)logp_prox[t]);
            const double lower = 1.0 - eps;
            const double upper = adaptive ? (1.0 + eps) / w : 1.0 + eps;
            double c = R > lower ? R : lower;
            if (c > upper) c = upper;
            const double A = (double)adv[t];
            const double u = R * A, v = c * A;
            if (u <= v) {
                tt = w * u;
                dt = w * A * R;
            } else {
                tt = w * v;
                ++clipped;
            }
            ++n;
            sum_term += tt;
            sum_w += w;
            capped += ratio_pb > C;
            sum_kl += (double)logp_behav[t] - (double)logp_prox[t];
        }
        if (term) term[t] = tt;
        if (dterm) dterm[t] = dt;
    }
    const double dn = (double)n;
    stats[0] = n ? sum_term / dn : 0.0;
    stats[1] = dn;
    stats[2] = n ? (double)clipped / dn : 0.0;
    stats[3] = n ? sum_w / dn : 0.0;
    stats[4] = n ? (double)capped / dn : 0.0;
    stats[5] = n ? sum_kl / dn : 0.0;
    return ORC_OK;
}
