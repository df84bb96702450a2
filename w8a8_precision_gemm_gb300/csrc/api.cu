// api.cu -- the C ABI of libqurl (include/qurl.h): host-side validation,
// per-device state (SM count, status word), TMA tensor maps, and dispatch to
// the kernels.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "objective.h"
#include "qurl.h"

namespace qurl {
std::atomic<unsigned long long> g_kernel_launches{0};
}  // namespace qurl

namespace {
std::atomic<int> g_inject_timeout{0};  // one-shot test hook, see qurl_debug_inject_timeout
std::atomic<int> g_fused_decode{1};    // 0 never, 1 where it pays, 2 always: see qurl_set_fused_decode
}  // namespace

namespace {

// Per-device status word: kernels latch a bounded-wait timeout here.
__device__ int g_qurl_status;

constexpr int kMaxDevices = 64;

struct DevState {
  bool ready = false;
  int num_sms = 0;
  int* status = nullptr;  // device address of g_qurl_status on that device
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];

qurl_status cuda_fail(cudaError_t e) {
  (void)e;
  cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return QURL_ERR_CUDA;
}

// State of the current device, initialised on first use.
qurl_status device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return QURL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_qurl_status);
    if (e != cudaSuccess) return cuda_fail(e);
    d.ready = true;
  }
  *out = &d;
  return QURL_OK;
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  long long rows, cols, ld;
  int box_cols, box_rows, swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && box_cols == o.box_cols &&
           box_rows == o.box_rows && swizzle == o.swizzle;
  }
};

struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used = false;
};

constexpr int kMapCache = 128;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

// 2-D map over a row-major byte matrix [rows, cols] with row pitch ld bytes;
// boxes of box_rows x box_cols bytes; out-of-range rows/columns read as 0.
qurl_status byte_map(const void* ptr, long long rows, long long cols, long long ld, int box_cols, int box_rows,
                     bool swizzle128, CUtensorMap* out) {
  const MapKey key{ptr, rows, cols, ld, box_cols, box_rows, swizzle128 ? 1 : 0};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry& e : g_maps)
      if (e.used && e.key == key) {
        *out = e.map;
        return QURL_OK;
      }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return QURL_ERR_CUDA;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return QURL_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    MapEntry& e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.key = key;
    e.map = m;
    e.used = true;
  }
  *out = m;
  return QURL_OK;
}

// ------------------------------------------------------------------ validation

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_qt(int qt) { return qt == QURL_INT8 || qt == QURL_FP8_E4M3; }
bool valid_dim(int x) { return x > 0; }

// X-like bf16 activation [M, K] with row stride ld (elements).
qurl_status check_act(const void* X, int M, int K, int ld) {
  if (!X) return QURL_ERR_INVALID_ARG;
  if (!valid_dim(M) || !valid_dim(K) || ld < K) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(X) || (static_cast<long long>(ld) * 2) % 16 != 0) return QURL_ERR_ALIGNMENT;
  return QURL_OK;
}

qurl_status check_gemm(const void* Xq, const void* Wq, int M, int N, int K, int qt, const void* ws, size_t ws_bytes) {
  if (!Xq || !Wq) return QURL_ERR_INVALID_ARG;
  if (!valid_dim(M) || !valid_dim(N) || !valid_dim(K) || !valid_qt(qt)) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(Xq) || !aligned16(Wq)) return QURL_ERR_ALIGNMENT;
  if (ws_bytes > 0 && !ws) return QURL_ERR_INVALID_ARG;
  if (ws && !aligned16(ws)) return QURL_ERR_ALIGNMENT;
  return QURL_OK;
}

#define QURL_TRY(expr)                    \
  do {                                    \
    const qurl_status _s = (expr);        \
    if (_s != QURL_OK) return _s;         \
  } while (0)

#define QURL_CUDA(expr)                   \
  do {                                    \
    const cudaError_t _e = (expr);        \
    if (_e != cudaSuccess) return cuda_fail(_e); \
  } while (0)

// Where the INT8 kernels that read an fp16 copy of the activation codes find
// its per-token, per-split sums of |code| (and, for the kernel with widened
// weights, of code^2).
qurl::CodeSums code_sums(const qurl::GemmPlan& p, void* ws) {
  qurl::CodeSums c{};
  if (p.tmem_a || p.wide) {
    c.asum = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + p.asum_off);
    c.sum_len = p.kb_per_split * p.bk;
    c.nsum = p.splits;
    if (p.wide) c.qsum = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(ws) + p.qsum_off);
  }
  return c;
}

// Run the GEMM; mode bf16 -> Y, otherwise raw accumulators -> acc_out.
// Workspace layout (see plan_gemm): [fp16 copy of the activation codes (INT8
// decode)][split-K partials].
//   x16_ready: the fp16 copy is already there (a fused quantizer wrote it);
//   w_indep:   the kernel launched just before the GEMM is one of this
//              library's quantizers (or the widening kernel): it does not write
//              Wq and lets the GEMM launch only after its own wait, so every
//              earlier kernel has completed and the GEMM may load weights
//              before that kernel ends.
//   fq:        a fused entry's quantizer for the decode GEMM to run first (null:
//              the activation codes are an input), writing its code sums to fsums.
// ------------------------------------------------------------------ attached fp16 weight copies

// INT8 weight matrices whose fp16 copy (and per-channel sums of code^2) the
// caller keeps in its own buffer (qurl_widen_weights): the CTA-pair prefill
// GEMM reads it instead of widening Wq into the workspace on every call.
// Layout of an attached buffer: fp16 codes [N, K], then (256-aligned) the sums [N].
constexpr int kWideInt8 = 0;   // INT8 codes: fp16 codes, then the per-channel sums of code^2
constexpr int kWideNvfp4 = 1;  // 4-bit rows: fp16 values dec(code) * dec(block scale)
struct WideEntry {
  const void* wq = nullptr;
  int N = 0, K = 0, kind = kWideInt8;
  uint8_t* wide = nullptr;
};
constexpr int kWideSlots = 1024;
std::mutex g_wide_mu;
WideEntry g_wide[kWideSlots];

size_t wide_qn_off(int N, int K) { return (static_cast<size_t>(N) * K * 2 + 255) & ~static_cast<size_t>(255); }

uint8_t* find_wide(const void* wq, int N, int K, int kind = kWideInt8) {
  std::lock_guard<std::mutex> lock(g_wide_mu);
  for (const WideEntry& e : g_wide)
    if (e.wq == wq && e.N == N && e.K == K && e.kind == kind) return e.wide;
  return nullptr;
}

// Record (or re-point) an attachment; false when every slot is taken.
bool attach_wide(const void* wq, int N, int K, int kind, void* wide) {
  std::lock_guard<std::mutex> lock(g_wide_mu);
  WideEntry* slot = nullptr;
  for (WideEntry& e : g_wide)
    if (e.wq == wq) {
      slot = &e;
      break;
    }
  if (!slot)
    for (WideEntry& e : g_wide)
      if (!e.wq) {
        slot = &e;
        break;
      }
  if (!slot) return false;
  slot->wq = wq;
  slot->N = N;
  slot->K = K;
  slot->kind = kind;
  slot->wide = reinterpret_cast<uint8_t*>(wide);
  return true;
}

// The plan of a call: INT8 on a matrix with an attached fp16 copy (`att`)
// takes the CTA-pair plan that reads it where that pays, else the shape's plan.
qurl::GemmPlan choose_plan(int M, int N, int K, int qt, int sms, size_t ws_avail, const uint8_t* att) {
  qurl::GemmPlan p{};
  if (qt == QURL_INT8 && att && qurl::plan_attached(p, M, N, K, sms, ws_avail)) return p;
  return qurl::plan_gemm(M, N, K, qt, sms, ws_avail);
}

qurl_status run_gemm(const void* Xq, const float* sx, const void* Wq, const float* sw, int M, int N, int K, int qt,
                     void* Y, int ldy, void* acc_out, void* ws, size_t ws_bytes, cudaStream_t st,
                     bool x16_ready = false, bool w_indep = false, const qurl::FusedQuant* fq = nullptr,
                     qurl::CodeSums fsums = qurl::CodeSums{}) {
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  uint8_t* att = (qt == QURL_INT8) ? find_wide(Wq, N, K) : nullptr;
  const qurl::GemmPlan p = choose_plan(M, N, K, qt, dev->num_sms, ws ? ws_bytes : 0, att);
  const bool int8 = (qt == QURL_INT8);
  const bool split = p.splits > 1;
  uint8_t* part = reinterpret_cast<uint8_t*>(ws) + p.x16_bytes;
  const qurl::CodeSums sums = code_sums(p, ws);
  CUtensorMap ta, tb;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  uint8_t* w16 = nullptr;
  const unsigned* qn = nullptr;
  if (p.wide) {
    if (!x16_ready) QURL_CUDA(qurl::launch_i8_to_f16(Xq, ws, M, K, sums, st));
    if (att) {  // the caller's fp16 copy, kept current by qurl_widen_weights / qurl_prepare_weights
      w16 = att;
      qn = reinterpret_cast<const unsigned*>(att + wide_qn_off(N, K));
    } else {
      w16 = wsb + p.w16_off;
      qn = reinterpret_cast<const unsigned*>(wsb + p.qn_off);
      QURL_CUDA(qurl::launch_widen_weights(Wq, N, K, w16, const_cast<unsigned*>(qn), dev->num_sms, st));
    }
    w_indep = false;
    QURL_TRY(byte_map(ws, M, 2LL * K, 2LL * K, 128, 128, true, &ta));
    QURL_TRY(byte_map(w16, N, 2LL * K, 2LL * K, 128, 128, true, &tb));
  } else if (p.tmem_a) {
    if (!x16_ready) {
      QURL_CUDA(qurl::launch_i8_to_f16(Xq, ws, M, K, sums, st));
      w_indep = true;  // the widening kernel writes only the workspace
    }
    QURL_TRY(byte_map(Wq, N, K, K, 128, 128, true, &ta));
    QURL_TRY(byte_map(ws, M, 2LL * K, 2LL * K, 128, p.pair ? 64 : p.bn, true, &tb));
  } else {
    const long long a_rows = p.swap ? N : M;
    const long long b_rows = p.swap ? M : N;
    QURL_TRY(byte_map(p.swap ? Wq : Xq, a_rows, K, K, p.bk, 128, !int8, &ta));
    QURL_TRY(byte_map(p.swap ? Xq : Wq, b_rows, K, K, p.bk, p.pair ? p.bn / 2 : p.bn, !int8, &tb));
  }
  qurl::GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.num_kb = p.num_kb;
  a.kb_per_split = p.kb_per_split;
  a.sx = sx;
  a.sw = sw;
  a.Y = reinterpret_cast<__nv_bfloat16*>(Y);
  a.ldy = ldy;
  a.status = dev->status;
  a.w_prefetch = w_indep ? 1 : 0;
  a.mode = (Y && !split) ? qurl::kModeBf16 : qurl::kModeAcc;
  a.part = split ? static_cast<void*>(part) : acc_out;
  a.acc_out = acc_out;
  a.fault = g_inject_timeout.exchange(0);
  a.asum = sums.asum;
  a.qsum = sums.qsum;
  a.qn = p.wide ? qn : nullptr;
  a.scratch = (p.wide || p.tmem_a) ? reinterpret_cast<int*>(wsb + p.scratch_off) : nullptr;
  a.whole_units = p.whole_units;
  // FP8 prefill pairs whose activations do not fit in L2 beside the weights
  // (more than 48 MB of codes): token groups of about 48 MB of activation tiles
  // (256 rows x K codes), at most 16 tiles.  32B down at M = 8192 (226 MB of
  // activations, groups of 7): 655 us a call against 698, DRAM reads 1.76 GB
  // against 2.55; smaller activations keep token tile fastest over all
  // (o_proj at M = 8192, 42 MB: 127.0 us against 128.8 grouped)
  const bool big_act = static_cast<long long>(M) * K > (48LL << 20);
  a.tok_group = (p.pair && !p.swap && !p.wide && !p.tmem_a && big_act)
                    ? std::max(1, std::min(16, static_cast<int>((48LL << 20) / (256LL * K))))
                    : 0;
  if (fq) {
    a.fq = *fq;
    a.fsums = fsums;
    a.w_prefetch = 0;  // the kernel before this one may write Wq; the fused kernel loads weights after its wait
  }
  const dim3 grid(p.tiles_tok, p.tiles_ch, p.splits);
  if (p.wide)
    QURL_CUDA(qurl::launch_gemm_i8w(ta, tb, a, grid, st));
  else if (p.tmem_a && p.pair)
    QURL_CUDA(qurl::launch_gemm_i8p(ta, tb, a, grid, st));
  else if (p.tmem_a)
    QURL_CUDA(qurl::launch_gemm_i8t(p.bn, ta, tb, a, grid, st));
  else if (p.pair)
    QURL_CUDA(qurl::launch_gemm_fp8_pair(p.swap, p.bn, ta, tb, a, grid, st));
  else
    QURL_CUDA(int8 ? qurl::launch_gemm_i8(p.swap, p.bn, ta, tb, a, grid, st)
                   : qurl::launch_gemm_fp8(p.swap, p.bn, ta, tb, a, grid, st));
  if (split && a.whole_units > 0) {  // only the split tail needs reducing
    qurl::GemmArgs r = a;
    r.tiles_tok = p.tiles_tok;
    r.tiles_ch = p.tiles_ch;
    r.splits = p.splits;
    r.part = part;
    QURL_CUDA(qurl::launch_tail_reduce(int8, p.wide ? qurl::kWideTokGroup : a.tok_group, r, st));
  } else if (split) {
    QURL_CUDA(qurl::launch_splitk_reduce(qt, part, p.splits, M, N, sx, sw, Y, ldy, Y ? nullptr : acc_out,
                                         dev->num_sms, st));
  }
  return QURL_OK;
}

int device_sms() {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    sms = 160;  // no device visible: size for the largest SM count this library targets
  }
  return sms;
}

qurl_status check_nvfp4_rows(const void* q4, const void* sblk, const float* g, int R, int K) {
  if (!q4 || !sblk || !g || !valid_dim(R) || !valid_dim(K)) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(q4)) return QURL_ERR_ALIGNMENT;
  return QURL_OK;
}

// The 4-bit linear: both operands widened to fp16 in the workspace (exact),
// then the CTA-pair GEMM in fp32 accumulation, with g_x and g_w as the token
// and channel scales of its epilogue (Y), or the raw fp32 sums (acc).
qurl_status run_nvfp4(const void* q4x, const void* sbx, const float* gx, const void* q4w, const void* sbw,
                      const float* gw, int M, int N, int K, void* Y, int ldy, float* acc, void* ws, size_t ws_bytes,
                      cudaStream_t st) {
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  uint8_t* att = find_wide(q4w, N, K, kWideNvfp4);  // the caller's fp16 copy of the weights, if attached
  qurl::GemmPlan p{};
  if (!ws || !qurl::plan_nvfp4(p, M, N, K, dev->num_sms, ws_bytes, att != nullptr)) return QURL_ERR_WORKSPACE;
  if (!aligned16(ws)) return QURL_ERR_ALIGNMENT;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  const bool split = p.splits > 1;
  uint8_t* w16 = att ? att : wsb + p.w16_off;
  QURL_CUDA(qurl::launch_nvfp4_widen(q4x, sbx, M, K, ws, dev->num_sms, st));
  if (!att) QURL_CUDA(qurl::launch_nvfp4_widen(q4w, sbw, N, K, w16, dev->num_sms, st));
  CUtensorMap ta, tb;
  QURL_TRY(byte_map(ws, M, 2LL * K, 2LL * K, 128, 128, true, &ta));
  QURL_TRY(byte_map(w16, N, 2LL * K, 2LL * K, 128, 128, true, &tb));
  qurl::GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.num_kb = p.num_kb;
  a.kb_per_split = p.kb_per_split;
  a.sx = gx;
  a.sw = gw;
  a.Y = reinterpret_cast<__nv_bfloat16*>(Y);
  a.ldy = ldy;
  a.status = dev->status;
  a.w_prefetch = 0;
  a.mode = (Y && !split) ? qurl::kModeBf16 : qurl::kModeAcc;
  a.part = split ? static_cast<void*>(wsb + p.x16_bytes) : static_cast<void*>(acc);
  a.acc_out = acc;
  a.fault = g_inject_timeout.exchange(0);
  a.scratch = reinterpret_cast<int*>(wsb + p.scratch_off);
  a.float_acc = 1;
  a.whole_units = p.whole_units;
  QURL_CUDA(qurl::launch_gemm_i8w(ta, tb, a, dim3(p.tiles_tok, p.tiles_ch, p.splits), st));
  if (split && a.whole_units > 0) {  // only the split tail needs reducing
    qurl::GemmArgs r = a;
    r.tiles_tok = p.tiles_tok;
    r.tiles_ch = p.tiles_ch;
    r.splits = p.splits;
    r.part = wsb + p.x16_bytes;
    QURL_CUDA(qurl::launch_tail_reduce(false, qurl::kWideTokGroup, r, st));
  } else if (split) {
    QURL_CUDA(qurl::launch_splitk_reduce(qurl::kQFp8, wsb + p.x16_bytes, p.splits, M, N, gx, gw, Y, ldy,
                                         Y ? nullptr : acc, dev->num_sms, st));
  }
  return QURL_OK;
}

}  // namespace

namespace qurl {
size_t plain_workspace_bytes(int M, int N, int K, int qt) {
  if (!valid_dim(M) || !valid_dim(N) || !valid_dim(K) || !valid_qt(qt)) return 0;
  return plan_gemm(M, N, K, qt, device_sms(), static_cast<size_t>(-1)).ws_bytes;
}
}  // namespace qurl

extern "C" {

const char* qurl_status_string(qurl_status s) {
  switch (s) {
    case QURL_OK: return "QURL_OK";
    case QURL_ERR_INVALID_ARG: return "QURL_ERR_INVALID_ARG";
    case QURL_ERR_UNSUPPORTED: return "QURL_ERR_UNSUPPORTED";
    case QURL_ERR_ALIGNMENT: return "QURL_ERR_ALIGNMENT";
    case QURL_ERR_WORKSPACE: return "QURL_ERR_WORKSPACE";
    case QURL_ERR_CUDA: return "QURL_ERR_CUDA";
    case QURL_ERR_TIMEOUT: return "QURL_ERR_TIMEOUT";
  }
  return "QURL_ERR_UNKNOWN";
}

int qurl_version(void) { return 102; }

unsigned long long qurl_kernel_launches(void) { return qurl::g_kernel_launches.load(); }

qurl_status qurl_debug_inject_timeout(void) {
  g_inject_timeout.store(1);
  return QURL_OK;
}

qurl_status qurl_set_fused_decode(int on, int* previous) {
  if (on < 0 || on > 2) return QURL_ERR_INVALID_ARG;
  const int old = g_fused_decode.exchange(on);
  if (previous) *previous = old;
  return QURL_OK;
}

qurl_status qurl_prepare_weights(const void* W, qurl_ftype w_type, int N, int K, int ldw, const float* gamma,
                                 float s, qurl_qtype qt, void* Wq, float* sw, float* gamma_folded, float* W_scaled,
                                 qurl_stream_t stream) {
  if (!W || !Wq || !sw) return QURL_ERR_INVALID_ARG;
  if (w_type != QURL_BF16 && w_type != QURL_FP32) return QURL_ERR_INVALID_ARG;
  if (!valid_dim(N) || !valid_dim(K) || ldw < K || !valid_qt(qt)) return QURL_ERR_INVALID_ARG;
  if (!(s > 0.0f) || !std::isfinite(s)) return QURL_ERR_INVALID_ARG;
  if (gamma && !gamma_folded) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  const int esize = (w_type == QURL_FP32) ? 4 : 2;
  if (!aligned16(W) || (static_cast<long long>(ldw) * esize) % 16 != 0 || !aligned16(Wq) ||
      (W_scaled && !aligned16(W_scaled)))
    return QURL_ERR_ALIGNMENT;
  if (W_scaled && reinterpret_cast<const void*>(W_scaled) == W && !(w_type == QURL_FP32 && ldw == K))
    return QURL_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_prepare_weights(W, w_type == QURL_FP32, N, K, ldw, gamma, s, qt, Wq, sw, gamma_folded,
                                         W_scaled, reinterpret_cast<cudaStream_t>(stream)));
  // new codes in an attached INT8 matrix: refresh its fp16 copy (the next kernel in the stream)
  if (uint8_t* att = (qt == QURL_INT8) ? find_wide(Wq, N, K) : nullptr)
    QURL_CUDA(qurl::launch_widen_weights(Wq, N, K, att, reinterpret_cast<unsigned*>(att + wide_qn_off(N, K)),
                                         dev->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_quant_act(const void* X, int M, int K, int ldx, float pre_scale, qurl_qtype qt, void* Xq,
                           float* sx, qurl_stream_t stream) {
  QURL_TRY(check_act(X, M, K, ldx));
  if (!Xq || !sx || !valid_qt(qt) || !std::isfinite(pre_scale)) return QURL_ERR_INVALID_ARG;
  if (!aligned16(Xq)) return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_quant_act(X, M, K, ldx, pre_scale, qt, Xq, sx, nullptr, qurl::CodeSums{},
                                   reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_rmsnorm_quant(const void* X, int M, int K, int ldx, const float* gamma_folded, float eps,
                               qurl_qtype qt, void* Xq, float* sx, float* ms_out, qurl_stream_t stream) {
  QURL_TRY(check_act(X, M, K, ldx));
  if (!gamma_folded || !Xq || !sx || !valid_qt(qt) || !(eps >= 0.0f) || !std::isfinite(eps))
    return QURL_ERR_INVALID_ARG;
  if (!aligned16(Xq) || !aligned16(gamma_folded)) return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_rmsnorm_quant(X, M, K, ldx, gamma_folded, eps, qt, Xq, sx, ms_out, nullptr,
                                       qurl::CodeSums{},
                                       reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_silu_mul_quant(const void* GU, int M, int I, int ldgu, float pre_scale, qurl_qtype qt, void* Xq,
                                float* sx, float* h_out, qurl_stream_t stream) {
  if (!GU || !Xq || !sx || !valid_qt(qt) || !std::isfinite(pre_scale)) return QURL_ERR_INVALID_ARG;
  if (!valid_dim(M) || !valid_dim(I) || ldgu < 2LL * I) return QURL_ERR_INVALID_ARG;
  if (I % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(GU) || (static_cast<long long>(ldgu) * 2) % 16 != 0 || !aligned16(Xq) ||
      (h_out && !aligned16(h_out)))
    return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_silu_mul_quant(GU, M, I, ldgu, pre_scale, qt, Xq, sx, h_out, nullptr,
                                        qurl::CodeSums{}, dev->status,
                                        reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_debug_mma_probe(int route, int ctas, int iters, double* ops, qurl_stream_t stream) {
  if (route < 0 || route > 3 || ctas < 1 || ctas > 4096 || iters < 1 || iters > (1 << 24) || !ops)
    return QURL_ERR_INVALID_ARG;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  if (route > 0 && ctas > dev->num_sms) return QURL_ERR_INVALID_ARG;  // one CTA per SM
  QURL_CUDA(qurl::launch_probe(route, ctas, iters, dev->status, reinterpret_cast<cudaStream_t>(stream)));
  *ops = qurl::probe_ops(route, ctas, iters);
  return QURL_OK;
}

qurl_status qurl_debug_plan(int M, int N, int K, qurl_qtype qt, int num_sms, size_t ws_bytes, long long* out) {
  if (!out || !valid_dim(M) || !valid_dim(N) || !valid_dim(K) || !valid_qt(qt) || num_sms <= 0)
    return QURL_ERR_INVALID_ARG;
  const qurl::GemmPlan p = qurl::plan_gemm(M, N, K, qt, num_sms, ws_bytes);
  out[0] = p.wide ? 4 : p.tmem_a ? (p.pair ? 2 : 1) : (p.pair ? 3 : 0);
  out[1] = p.swap ? 1 : 0;
  out[2] = p.bn;
  out[3] = p.tiles_tok;
  out[4] = p.tiles_ch;
  out[5] = p.splits;
  out[6] = p.kb_per_split;
  out[7] = static_cast<long long>(p.ws_bytes);
  return QURL_OK;
}

qurl_status qurl_debug_plan_ex(int M, int N, int K, qurl_qtype qt, int num_sms, size_t ws_bytes, int attached,
                               long long* out) {
  if (!out || !valid_dim(M) || !valid_dim(N) || !valid_dim(K) || !valid_qt(qt) || num_sms <= 0)
    return QURL_ERR_INVALID_ARG;
  qurl::GemmPlan p{};
  if (!(attached && qt == QURL_INT8 && qurl::plan_attached(p, M, N, K, num_sms, ws_bytes)))
    p = qurl::plan_gemm(M, N, K, qt, num_sms, ws_bytes);
  out[0] = p.wide ? 4 : p.tmem_a ? (p.pair ? 2 : 1) : (p.pair ? 3 : 0);
  out[1] = p.swap ? 1 : 0;
  out[2] = p.bn;
  out[3] = p.tiles_tok;
  out[4] = p.tiles_ch;
  out[5] = p.splits;
  out[6] = p.kb_per_split;
  out[7] = static_cast<long long>(p.ws_bytes);
  out[8] = p.whole_units;
  return QURL_OK;
}

size_t qurl_workspace_size(int M, int N, int K, qurl_qtype qt) {
  if (!valid_dim(M) || !valid_dim(N) || !valid_dim(K) || !valid_qt(qt)) return 0;
  int sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    sms = 160;  // no device visible: size for the largest SM count this library targets
  }
  size_t bytes = qurl::plan_gemm(M, N, K, qt, sms, static_cast<size_t>(-1)).ws_bytes;
  qurl::GemmPlan a{};
  if (qt == QURL_INT8 && qurl::plan_attached(a, M, N, K, sms, static_cast<size_t>(-1)))
    bytes = std::max(bytes, a.ws_bytes);  // enough for the plan of a matrix with an attached fp16 copy too
  return bytes;
}

qurl_status qurl_w8a8_linear(const void* Xq, const float* sx, const void* Wq, const float* sw, int M, int N, int K,
                             qurl_qtype qt, void* Y, int ldy, void* workspace, size_t ws_bytes,
                             qurl_stream_t stream) {
  QURL_TRY(check_gemm(Xq, Wq, M, N, K, qt, workspace, ws_bytes));
  if (!sx || !sw || !Y || ldy < N) return QURL_ERR_INVALID_ARG;
  if (!aligned16(Y) || (static_cast<long long>(ldy) * 2) % 16 != 0) return QURL_ERR_ALIGNMENT;
  return run_gemm(Xq, sx, Wq, sw, M, N, K, qt, Y, ldy, nullptr, workspace, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

qurl_status qurl_w8a8_gemm_acc(const void* Xq, const void* Wq, int M, int N, int K, qurl_qtype qt, void* acc,
                               void* workspace, size_t ws_bytes, qurl_stream_t stream) {
  QURL_TRY(check_gemm(Xq, Wq, M, N, K, qt, workspace, ws_bytes));
  if (!acc) return QURL_ERR_INVALID_ARG;
  if (!aligned16(acc)) return QURL_ERR_ALIGNMENT;
  return run_gemm(Xq, nullptr, Wq, nullptr, M, N, K, qt, nullptr, N, acc, workspace, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

// Where the GEMM plan reads an fp16 copy of the INT8 codes (and their
// per-token sums of |code|) from the workspace, the fused quantizer writes
// them there directly.
struct FusedAct {
  void* x16 = nullptr;
  qurl::CodeSums sums{};
  bool in_gemm = false;      // the GEMM kernel runs the quantizer itself
  unsigned* sync = nullptr;  // its handoff counters (the workspace's last bytes)
};

// Whether the GEMM kernel's own CTAs quantize a decode batch faster than a
// quantizer kernel launched before the GEMM (which overlaps the GEMM's weight
// prefetch).  Measured on GB300 for the 7B- and 32B-class chains at M = 64 and
// 256: RMSNorm rows pay for INT8 at both sizes and for FP8 at M = 64 (1-5 us
// per call); per-token rows pay for INT8 at M = 64; SiLU * up rows, whose
// intermediate-size rows leave one CTA per row with 19-28 k values to
// transform, never do (up to 2.3x slower at M = 256).
bool in_gemm_pays(int kind, int qt, int M) {
  if (kind == qurl::kFuseRmsNorm) return qt == QURL_INT8 || M <= 64;
  if (kind == qurl::kFuseQuant) return qt == QURL_INT8 && M <= 64;
  return false;
}

FusedAct fused_x16(int kind, const void* Wq, int M, int N, int K, int qt, void* ws, size_t ws_bytes) {
  FusedAct f;
  DevState* dev = nullptr;
  if (device_state(&dev) != QURL_OK) return f;
  const qurl::GemmPlan p = choose_plan(M, N, K, qt, dev->num_sms, ws ? ws_bytes : 0,
                                       qt == QURL_INT8 ? find_wide(Wq, N, K) : nullptr);
  if (p.tmem_a || p.wide) {
    f.x16 = ws;
    f.sums = code_sums(p, ws);
  }
  // decode plans whose GEMM kernel can run the quantizer itself: the INT8
  // kernel with the widened weights in TMEM (single CTA) and the FP8 decode
  // kernels
  const int mode = g_fused_decode.load(std::memory_order_relaxed);
  f.in_gemm = mode != 0 && (mode == 2 || in_gemm_pays(kind, qt, M)) && ws != nullptr && ws_bytes >= p.ws_bytes &&
              M <= 256 && p.swap && !p.wide && (qt == QURL_INT8 ? (p.tmem_a && !p.pair) : true);
  if (f.in_gemm)
    f.sync = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(ws) +
                                         ((ws_bytes - qurl::kSyncBytes) & ~static_cast<size_t>(15)));
  return f;
}

// A fused entry as one GEMM kernel that quantizes its input rows first (plus
// the split-K reduction where K is split).
qurl_status run_fused(const FusedAct& f, int kind, const void* X, int ldx, const float* gamma, float eps, float pre,
                      const void* Wq, const float* sw, int M, int N, int K, int qt, void* Y, int ldy, void* Xq,
                      float* sx, void* ws, size_t ws_bytes, cudaStream_t st) {
  qurl::FusedQuant fq{};
  fq.kind = kind;
  fq.X = X;
  fq.ldx = ldx;
  fq.gamma = gamma;
  fq.eps = eps;
  fq.pre = pre;
  fq.Xq = Xq;
  fq.sx = sx;
  fq.x16 = f.x16;
  fq.sync = f.sync;
  return run_gemm(Xq, sx, Wq, sw, M, N, K, qt, Y, ldy, nullptr, ws, ws_bytes, st, true, false, &fq, f.sums);
}

qurl_status check_fused_out(const void* Wq, const float* sw, int M, int N, int K, int qt, void* Y, int ldy,
                            const void* Xq_scratch, const float* sx_scratch, const void* ws, size_t ws_bytes) {
  QURL_TRY(check_gemm(Xq_scratch, Wq, M, N, K, qt, ws, ws_bytes));
  if (!sw || !Y || !sx_scratch || ldy < N) return QURL_ERR_INVALID_ARG;
  if (!aligned16(Y) || (static_cast<long long>(ldy) * 2) % 16 != 0) return QURL_ERR_ALIGNMENT;
  return QURL_OK;
}

qurl_status qurl_rmsnorm_quant_linear(const void* X, int ldx, const float* gamma_folded, float eps, const void* Wq,
                                      const float* sw, int M, int N, int K, qurl_qtype qt, void* Y, int ldy,
                                      void* Xq_scratch, float* sx_scratch, void* workspace, size_t ws_bytes,
                                      qurl_stream_t stream) {
  QURL_TRY(check_act(X, M, K, ldx));
  QURL_TRY(check_fused_out(Wq, sw, M, N, K, qt, Y, ldy, Xq_scratch, sx_scratch, workspace, ws_bytes));
  if (!gamma_folded || !(eps >= 0.0f) || !std::isfinite(eps)) return QURL_ERR_INVALID_ARG;
  if (!aligned16(gamma_folded)) return QURL_ERR_ALIGNMENT;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const FusedAct f = fused_x16(qurl::kFuseRmsNorm, Wq, M, N, K, qt, workspace, ws_bytes);
  if (f.in_gemm)
    return run_fused(f, qurl::kFuseRmsNorm, X, ldx, gamma_folded, eps, 1.0f, Wq, sw, M, N, K, qt, Y, ldy, Xq_scratch,
                     sx_scratch, workspace, ws_bytes, st);
  QURL_CUDA(qurl::launch_rmsnorm_quant(X, M, K, ldx, gamma_folded, eps, qt, Xq_scratch, sx_scratch, nullptr, f.x16,
                                       f.sums, st));
  return run_gemm(Xq_scratch, sx_scratch, Wq, sw, M, N, K, qt, Y, ldy, nullptr, workspace, ws_bytes, st,
                  f.x16 != nullptr, true);
}

qurl_status qurl_quant_act_linear(const void* X, int ldx, float pre_scale, const void* Wq, const float* sw, int M,
                                  int N, int K, qurl_qtype qt, void* Y, int ldy, void* Xq_scratch, float* sx_scratch,
                                  void* workspace, size_t ws_bytes, qurl_stream_t stream) {
  QURL_TRY(check_act(X, M, K, ldx));
  QURL_TRY(check_fused_out(Wq, sw, M, N, K, qt, Y, ldy, Xq_scratch, sx_scratch, workspace, ws_bytes));
  if (!std::isfinite(pre_scale)) return QURL_ERR_INVALID_ARG;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const FusedAct f = fused_x16(qurl::kFuseQuant, Wq, M, N, K, qt, workspace, ws_bytes);
  if (f.in_gemm)
    return run_fused(f, qurl::kFuseQuant, X, ldx, nullptr, 0.0f, pre_scale, Wq, sw, M, N, K, qt, Y, ldy, Xq_scratch,
                     sx_scratch, workspace, ws_bytes, st);
  QURL_CUDA(qurl::launch_quant_act(X, M, K, ldx, pre_scale, qt, Xq_scratch, sx_scratch, f.x16, f.sums, st));
  return run_gemm(Xq_scratch, sx_scratch, Wq, sw, M, N, K, qt, Y, ldy, nullptr, workspace, ws_bytes, st,
                  f.x16 != nullptr, true);
}

qurl_status qurl_silu_mul_quant_linear(const void* GU, int ldgu, float pre_scale, const void* Wq, const float* sw,
                                       int M, int N, int I, qurl_qtype qt, void* Y, int ldy, void* Xq_scratch,
                                       float* sx_scratch, void* workspace, size_t ws_bytes, qurl_stream_t stream) {
  if (!GU || !valid_dim(M) || !valid_dim(I) || ldgu < 2LL * I || !std::isfinite(pre_scale))
    return QURL_ERR_INVALID_ARG;
  if (I % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(GU) || (static_cast<long long>(ldgu) * 2) % 16 != 0) return QURL_ERR_ALIGNMENT;
  QURL_TRY(check_fused_out(Wq, sw, M, N, I, qt, Y, ldy, Xq_scratch, sx_scratch, workspace, ws_bytes));
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const FusedAct f = fused_x16(qurl::kFuseSiluMul, Wq, M, N, I, qt, workspace, ws_bytes);
  if (f.in_gemm)
    return run_fused(f, qurl::kFuseSiluMul, GU, ldgu, nullptr, 0.0f, pre_scale, Wq, sw, M, N, I, qt, Y, ldy,
                     Xq_scratch, sx_scratch, workspace, ws_bytes, st);
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_silu_mul_quant(GU, M, I, ldgu, pre_scale, qt, Xq_scratch, sx_scratch, nullptr, f.x16,
                                        f.sums, dev->status, st));
  return run_gemm(Xq_scratch, sx_scratch, Wq, sw, M, N, I, qt, Y, ldy, nullptr, workspace, ws_bytes, st,
                  f.x16 != nullptr, true);
}

qurl_status qurl_count_diff(const void* a, const void* b, size_t n, unsigned long long* count,
                            qurl_stream_t stream) {
  if (!a || !b || !count) return QURL_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || (reinterpret_cast<uintptr_t>(count) & 7u) != 0) return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_count_diff(a, b, n, count, dev->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

size_t qurl_wide_weights_size(int N, int K) {
  if (!valid_dim(N) || !valid_dim(K)) return 0;
  return wide_qn_off(N, K) + ((static_cast<size_t>(N) * 4 + 255) & ~static_cast<size_t>(255));
}

qurl_status qurl_widen_weights(const void* Wq, int N, int K, void* wide, qurl_stream_t stream) {
  if (!Wq || !wide || !valid_dim(N) || !valid_dim(K)) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(Wq) || !aligned16(wide)) return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  if (!attach_wide(Wq, N, K, kWideInt8, wide)) return QURL_ERR_UNSUPPORTED;  // every slot taken
  uint8_t* w = reinterpret_cast<uint8_t*>(wide);
  QURL_CUDA(qurl::launch_widen_weights(Wq, N, K, w, reinterpret_cast<unsigned*>(w + wide_qn_off(N, K)),
                                       dev->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_detach_wide_weights(const void* Wq) {
  if (!Wq) return QURL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_wide_mu);
  for (WideEntry& e : g_wide)
    if (e.wq == Wq) e = WideEntry{};
  return QURL_OK;
}

qurl_status qurl_nvfp4_quant(const void* X, qurl_ftype x_type, int R, int K, int ldx, float pre_scale, void* q4,
                             void* sblk, float* g, qurl_stream_t stream) {
  if (!X || !q4 || !sblk || !g || R < 0 || !valid_dim(K) || ldx < K || !std::isfinite(pre_scale))
    return QURL_ERR_INVALID_ARG;
  if (x_type != QURL_BF16 && x_type != QURL_FP32) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  const int esize = (x_type == QURL_FP32) ? 4 : 2;
  if (!aligned16(X) || (static_cast<long long>(ldx) * esize) % 16 != 0 || !aligned16(q4)) return QURL_ERR_ALIGNMENT;
  if (R == 0) return QURL_OK;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_nvfp4_quant(X, x_type == QURL_FP32, R, K, ldx, pre_scale, q4, sblk, g,
                                     reinterpret_cast<cudaStream_t>(stream)));
  // new codes in attached rows: refresh their fp16 copy (the next kernel in the stream)
  if (uint8_t* att = find_wide(q4, R, K, kWideNvfp4))
    QURL_CUDA(qurl::launch_nvfp4_widen(q4, sblk, R, K, att, dev->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_nvfp4_widen_weights(const void* q4, const void* sblk, int N, int K, void* wide,
                                     qurl_stream_t stream) {
  if (!q4 || !sblk || !wide || !valid_dim(N) || !valid_dim(K)) return QURL_ERR_INVALID_ARG;
  if (K % 16 != 0) return QURL_ERR_UNSUPPORTED;
  if (!aligned16(q4) || !aligned16(wide)) return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  if (!attach_wide(q4, N, K, kWideNvfp4, wide)) return QURL_ERR_UNSUPPORTED;
  QURL_CUDA(qurl::launch_nvfp4_widen(q4, sblk, N, K, wide, dev->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

size_t qurl_nvfp4_workspace_size(int M, int N, int K) {
  if (!valid_dim(M) || !valid_dim(N) || !valid_dim(K)) return 0;
  qurl::GemmPlan p{};
  qurl::plan_nvfp4(p, M, N, K, device_sms(), static_cast<size_t>(-1));
  return p.ws_bytes;
}

qurl_status qurl_nvfp4_linear(const void* q4x, const void* sbx, const float* gx, const void* q4w, const void* sbw,
                              const float* gw, int M, int N, int K, void* Y, int ldy, void* workspace,
                              size_t ws_bytes, qurl_stream_t stream) {
  QURL_TRY(check_nvfp4_rows(q4x, sbx, gx, M, K));
  QURL_TRY(check_nvfp4_rows(q4w, sbw, gw, N, K));
  if (!Y || ldy < N) return QURL_ERR_INVALID_ARG;
  if (!aligned16(Y) || (static_cast<long long>(ldy) * 2) % 16 != 0) return QURL_ERR_ALIGNMENT;
  return run_nvfp4(q4x, sbx, gx, q4w, sbw, gw, M, N, K, Y, ldy, nullptr, workspace, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

qurl_status qurl_nvfp4_gemm_acc(const void* q4x, const void* sbx, const void* q4w, const void* sbw, int M, int N,
                                int K, float* acc, void* workspace, size_t ws_bytes, qurl_stream_t stream) {
  static const float one = 1.0f;
  QURL_TRY(check_nvfp4_rows(q4x, sbx, &one, M, K));
  QURL_TRY(check_nvfp4_rows(q4w, sbw, &one, N, K));
  if (!acc) return QURL_ERR_INVALID_ARG;
  if (!aligned16(acc)) return QURL_ERR_ALIGNMENT;
  return run_nvfp4(q4x, sbx, nullptr, q4w, sbw, nullptr, M, N, K, nullptr, N, acc, workspace, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

qurl_status qurl_kv_cache_quant(const void* qkv, int M, int ldq, int q_dim, int kv_heads, int head_dim,
                                const int64_t* slot_mapping, long long num_slots, void* k_cache, float* k_scale,
                                void* v_cache, float* v_scale, qurl_stream_t stream) {
  if (M < 0 || q_dim < 0 || kv_heads <= 0 || head_dim <= 0 || num_slots < 0) return QURL_ERR_INVALID_ARG;
  if (head_dim % 16 != 0 || head_dim > 256 || q_dim % 8 != 0) return QURL_ERR_UNSUPPORTED;
  if (static_cast<long long>(ldq) < static_cast<long long>(q_dim) + 2LL * kv_heads * head_dim)
    return QURL_ERR_INVALID_ARG;
  if (M == 0) return QURL_OK;
  if (!qkv || !slot_mapping || !k_cache || !k_scale || !v_cache || !v_scale) return QURL_ERR_INVALID_ARG;
  if (!aligned16(qkv) || (static_cast<long long>(ldq) * 2) % 16 != 0 || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0 || (reinterpret_cast<uintptr_t>(k_scale) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(v_scale) & 3u) != 0)
    return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_kv_cache_quant(qkv, M, ldq, q_dim, kv_heads, head_dim,
                                        reinterpret_cast<const long long*>(slot_mapping), num_slots, k_cache, k_scale,
                                        v_cache, v_scale, dev->status, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_kv_cache_dequant(const void* cache, const float* scale, const int64_t* slots, int n, int kv_heads,
                                  int head_dim, long long num_slots, void* out, qurl_stream_t stream) {
  if (n < 0 || kv_heads <= 0 || head_dim <= 0 || num_slots < 0) return QURL_ERR_INVALID_ARG;
  if (head_dim % 16 != 0 || head_dim > 256) return QURL_ERR_UNSUPPORTED;
  if (n == 0) return QURL_OK;
  if (!cache || !scale || !slots || !out) return QURL_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(out) || (reinterpret_cast<uintptr_t>(slots) & 7u) != 0 ||
      (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
    return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_kv_cache_dequant(cache, scale, reinterpret_cast<const long long*>(slots), n, kv_heads,
                                          head_dim, num_slots, out, dev->status,
                                          reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

size_t qurl_acr_workspace_size(void) { return qurl::kAcrWorkspaceBytes; }

qurl_status qurl_acr_objective(const float* logp, const float* logp_prox, const float* logp_behav, const float* adv,
                               const uint8_t* mask, long long T, float eps, float C, int adaptive, float* term,
                               float* dterm, double* stats, void* workspace, size_t ws_bytes, qurl_stream_t stream) {
  if (!stats || !workspace || T < 0 || T >= (1LL << 40)) return QURL_ERR_INVALID_ARG;
  if (T > 0 && (!logp || !logp_prox || !logp_behav || !adv || !mask)) return QURL_ERR_INVALID_ARG;
  if (!(eps > 0.f && eps < 1.f) || !(C > 0.f && C <= 3.0e38f) || (adaptive != 0 && adaptive != 1))
    return QURL_ERR_INVALID_ARG;
  if (ws_bytes < qurl::kAcrWorkspaceBytes) return QURL_ERR_WORKSPACE;
  if (!aligned16(logp) || !aligned16(logp_prox) || !aligned16(logp_behav) || !aligned16(adv) || !aligned16(mask) ||
      (term && !aligned16(term)) || (dterm && !aligned16(dterm)) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(stats) & 7u) != 0)
    return QURL_ERR_ALIGNMENT;
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(qurl::launch_acr_objective(logp, logp_prox, logp_behav, adv, mask, T, eps, C, adaptive, term, dterm, stats,
                                       workspace, dev->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QURL_OK;
}

qurl_status qurl_check_device_status(qurl_stream_t stream) {
  DevState* dev = nullptr;
  QURL_TRY(device_state(&dev));
  QURL_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int v = 0;
  QURL_CUDA(cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (v != 0) {
    const int zero = 0;
    QURL_CUDA(cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice));
    return v == qurl::kDevTimeout ? QURL_ERR_TIMEOUT : v == qurl::kDevBadIndex ? QURL_ERR_INVALID_ARG : QURL_ERR_CUDA;
  }
  return QURL_OK;
}

}  // extern "C"
