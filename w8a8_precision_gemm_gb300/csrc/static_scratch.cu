// static_scratch.cu -- qurl_w8a8_linear_static_scratch: the W8A8 linear with a
// scratch buffer compiled into the library, for callers that cannot allocate
// device memory (include/qurl.h says which, and why).
//
// The buffer is the only device variable of this translation unit, so it sits
// in a CUDA module of its own: under the CUDA runtime's default lazy module
// loading that module -- and with it the buffer's bytes -- is committed on a
// device only when this file first looks the buffer up there, i.e. on the
// first call of this entry point with that device current.  (With
// CUDA_MODULE_LOADING=EAGER every module of the library, this one included,
// is loaded when the library's first call creates or binds a context.)
//
// The entry point only sizes, looks up and hands over the buffer: the
// computation is qurl_w8a8_linear's, with the buffer as its workspace.  Given
// at least qurl_workspace_size() bytes the planner takes the same tiles, K
// splits and summation order as for a caller's workspace, so the results are
// bit-identical to qurl_w8a8_linear's.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "qurl.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

// In host code this name stands for the variable, not for a device address:
// the address is looked up per device with cudaGetSymbolAddress below.
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of the buffer on the current device; the first call made with
// a device current looks it up (which also loads this module there).
qurl_status scratch_of_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QURL_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return QURL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return QURL_ERR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return QURL_OK;
}

}  // namespace

extern "C" qurl_status qurl_w8a8_linear_static_scratch(const void* Xq, const float* sx, const void* Wq,
                                                       const float* sw, int M, int N, int K, qurl_qtype qt, void* Y,
                                                       int ldy, qurl_stream_t stream) {
  if (!Xq || !sx || !Wq || !sw || !Y || M <= 0 || N <= 0 || K <= 0 || ldy < N) return QURL_ERR_INVALID_ARG;
  if (qt != QURL_INT8 && qt != QURL_FP8_E4M3) return QURL_ERR_INVALID_ARG;
  // the scratch this shape's plan uses (on the current device) must fit; an
  // attached fp16 weight copy's plan that does not fit falls back to it
  if (qurl::plain_workspace_bytes(M, N, K, qt) > kStaticScratchBytes) return QURL_ERR_WORKSPACE;
  void* scratch = nullptr;
  const qurl_status s = scratch_of_current_device(&scratch);
  if (s != QURL_OK) return s;
  // Nothing in the buffer has to start at zero: every byte the kernels read
  // there (the fp16 activation codes and their sums, split-K partials) is
  // written earlier in the same call.  qurl_w8a8_linear validates the rest
  // (alignment, K % 16) before launching anything.
  return qurl_w8a8_linear(Xq, sx, Wq, sw, M, N, K, qt, Y, ldy, scratch, kStaticScratchBytes, stream);
}
