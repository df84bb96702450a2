// probe.cu -- tensor-rate probes: kernels that issue a fixed number of
// multiply-accumulate instructions of one kind and nothing else, so that a
// caller timing a launch with CUDA events obtains the rate of that instruction
// on this GPU.  They measure the denominators of the roofline (which 8-bit
// integer route is fastest on sm_103a), not a step of the method.
//
//   route 0  mma.sync.m16n8k32 s8 x s8 -> s32: the warp-level integer MMA
//            (8 warps per CTA, four independent accumulator chains per warp);
//   route 1  tcgen05.mma kind::f16, fp16 x fp16 -> fp32, M = 128, N = 256,
//            K = 16, both operands in shared memory (the route the INT8 GEMMs
//            take, with the codes widened to fp16 exactly);
//   route 2  the same with the A operand read from tensor memory;
//   route 3  tcgen05.mma kind::f8f6f4, e4m3 x e4m3 -> fp32, M = 128, N = 256,
//            K = 32, both operands in shared memory (the FP8 route).
//
// The operand tiles are zero, so the accumulators stay zero; the instructions
// run at full rate regardless of the values.
#include "gemm.cuh"

namespace qurl {
namespace {

constexpr int kProbeWarps = 8;
// tcgen05 probe: more dynamic shared memory than its tiles need, so that one
// CTA runs per SM (each allocates all 512 TMEM columns)
constexpr int kTcProbeSmem = 120 * 1024;

__device__ int g_probe_sink;

__global__ void __launch_bounds__(kProbeWarps * 32) mma_s8_probe_kernel(int iters, int* sink) {
  griddep_wait();
  griddep_launch_dependents();
  uint32_t a[4] = {threadIdx.x * 0x01010101u, 0x02020202u, 0x03030303u, 0x04040404u};
  uint32_t b[2] = {0x01010101u, threadIdx.x};
  int acc[4][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  int s = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) s += acc[c][0] ^ acc[c][1] ^ acc[c][2] ^ acc[c][3];
  if (s == 0x7F3A19C5) sink[0] = s;  // keeps the chains alive; never true for these inputs
}

// One CTA per SM; one thread issues `iters` MMAs into one accumulator.
// route 1: f16 SS; route 2: f16 with A in TMEM; route 3: e4m3 SS.
__global__ void __launch_bounds__(128, 1) tc_probe_kernel(int route, int iters, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tA = smem;              // 128 rows x 128 B, 128-byte swizzled K-major
  uint8_t* tB = smem + 128 * 128;  // 256 rows x 128 B
  const int warp = threadIdx.x >> 5;
  griddep_wait();
  griddep_launch_dependents();
  for (int i = threadIdx.x; i < (128 + 256) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (route == 2) {
    // zero the A operand's TMEM columns 256 .. 263 (one K = 16 slice of fp16 per lane)
    uint32_t z[32] = {};
    tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t sa = smem_addr(tA), sb = smem_addr(tB);
    const uint32_t idesc = umma_idesc_f32acc(0, 0, 128, 256);
    for (int i = 0; i < iters; ++i) {
      const int kk = i & 3;
      if (route == 1)
        umma_f16(tmem, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), idesc, i != 0);
      else if (route == 3)
        umma_f8f6f4(tmem, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), idesc, i != 0);
      else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
            "r"(tmem + 256), "l"(umma_desc_sw128(sb + kk * 32)), "r"(idesc), "r"(static_cast<uint32_t>(i != 0))
            : "memory");
    }
    umma_commit(&done);
    mbar_wait_drain(&done, 0, status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Multiply-add operations x 2 of one probe launch.
double probe_ops(int route, int ctas, int iters) {
  if (route == 0) return static_cast<double>(ctas) * kProbeWarps * iters * 4 * (2.0 * 16 * 8 * 32);
  const double per = (route == 3) ? 2.0 * 128 * 256 * 32 : 2.0 * 128 * 256 * 16;
  return static_cast<double>(ctas) * iters * per;
}

cudaError_t launch_probe(int route, int ctas, int iters, int* status, cudaStream_t st) {
  if (route == 0) {
    int* sink = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&sink), g_probe_sink);
    if (e != cudaSuccess) return e;
    return launch_pdl(mma_s8_probe_kernel, dim3(ctas), dim3(kProbeWarps * 32), 0, st, iters, sink);
  }
  const int smem = kTcProbeSmem;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_pdl(tc_probe_kernel, dim3(ctas), dim3(128), smem, st, route, iters, status);
}

}  // namespace qurl
