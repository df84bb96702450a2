// gemm_fp8.cu -- instantiations of the FP8-E4M3 W8A8 GEMM (tcgen05 kind::f8f6f4).
#include "gemm.cuh"

namespace qurl {

// Stage counts fill ~192 KB of shared memory: (128 + BN) x 128 B per stage.
cudaError_t launch_gemm_fp8(bool swap, int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                            dim3 grid, cudaStream_t st) {
  if (swap) {
    switch (bn) {
      case 16: return launch_gemm_inst<kQFp8, true, 16, 8>(ta, tb, a, grid, st);
      case 32: return launch_gemm_inst<kQFp8, true, 32, 8>(ta, tb, a, grid, st);
      case 64: return launch_gemm_inst<kQFp8, true, 64, 8>(ta, tb, a, grid, st);
      case 128: return launch_gemm_inst<kQFp8, true, 128, 6>(ta, tb, a, grid, st);
      case 256: return launch_gemm_inst<kQFp8, true, 256, 4>(ta, tb, a, grid, st);
      default: break;
    }
  } else if (bn == 256) {
    return launch_gemm_inst<kQFp8, false, 256, 4>(ta, tb, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qurl
