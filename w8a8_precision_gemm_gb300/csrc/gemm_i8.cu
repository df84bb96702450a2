// gemm_i8.cu -- instantiations of the INT8 W8A8 GEMM (int8 codes widened to
// fp16 in shared memory, tcgen05 kind::f16, exact chunked int32 accumulation).
#include "gemm.cuh"

namespace qurl {

// Shared memory: STAGES x (128 + BN) x 64 B of int8 staging plus
// 3 x (128 + BN) x 128 B of fp16 tiles.
cudaError_t launch_gemm_i8(bool swap, int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a,
                            dim3 grid, cudaStream_t st) {
  if (swap) {
    switch (bn) {
      case 16: return launch_gemm_inst<kQInt8, true, 16, 6>(ta, tb, a, grid, st);
      case 32: return launch_gemm_inst<kQInt8, true, 32, 6>(ta, tb, a, grid, st);
      case 64: return launch_gemm_inst<kQInt8, true, 64, 6>(ta, tb, a, grid, st);
      case 128: return launch_gemm_inst<kQInt8, true, 128, 6>(ta, tb, a, grid, st);
      default: break;
    }
  } else if (bn == 128) {
    return launch_gemm_inst<kQInt8, false, 128, 6>(ta, tb, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qurl
