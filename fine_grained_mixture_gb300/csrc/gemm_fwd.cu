// gemm_fwd.cu - forward instantiations of the grouped-GEMM kernel: up-projection with the token gather and
// SwiGLU epilogue, down-projection with the score-weighted aggregation epilogue (reading A, or recomputing it
// from the cached H).
#include "gemm.cuh"

namespace moe {

int launch_up(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s) { return launch_gemm<kUp, 256, 4>(a, tm, s); }

int launch_down(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, bool det) {
  if (use_cta_pairs(a.Kdim)) {
    if (det) return launch_gemm<kDown, 256, 4, 1, true, 2>(a, tm, s);
    return launch_gemm<kDown, 256, 4, 1, false, 2>(a, tm, s);
  }
  if (det) return launch_gemm<kDown, 256, 3, 1, true>(a, tm, s);
  return launch_gemm<kDown, 256, 3>(a, tm, s);
}

int launch_down_h(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, bool det) {
  if (det) return launch_gemm<kDownH, 256, 3, 1, true>(a, tm, s);
  return launch_gemm<kDownH, 256, 3>(a, tm, s);
}

}  // namespace moe
