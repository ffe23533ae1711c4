// gemm_bwd.cu - backward instantiations of the grouped-GEMM kernel: dH (dSwiGLU and dS in the epilogue),
// dX~ with the scatter-sum into dX, and the varlen-K weight gradients dW1 and dW2.
#include "gemm.cuh"

namespace moe {

int launch_dh(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, int bn, bool det) {
  if (det) {
    if (bn == 256) return launch_gemm<kDH, 256, 4, 1, true>(a, tm, s);
    return launch_gemm<kDH, 128, 4, 1, true>(a, tm, s);
  }
  if (bn == 256) return launch_gemm<kDH, 256, 4>(a, tm, s);
  return launch_gemm<kDH, 128, 4>(a, tm, s);
}

int launch_dx(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s, bool det) {
  if (use_cta_pairs(a.Kdim)) {
    if (det) return launch_gemm<kDX, 256, 4, 1, true, 2>(a, tm, s);
    return launch_gemm<kDX, 256, 4, 1, false, 2>(a, tm, s);
  }
  if (det) return launch_gemm<kDX, 256, 3, 1, true>(a, tm, s);
  return launch_gemm<kDX, 256, 3>(a, tm, s);
}

// 256-row M blocks (see Smem) when the weight's row count allows it and the experts' K loops are long
// enough (experts averaging >= 256 rows); else 128-row blocks with double-buffered TMEM.
int launch_dw1(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s) {
  if (a.wide_m && a.Mdim % 256 == 0) return launch_gemm<kDW1, 256, 3, 2>(a, tm, s);
  return launch_gemm<kDW1, 256, 4, 1>(a, tm, s);
}

int launch_dw2(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s) {
  if (a.wide_m && a.Mdim % 256 == 0) return launch_gemm<kDW2, 256, 3, 2>(a, tm, s);
  return launch_gemm<kDW2, 256, 4, 1>(a, tm, s);
}

// 256 x 256 tiles.  (256 x 128 tiles with two overlapping accumulators measured slower, fine7b 371 -> 565 us:
// they double the k-block iterations of the token gather, which sets the pace.)
int launch_dw12(const GemmArgs &a, const TensorMaps &tm, cudaStream_t s) {
  return launch_gemm<kDW, 256, 3, 2>(a, tm, s);
}

}  // namespace moe
