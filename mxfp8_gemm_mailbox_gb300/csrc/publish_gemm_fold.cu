// The folded publishing GEMM kernels (F = 2 and 4 K pieces stacked in the
// MMA's rows with split-K 1, 2 or 4; F = 8 unsplit; 32x32b accumulator
// loads), compiled apart from the unfolded ones so the two translation units
// build in parallel.
#include "publish_gemm_kernel.cuh"

namespace mxfp8 {
namespace {

template <int F>
cudaError_t set_for_fold(int split_k, int bytes) {
  switch (split_k) {
    case 1:
      return set_smem_impl<1, false, F>(bytes);
    case 2:
      return set_smem_impl<2, false, F>(bytes);
    case 4:
      return set_smem_impl<4, false, F>(bytes);
    default:
      return cudaErrorInvalidValue;
  }
}

template <int F>
cudaError_t launch_for_fold(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                            const GemmParams& p, int split_k, cudaStream_t stream,
                            bool programmatic) {
  switch (split_k) {
    case 1:
      return launch_impl<1, false, F>(tmap_w, tmap_x, p, stream, programmatic);
    case 2:
      return launch_impl<2, false, F>(tmap_w, tmap_x, p, stream, programmatic);
    case 4:
      return launch_impl<4, false, F>(tmap_w, tmap_x, p, stream, programmatic);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t set_folded_gemm_smem_attribute(int split_k, int fold, int bytes) {
  if (fold == 2) return set_for_fold<2>(split_k, bytes);
  if (fold == 4) return set_for_fold<4>(split_k, bytes);
  if (fold == 8 && split_k == 1) return set_smem_impl<1, false, 8>(bytes);
  return cudaErrorInvalidValue;
}

cudaError_t launch_folded_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                       const GemmParams& p, int split_k, cudaStream_t stream,
                                       bool programmatic) {
  if (p.tmem_load == MXFP8_TMEM_LOAD_16X256B) return cudaErrorInvalidValue;
  if (p.fold == 2) return launch_for_fold<2>(tmap_w, tmap_x, p, split_k, stream, programmatic);
  if (p.fold == 4) return launch_for_fold<4>(tmap_w, tmap_x, p, split_k, stream, programmatic);
  if (p.fold == 8 && split_k == 1 && p.pipes <= 2)
    return launch_impl<1, false, 8>(tmap_w, tmap_x, p, stream, programmatic);
  return cudaErrorInvalidValue;
}

}  // namespace mxfp8
