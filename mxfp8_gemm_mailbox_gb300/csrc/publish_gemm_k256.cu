// The publishing GEMM kernels with two K tiles per pipeline stage (cta_k 256:
// 256 F K per stage), folds 1, 2 and 4 with split-K 1, 2 or 4 and the 32x32b
// accumulator read-out, compiled apart so the translation units build in
// parallel.
#include "publish_gemm_kernel.cuh"

namespace mxfp8 {
namespace {

template <int F>
cudaError_t set_for_fold(int split_k, int bytes) {
  switch (split_k) {
    case 1:
      return set_smem_impl<1, false, F, 2>(bytes);
    case 2:
      return set_smem_impl<2, false, F, 2>(bytes);
    case 4:
      return set_smem_impl<4, false, F, 2>(bytes);
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
      return launch_impl<1, false, F, 2>(tmap_w, tmap_x, p, stream, programmatic);
    case 2:
      return launch_impl<2, false, F, 2>(tmap_w, tmap_x, p, stream, programmatic);
    case 4:
      return launch_impl<4, false, F, 2>(tmap_w, tmap_x, p, stream, programmatic);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t set_wide_stage_gemm_smem_attribute(int split_k, int fold, int bytes) {
  if (fold == 1) return set_for_fold<1>(split_k, bytes);
  if (fold == 2) return set_for_fold<2>(split_k, bytes);
  if (fold == 4) return set_for_fold<4>(split_k, bytes);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wide_stage_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                           const GemmParams& p, int split_k, cudaStream_t stream,
                                           bool programmatic) {
  if (p.tmem_load == MXFP8_TMEM_LOAD_16X256B) return cudaErrorInvalidValue;
  if (p.fold == 1) return launch_for_fold<1>(tmap_w, tmap_x, p, split_k, stream, programmatic);
  if (p.fold == 2) return launch_for_fold<2>(tmap_w, tmap_x, p, split_k, stream, programmatic);
  if (p.fold == 4) return launch_for_fold<4>(tmap_w, tmap_x, p, split_k, stream, programmatic);
  return cudaErrorInvalidValue;
}

}  // namespace mxfp8
