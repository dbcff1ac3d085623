// The fused forward's instances with phase-trace stamps (the kernel is in
// fused_kernel.cuh), launched while a trace buffer is set; compiled in their
// own translation unit beside fused.cu.
#include "fused_kernel.cuh"

namespace dlrm {

cudaError_t fused_prepare_traced(int bm, int cw, int lda) {
  return prepare_fused_instances<true>(bm, cw, lda);
}

cudaError_t launch_fused_traced(const FusedParams& p, int bm, cudaStream_t stream) {
  return launch_fused_instances<true>(p, bm, stream);
}

}  // namespace dlrm
