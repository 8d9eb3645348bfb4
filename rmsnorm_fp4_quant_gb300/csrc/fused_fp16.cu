// fp16 instances of the fused kernels (their own translation unit).
#include "fused_launch.cuh"

namespace fp4q {
cudaError_t launch_fused_fp16(int fmt, const FusedShape& s, const FusedParams& p,
                              cudaStream_t stream) {
  return launch_dtype<__half>(fmt, s, p, stream);
}
int tma_ctas_per_sm_fp16(int fmt, int cpt, int threads, size_t smem) {
  return ctas_per_sm_dtype<__half>(fmt, cpt, threads, smem);
}
}  // namespace fp4q
