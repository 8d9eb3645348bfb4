// bf16 instances of the fused kernel (compiled in their own translation unit).
#include "fused_kernel.cuh"

namespace fp4q {
cudaError_t launch_fused_bf16(int fmt, const FusedShape& s, const FusedParams& p,
                              cudaStream_t stream) {
  return launch_fused_dtype<__nv_bfloat16>(fmt, s, p, stream);
}
}  // namespace fp4q
