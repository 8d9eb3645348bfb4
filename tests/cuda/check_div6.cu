// Exhaustive check of the library's div6_rn (the block-scale quotient amax/6)
// against CUDA's correctly rounded division __fdiv_rn(a, 6.0f), for every
// non-negative float bit pattern from +0 up to +inf.  Prints the mismatch
// count; exit status 0 when the kernel ran.
#include <cstdio>

#include "fp4q_device.cuh"

__device__ unsigned long long g_mismatch;
__device__ unsigned int g_first_bad;

__global__ void check(unsigned int last) {
  for (unsigned long long i = blockIdx.x * 256ull + threadIdx.x; i <= last;
       i += static_cast<unsigned long long>(gridDim.x) * 256ull) {
    const float a = __uint_as_float(static_cast<unsigned int>(i));
    const float got = fp4q::div6_rn(a);
    const float want = __fdiv_rn(a, 6.0f);
    if (__float_as_uint(got) != __float_as_uint(want)) {
      if (atomicAdd(&g_mismatch, 1ull) == 0) g_first_bad = static_cast<unsigned int>(i);
    }
  }
}

int main() {
  const unsigned long long zero = 0;
  if (cudaMemcpyToSymbol(g_mismatch, &zero, sizeof(zero)) != cudaSuccess) return 2;
  check<<<152 * 16, 256>>>(0x7F800000u);
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  unsigned long long bad = 0;
  unsigned int first = 0;
  cudaMemcpyFromSymbol(&bad, g_mismatch, sizeof(bad));
  cudaMemcpyFromSymbol(&first, g_first_bad, sizeof(first));
  std::printf("mismatches=%llu first=0x%08x\n", bad, first);
  return 0;
}
