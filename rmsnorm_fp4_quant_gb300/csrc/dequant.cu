// dequant.cu - validation kernel: packed E2M1 codes times their block scale
// (format 0: 16-element blocks, E4M3; 1: 32, UE8M0; 2: 32, E4M3),
// fp32 out (FlashRT `fp4-gemm` README, Validation: compare through the
// dequantised values; `dequantize_fp4_sfa_fp16`).  One thread per 16-element
// chunk: one 64-bit code load, one scale byte, four 128-bit stores.
#include "fp4q_device.cuh"
#include "fp4q_launch.h"

namespace fp4q {
namespace {

// E2M1 magnitude of a 3-bit index: exponent bits e = idx >> 1, mantissa bit
// m = idx & 1; e == 0 is subnormal (m * 0.5), else (1 + m/2) * 2^(e-1).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t idx = code & 7u;
  const uint32_t e = idx >> 1, m = idx & 1u;
  const float mag = e ? (1.0f + 0.5f * static_cast<float>(m)) * static_cast<float>(1u << (e - 1))
                      : 0.5f * static_cast<float>(m);
  return (code & 8u) ? -mag : mag;
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  if (e == 15u && m == 7u) return __uint_as_float(0x7FC00000u);   // NaN
  const float sig = static_cast<float>(e ? (8u + m) : m);
  const float pw = __uint_as_float(((e ? e : 1u) + 117u) << 23);   // 2^(max(E,1) - 10)
  const float mag = sig * pw;
  return (code & 0x80u) ? -mag : mag;
}

__device__ __forceinline__ float ue8m0_value(uint32_t code) {
  if (code == 255u) return __uint_as_float(0x7FC00000u);
  return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);   // 2^(code-127)
}

template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(const DequantParams p) {
  const int64_t total = p.M * static_cast<int64_t>(p.nchunk);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / p.nchunk;
    const int c = static_cast<int>(i - row * p.nchunk);
    const int kb = FMT == 0 ? c : (c >> 1);          // 16- or 32-element blocks
    const uint8_t* crow = p.packed + row * (p.H / 2);
    const uint64_t codes = *reinterpret_cast<const uint64_t*>(crow + static_cast<int64_t>(c) * 8);
    const int64_t soff = p.tiled ? tiled_sf_offset(row, kb, p.nkt) : row * p.nb + kb;
    const uint32_t sb = p.sf[soff];
    const float s = FMT == 1 ? ue8m0_value(sb) : e4m3_value(sb);
    float4* out = reinterpret_cast<float4*>(p.out + row * p.H + static_cast<int64_t>(c) * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t nib = static_cast<uint32_t>(codes >> (16 * q));
      out[q] = make_float4(e2m1_value(nib & 0xF) * s, e2m1_value((nib >> 4) & 0xF) * s,
                           e2m1_value((nib >> 8) & 0xF) * s, e2m1_value((nib >> 12) & 0xF) * s);
    }
  }
}

}  // namespace

cudaError_t launch_dequant(int fmt, const DequantParams& p, cudaStream_t stream) {
  const int64_t total = p.M * static_cast<int64_t>(p.nchunk);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  // cudaLaunchKernelEx reports this launch's own error; the thread's sticky
  // last error (which may be the caller's) is left alone
  if (fmt == 0) return cudaLaunchKernelEx(&cfg, dequant_kernel<0>, p);
  if (fmt == 1) return cudaLaunchKernelEx(&cfg, dequant_kernel<1>, p);
  return cudaLaunchKernelEx(&cfg, dequant_kernel<2>, p);
}

}  // namespace fp4q
