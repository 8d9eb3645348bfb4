// gemm_launch.h - parameter block and launch entry of the FP4 GEMM kernels
// (gemm_nvfp4.cu), used by the C entry points in gemm_api.cu.  Internal.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "debug_checks.h"

namespace fp4q {

// NVFP4 x NVFP4 -> bf16 GEMM (bf16 tensors as raw 16-bit words).
constexpr int kEpiPlain = 0;      // alpha * acc (+ bias) (+ residual) -> bf16
constexpr int kEpiGelu = 1;       // GELU(alpha * acc (+ bias)) -> bf16
constexpr int kEpiGeluFp4 = 2;    // GELU(alpha * acc (+ bias)) -> NVFP4 codes + tiled scales
struct GemmParams {
  const uint8_t* sfa;          // tiled scales of A, ceil(M/128) * nkt * 512 bytes
  const uint8_t* sfb;          // tiled scales of B, ceil(N/128) * nkt * 512 bytes
  const uint16_t* bias;        // [N] bf16 or null
  const uint16_t* residual;    // [M, N] bf16 or null
  uint16_t* out;               // [M, N] bf16 (kEpiPlain, kEpiGelu)
  uint8_t* out_packed;         // [M, N/2] E2M1 codes (kEpiGeluFp4)
  uint8_t* out_sf;             // tiled E4M3 scales of the output (kEpiGeluFp4)
  int* status;                 // optional device status word: the timeout status on a timeout
  int epilogue;                // kEpi*
  int out_nkt;                 // ceil(N / 64): scale groups per output row (kEpiGeluFp4)
  int rows_out;                // rows the epilogue visits: M, or 128 * ceil(M / 128) (kEpiGeluFp4)
  float alpha;
  int M, N, K;
  int nkt;                     // 128x4 scale tiles per 128 rows: ceil(K / 64) (NVFP4),
                               // ceil(K / 128) (MXFP4)
  int num_kb;                  // ceil(K / 256): K blocks, the last one possibly ragged
  int mma_last;                // K = 64 MMAs in the last K block (1..4)
  int sf_tiles_last;           // scale tiles per 128 rows in the last K block
  int stages;                  // shared-memory ring depth, 2..6
  int sf_stages;               // scale ring depth of the persistent kernel: stages or stages + 1
  int split;                   // CTAs of a cluster sharing one tile's K loop (1 = none)
  int b_static;                // 1: the kernel before this one (PDL) writes neither B nor its scales
  uint32_t tmem_cols;          // tensor-memory columns taken per CTA
  FP4Q_DEBUG_FIELD             // debug build only: checks and fault injection
};

// K % 32 == 0, N % 8 == 0, a / b 16-byte aligned (checked by the caller);
// bn = output tile width, 128 or 256; persistent = one CTA per SM walking the
// tiles (else one CTA per tile); mx = MXFP4 operands (UE8M0 scale per 32
// codes) instead of NVFP4 (E4M3 per 16).
cudaError_t launch_gemm_nvfp4(const uint8_t* a, const uint8_t* b, GemmParams p, int bn,
                              bool persistent, bool mx, int pdl, cudaStream_t stream);

}  // namespace fp4q
