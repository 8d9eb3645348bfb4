// fp4q_launch.h - host/device shared parameter blocks and the launch entry
// points behind the C ABI (include/fp4q.h).  Internal to the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "debug_checks.h"

namespace fp4q {

// Shared by the C entry points (api.cu, gemm_api.cu).
int record_cuda_error(cudaError_t err);   // 0, or the CUDA-error status after noting err
int sm_count_current_device();            // SMs of the current device (cached)
inline bool abi_aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
inline bool abi_overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

// Threads per CTA allowed for a kernel instance holding `cpt` chunks per
// thread: one chunk fits 64 registers (1024 threads), more chunks need up to 128.
__host__ __device__ constexpr int max_threads_for_cpt(int cpt) { return cpt <= 1 ? 1024 : 512; }

// One fused launch.  All pointers are device pointers; sf_tiled / sf_rm are
// null when that layout is not written.
struct FusedParams {
  const void* x;
  void* r;
  const void* w;
  uint8_t* packed;
  uint8_t* sf_tiled;
  uint8_t* sf_rm;
  const float* gs;     // device global scale (one fp32) or null for 1
  void* y;             // optional [M, H] dtype output of y (dense), or null
  int* status;         // optional device status word: set to the timeout status on a timeout
  int64_t x_stride;    // elements between rows of x
  int64_t r_stride;    // elements between rows of the residual
  float eps;
  int64_t M;           // valid rows
  int64_t rows;        // row slots covered by the grid (M, or 128*ceil(M/128) when tiled)
  int H;
  int nchunk;          // H / 16
  int nb;              // H / block
  int nkt;             // ceil(nb / 4)
  int tpr;             // threads per row slice
  int rows_per_cta;    // row slices per CTA (rows per stage for the TMA kernel)
  int cluster;         // CTAs per row (direct kernel), 1 otherwise
  int chunks_per_cta;  // nchunk / cluster
  int stages;          // shared-memory ring depth (TMA kernel)
  int64_t groups;      // ceil(rows / rows_per_cta) (TMA kernel)
  FP4Q_DEBUG_FIELD     // debug build only: checks and fault injection
};

// Byte extents of the buffers of a fused call, as the C ABI defines them.
__host__ __device__ inline long long x_extent(const FusedParams& p) {
  return ((p.M - 1) * p.x_stride + p.H) * 2;
}
__host__ __device__ inline long long r_extent(const FusedParams& p) {
  return ((p.M - 1) * p.r_stride + p.H) * 2;
}
__host__ __device__ inline long long packed_extent(int64_t M, int H) {
  return M * static_cast<long long>(H) / 2;
}
__host__ __device__ inline long long tiled_extent(int64_t M, int nkt) {
  return (M + 127) / 128 * static_cast<long long>(nkt) * 512;
}

constexpr int kPathTma = 0;       // persistent CTAs, TMA bulk-copy row ring
constexpr int kPathDirect = 1;    // register-resident rows, optionally one row per cluster

// Launch shape chosen on the host for one (M, H, format, dtype).
struct FusedShape {
  int path;
  int cpt;             // chunks per thread (template instance)
  int tpr;
  int rows_per_cta;
  int cluster;
  int chunks_per_cta;
  int stages;
  int threads;         // tpr * rows_per_cta
  size_t smem;         // dynamic shared memory bytes
  int64_t grid;        // CTAs
  int pdl;             // launch as a programmatic dependent of the previous kernel
};

// Picks the launch shape; returns false when the shape cannot be handled.
bool choose_fused_shape(int64_t M, int64_t rows, int H, int fmt, int dtype, int num_sms,
                        FusedShape* out);

// Launches the fused kernel (dtype 0 = bf16, 1 = fp16; fmt 0 = NVFP4, 1 = MXFP4).
cudaError_t launch_fused(int dtype, int fmt, const FusedShape& shape, const FusedParams& p,
                         cudaStream_t stream);

// CTAs of the TMA kernel instance that fit one SM (0 if none), after raising
// its dynamic shared-memory limit to `smem`.
int tma_ctas_per_sm(int dtype, int fmt, int cpt, int threads, size_t smem);

struct DequantParams {
  const uint8_t* packed;
  const uint8_t* sf;
  float* out;
  int64_t M;
  int H;
  int nchunk;
  int nb;
  int nkt;
  int tiled;           // 1: sf is in the 128x4 tiled layout, 0: row-major
};

cudaError_t launch_dequant(int fmt, const DequantParams& p, cudaStream_t stream);

// Standalone block quantization of x (no add, no normalisation).
struct QuantParams {
  const void* x;
  uint8_t* packed;
  uint8_t* sf_tiled;
  uint8_t* sf_rm;
  const float* gs;
  int64_t M;
  int64_t rows;        // row slots: M, or 128*ceil(M/128) with the tiled layout
  int H;
  int nchunk;
  int nb;
  int nkt;
  int evict_first;     // read the input with the L2 evict-first policy (set by the launcher)
  FP4Q_DEBUG_FIELD     // debug build only: checks
};

cudaError_t launch_quantize(int dtype, int fmt, const QuantParams& p, int pdl,
                            cudaStream_t stream);

}  // namespace fp4q
