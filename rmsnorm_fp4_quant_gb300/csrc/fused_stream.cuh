// fused_stream.cuh - persistent form of the register-resident fused kernel for
// long batches of rows up to a few thousand elements.
//
// Why: the one-row-per-CTA kernel keeps a row's bytes in flight only while
// that CTA is in its load phase; its add, reduction and stores leave the
// memory pipe idle for that CTA, and a grid of many waves ends in a partial
// wave (8192 rows over 608 resident CTAs: 13.5 waves).  Here a grid of
// resident CTAs walks the row groups g = blockIdx.x, blockIdx.x + G, ...
// and every thread holds two row buffers in registers: while it adds,
// reduces and quantizes the row of group g, the 256-bit loads of group g + G
// are already in flight.  The loop is unrolled by two so the buffers keep
// fixed register names.  All CTAs do the same number of groups up to one,
// so the grid ends together.
//
// Per group: R row slices of tpr threads, one row each, chunks c = lane,
// lane + tpr, ... as in the other kernels.  The slice sum of squares goes
// through a shared array double-buffered by iteration parity, so one CTA
// barrier per group suffices (none when a slice is one warp or less).
#pragma once

#include "async_copy.cuh"
#include "fused_common.cuh"

namespace fp4q {

template <typename T, int CPT, bool EX>
__device__ __forceinline__ void stream_load(const FusedParams& p, int64_t row, int lane, int tpr,
                                            Chunk (&x)[CPT], Chunk (&r)[CPT]) {
  if (row >= p.M) return;
  const T* xrow = static_cast<const T*>(p.x) +
                  static_cast<size_t>(row) * static_cast<size_t>(EX ? p.x_stride : p.H);
  const T* rrow = static_cast<const T*>(p.r) +
                  static_cast<size_t>(row) * static_cast<size_t>(EX ? p.r_stride : p.H);
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = lane + k * tpr;
    if (c < p.nchunk) {
      if (FP4Q_IN_RANGE(p, xrow + c * 16, 32, p.x, x_extent(p))) x[k] = ld_stream_ro(xrow + c * 16);
      if (FP4Q_IN_RANGE(p, rrow + c * 16, 32, p.r, r_extent(p))) r[k] = ld_stream_rw(rrow + c * 16);
    }
  }
}

// One row of one slice: x arrives in h[], r in rr[]; everything after the
// loads (phases 2 and 3), with the CTA barrier of the slice reduction.
template <typename T, int FMT, int CPT, bool EX>
__device__ __forceinline__ void stream_row(const FusedParams& p, int64_t row, int lane, int tpr,
                                           int grp, float* part, float gs, Chunk (&h)[CPT],
                                           const Chunk (&rr)[CPT]) {
  const bool row_ok = row < p.M;
  T* rrow = static_cast<T*>(p.r) + static_cast<size_t>(row_ok ? row : 0) *
                                       static_cast<size_t>(EX ? p.r_stride : p.H);
  float ss = add_and_write_back<T, CPT>(p, h, rr, rrow, lane, tpr, p.nchunk, row_ok);
  const int width = tpr < 32 ? tpr : 32;
  for (int o = width >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
  if (tpr > 32) {
    const int wpr = tpr >> 5;
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    ss = 0.0f;
    for (int i = 0; i < wpr; ++i) ss += part[grp * wpr + i];
  }
  const float rstd = row_rstd(ss, p.H, p.eps);
  quantize_and_store<T, FMT, CPT, EX>(h, rstd, gs, p, row, lane, tpr, p.nchunk, row_ok);
  if (p.sf_tiled && !row_ok && row < p.rows) zero_tiled_row(p, row, lane, tpr);
}

template <typename T, int FMT, int CPT, bool EX>
__global__ void __launch_bounds__(max_threads_for_cpt(CPT))
fused_stream_kernel(const FusedParams p) {
  __shared__ float part[2][32];
  const int tid = threadIdx.x;
  const int tpr = p.tpr;
  const int grp = tid / tpr;
  const int lane = tid - grp * tpr;
  const int R = p.rows_per_cta;
  const int64_t G = gridDim.x;
  int64_t g = blockIdx.x;
  if (g >= p.groups) return;                 // whole CTA

  griddep_wait();                            // inputs may come from the kernel before (PDL)
  Chunk xa[CPT], ra[CPT], xb[CPT], rb[CPT];
  stream_load<T, CPT, EX>(p, g * R + grp, lane, tpr, xa, ra);
  griddep_launch_dependents();
  const float gs = load_global_scale(p.gs);
  for (;;) {
    const int64_t g1 = g + G;
    if (g1 < p.groups) stream_load<T, CPT, EX>(p, g1 * R + grp, lane, tpr, xb, rb);
    stream_row<T, FMT, CPT, EX>(p, g * R + grp, lane, tpr, grp, part[0], gs, xa, ra);
    if (g1 >= p.groups) break;
    const int64_t g2 = g1 + G;
    if (g2 < p.groups) stream_load<T, CPT, EX>(p, g2 * R + grp, lane, tpr, xa, ra);
    stream_row<T, FMT, CPT, EX>(p, g1 * R + grp, lane, tpr, grp, part[1], gs, xb, rb);
    if (g2 >= p.groups) break;
    g = g2;
  }
}

}  // namespace fp4q
