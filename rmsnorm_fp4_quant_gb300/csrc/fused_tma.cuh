// fused_tma.cuh - the main fused kernel: persistent CTAs that stream rows
// through a shared-memory ring filled by the TMA bulk-copy engine.
//
// Why: the op is HBM-bound (about 6.5 bytes and ~8 instructions per element),
// and a thread can only keep its own chunks in flight while it holds them in
// registers, so a register-resident design ties the bytes in flight per SM to
// the occupancy.  Here one elected thread per CTA issues cp.async.bulk copies
// of whole rows of x and r (rows are contiguous, so one copy per tensor per
// stage) up to S stages ahead into shared memory, completing on an mbarrier;
// the CTA computes the current row from registers while the next rows land.
// Bytes in flight per SM = CTAs/SM * S * stage bytes, independent of registers.
//
// Pipeline of one CTA (rows_per_cta R rows per stage, CTA b of G handles row
// groups b, b + G, b + 2G, ...):
//   wait full[s]  ->  each row slice copies its chunks smem -> registers,
//   h = rn(x + r), h -> residual (global), partial sums -> shared  ->
//   __syncthreads (stage s is free; partials visible)  ->
//   thread 0 refills stage s with group i + S  ->  rstd  ->  phase 3 stores.
// The partial-sum array is double-buffered by iteration parity, so one
// barrier per row group suffices.
//
// Every mbarrier wait is bounded (~1 s of clock cycles).  A CTA whose wait
// runs out agrees on it with __syncthreads_or, marks the scale bytes of its
// remaining rows 0xFF (NaN in E4M3 and UE8M0), stores the timeout status in
// the caller's status word (if any), lets thread 0 drain the copies still in
// flight, and returns.  The drain waits, each bounded the same way, for every
// stage that has a copy issued; a stage whose wait ran out because the bytes
// it expects never arrive holds no copy that could still land.  A bulk copy
// from device memory that has been issued either completes or faults the
// context, so once those waits end no copy can still be writing into this
// CTA's shared memory.
#pragma once

#include "async_copy.cuh"
#include "fused_common.cuh"

namespace fp4q {

__device__ __forceinline__ void ld_shared_chunk(const void* p, Chunk& c) {
  const uint32_t a = smem_addr(p);
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3]) : "r"(a));
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4+16];"
               : "=r"(c.u[4]), "=r"(c.u[5]), "=r"(c.u[6]), "=r"(c.u[7]) : "r"(a));
}


// Dynamic shared memory of one CTA: S stages of {x rows, r rows}, S full
// barriers, a double-buffered array of 32 warp partials.
__host__ __device__ constexpr size_t tma_smem_bytes(int stages, int rows_per_cta, int H) {
  return static_cast<size_t>(stages) * 4u * rows_per_cta * H + 8u * stages + 2u * 32u * 4u;
}

#if defined(FP4Q_TMA_MAXNREG) && FP4Q_TMA_MAXNREG > 0
#define FP4Q_TMA_REGS(CPT) __maxnreg__((CPT) <= 2 ? FP4Q_TMA_MAXNREG : 128)
#else
#define FP4Q_TMA_REGS(CPT) __launch_bounds__(max_threads_for_cpt(CPT))
#endif

template <typename T, int FMT, int CPT, bool EX>
__global__ void FP4Q_TMA_REGS(CPT)
fused_tma_kernel(const FusedParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = p.stages;
  const int R = p.rows_per_cta;
  const int H = p.H;
  const uint32_t half_stage = 2u * R * H;          // bytes of R rows of one tensor
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * 2u * half_stage);
  float* part = reinterpret_cast<float*>(full + S);

  const int tid = threadIdx.x;
  const int tpr = p.tpr;
  const int grp = tid / tpr;                        // row slice within the stage
  const int lane = tid - grp * tpr;
  const int c_end = p.nchunk;

  const int64_t G = gridDim.x;
  const int64_t b = blockIdx.x;
  const int64_t n_iter = b < p.groups ? (p.groups - b + G - 1) / G : 0;

  // producer side, thread 0 only
  auto issue = [&](int64_t it) {
    const int s = static_cast<int>(it % S);
    const int64_t row0 = (b + it * G) * R;
    const int64_t left = p.M - row0;
    const uint32_t nrows = left <= 0 ? 0u : static_cast<uint32_t>(left < R ? left : R);
    const uint32_t bytes = nrows * 2u * H;
    mbar_arrive_expect_tx(&full[s], 2u * bytes);   // zero bytes completes the phase at once
    if (FP4Q_DROP(p, 1, static_cast<int>(b), static_cast<int>(it))) return;   // debug build
    if (bytes) {
      uint8_t* st = smem + static_cast<size_t>(s) * 2u * half_stage;
      // rows of a stage are contiguous in memory (strided rows run with R = 1)
      const T* xs = static_cast<const T*>(p.x) + row0 * (EX ? p.x_stride : H);
      const T* rs = static_cast<const T*>(p.r) + row0 * (EX ? p.r_stride : H);
      if (FP4Q_IN_RANGE(p, xs, bytes, p.x, x_extent(p))) bulk_g2s(st, xs, bytes, &full[s]);
      if (FP4Q_IN_RANGE(p, rs, bytes, p.r, r_extent(p))) bulk_g2s(st + half_stage, rs, bytes, &full[s]);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    mbar_init_fence();
  }
  __syncthreads();
  griddep_wait();                            // inputs may come from the kernel before (PDL)
  if (tid == 0) {
    for (int64_t it = 0; it < n_iter && it < S; ++it) issue(it);
  }
  griddep_launch_dependents();

  const int warp = tid >> 5;
  const int wpr = tpr >> 5;                         // warps per slice (tpr >= 32)
  const float gs = load_global_scale(p.gs);
  for (int64_t it = 0; it < n_iter; ++it) {
    const int s = static_cast<int>(it % S);
    const uint32_t parity = static_cast<uint32_t>((it / S) & 1);
    const int64_t row = (b + it * G) * R + grp;
    const bool row_ok = row < p.M;

    const bool ok = mbar_wait_bounded(&full[s], parity, FP4Q_WAIT_LIMIT(p));
    Chunk h[CPT];
    Chunk rr[CPT];
    if (ok && row_ok) {
      const uint8_t* sx = smem + static_cast<size_t>(s) * 2u * half_stage + static_cast<size_t>(grp) * 2u * H;
      const uint8_t* sr = sx + half_stage;
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const int c = lane + k * tpr;
        if (c < c_end) {
          ld_shared_chunk(sx + c * 32, h[k]);
          ld_shared_chunk(sr + c * 32, rr[k]);
        }
      }
    }
    T* rrow = static_cast<T*>(p.r) + static_cast<size_t>(row_ok ? row : 0) *
                                         static_cast<size_t>(EX ? p.r_stride : H);
    float ss = add_and_write_back<T, CPT>(p, h, rr, rrow, lane, tpr, c_end, ok && row_ok);

    const int width = tpr < 32 ? tpr : 32;
    for (int o = width >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
    float* pp = part + (it & 1) * 32;
    if (tpr > 32 && (tid & 31) == 0) pp[warp] = ss;

    // stage s consumed by every thread, partials visible; agree on failure
    if (__syncthreads_or(!ok)) {
      for (int64_t j = it; j < n_iter; ++j)
        mark_row_failed<FMT>(p, (b + j * G) * R + grp, lane, tpr, c_end);
      if (tid == 0) {
        if (p.status) atomicExch(p.status, kStatusTimeout);
        // stages it .. it + S - 1 were issued (the last refill was issue(it - 1 + S))
        for (int64_t j = it; j < n_iter && j < it + S; ++j)
          mbar_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1), FP4Q_WAIT_LIMIT(p));
      }
      return;
    }
    if (tid == 0 && it + S < n_iter) issue(it + S);

    if (tpr > 32) {
      ss = 0.0f;
      for (int i = 0; i < wpr; ++i) ss += pp[grp * wpr + i];
    }
    const float rstd = row_rstd(ss, H, p.eps);
    quantize_and_store<T, FMT, CPT, EX>(h, rstd, gs, p, row, lane, tpr, c_end, row_ok);
    if (p.sf_tiled && !row_ok && row < p.rows) zero_tiled_row(p, row, lane, tpr);
  }
}

}  // namespace fp4q
