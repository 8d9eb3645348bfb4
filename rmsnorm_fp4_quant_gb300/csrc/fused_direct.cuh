// fused_direct.cuh - the register-resident fused kernel: every CTA loads its
// rows straight into registers with 256-bit streaming loads, one row per row
// slice of `tpr` threads, `rows_per_cta` slices per CTA; many CTAs per SM keep
// the rows in flight.  Used for rows up to a few thousand elements and, with a
// thread-block cluster, for short batches and very wide rows.
//
// Cluster mode splits one row over a cluster of C CTAs (FlashInfer
// `add_rmsnorm_fp4quant.py`, `_compute_cluster_n` and the cluster branch of
// `kernel`, which split H over a cluster the same way): CTA rank q owns chunks
// [q * nchunk/C, (q+1) * nchunk/C), reduces its partial sum of squares in the
// CTA and stores it into slot q of every peer's shared memory
// (st.shared::cluster via mapa).  A hardware cluster barrier (arrive.release /
// wait.acquire) orders those stores before the peers read them, so no thread
// ever spins on a flag; every CTA then sums the C partials in rank order and
// gets the same rstd.  Row slots beyond M (the padding rows of the tiled scale
// layout) only zero their scale bytes.
#pragma once

#include "async_copy.cuh"
#include "fused_common.cuh"

namespace fp4q {

__device__ __forceinline__ void st_peer_f32(float* local_slot, uint32_t peer, float v) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(local_slot));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(peer));
  asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(remote), "f"(v) : "memory");
}

// Register budget: the launch bound of the instance, or a cap on the one- and
// two-chunk instances (more CTAs resident per SM) when FP4Q_DIRECT_MAXNREG is set.
#if defined(FP4Q_DIRECT_MAXNREG) && FP4Q_DIRECT_MAXNREG > 0
#define FP4Q_DIRECT_REGS(CPT) __maxnreg__((CPT) <= 2 ? FP4Q_DIRECT_MAXNREG : 128)
#else
#define FP4Q_DIRECT_REGS(CPT) __launch_bounds__(max_threads_for_cpt(CPT))
#endif

template <typename T, int FMT, int CPT, bool EX>
__global__ void FP4Q_DIRECT_REGS(CPT)
fused_direct_kernel(const FusedParams p) {
  __shared__ float warp_part[32];
  __shared__ float cluster_part[16];

  const int tid = threadIdx.x;
  const int tpr = p.tpr;
  const int grp = tid / tpr;
  const int lane = tid - grp * tpr;

  int64_t row;
  int rank = 0;
  if (p.cluster > 1) {
    rank = static_cast<int>(cluster_ctarank());
    row = blockIdx.x / p.cluster;
    cluster_arrive_relaxed();                // matched by the wait before the DSMEM stores
  } else {
    row = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta + grp;
  }
  const bool row_ok = row < p.M;
  const int c_begin = rank * p.chunks_per_cta;
  const int c_end = c_begin + p.chunks_per_cta;
  const int c0 = c_begin + lane;
  const size_t rsafe = static_cast<size_t>(row_ok ? row : 0);
  const size_t xoff = rsafe * static_cast<size_t>(EX ? p.x_stride : p.H);
  const T* xrow = static_cast<const T*>(p.x) + xoff;
  T* rrow = static_cast<T*>(p.r) + (EX ? rsafe * static_cast<size_t>(p.r_stride) : xoff);

  griddep_wait();                            // inputs may come from the kernel before (PDL)
  Chunk h[CPT];
  Chunk rr[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = c0 + k * tpr;
    if (row_ok && c < c_end) {
      if (FP4Q_IN_RANGE(p, xrow + c * 16, 32, p.x, x_extent(p))) h[k] = ld_stream_ro(xrow + c * 16);
      if (FP4Q_IN_RANGE(p, rrow + c * 16, 32, p.r, r_extent(p))) rr[k] = ld_stream_rw(rrow + c * 16);
    }
  }
  griddep_launch_dependents();
  float ss = add_and_write_back<T, CPT>(p, h, rr, rrow, c0, tpr, c_end, row_ok);

  // slice reduction: shuffles within the slice's lanes, then its warps in order
  const int width = tpr < 32 ? tpr : 32;
  for (int o = width >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
  if (tpr > 32) {
    const int wpr = tpr >> 5;
    if ((tid & 31) == 0) warp_part[tid >> 5] = ss;
    __syncthreads();
    ss = 0.0f;
    for (int i = 0; i < wpr; ++i) ss += warp_part[grp * wpr + i];
  }
  if (p.cluster > 1) {                       // cluster reduction through DSMEM
    cluster_wait_acquire();                  // every CTA of the cluster is running
    if (tid < p.cluster) st_peer_f32(&cluster_part[rank], static_cast<uint32_t>(tid), ss);
    cluster_arrive_release();
    cluster_wait_acquire();                  // all partials have landed here
    ss = 0.0f;
    for (int i = 0; i < p.cluster; ++i) ss += cluster_part[i];
  }

  const float rstd = row_rstd(ss, p.H, p.eps);
  const float gs = load_global_scale(p.gs);
  quantize_and_store<T, FMT, CPT, EX>(h, rstd, gs, p, row, c0, tpr, c_end, row_ok);
  if (p.sf_tiled && !row_ok && row < p.rows && rank == 0) zero_tiled_row(p, row, lane, tpr);
}

}  // namespace fp4q
