// fused_kernel.cuh - the fused residual-add + RMSNorm + FP4 quantization
// kernel for sm_103a (FlashInfer `add_rmsnorm_fp4quant.py`,
// `AddRMSNormFP4QuantKernel.kernel`, phases 1-3).
//
// Work decomposition.  A row of H elements is cut into 16-element chunks (32
// bytes of bf16/fp16: one NVFP4 block, half an MXFP4 block).  A "row slice" of
// `tpr` threads owns chunks lane, lane + tpr, lane + 2 tpr, ... (CPT of them),
// so each 256-bit load instruction of a warp reads 1 KiB of contiguous memory.
// Without clusters a CTA holds `rows_per_cta` slices, one row each.  With a
// cluster of C CTAs one row is split into C slices of nchunk / C chunks and the
// partial sums of squares are exchanged through distributed shared memory (the
// page's cluster path does the same with an mbarrier; here a hardware cluster
// barrier orders the st.shared::cluster stores, so no thread ever spins).
//
// Per row the kernel:
//   1. loads x and r (256-bit, streaming), forms h = rn(x + r) with the packed
//      bf16x2 / f16x2 add and writes h back to the residual at once;
//   2. reduces sum(h^2): fp32 per thread (two packed f32x2 lanes, chunk
//      order), a shuffle tree in the warp, warps in order through shared
//      memory, cluster ranks in order;
//   3. rstd = 1 / sqrt(ss / H + eps) with correctly rounded division and root;
//   4. per chunk: y = (h * rstd) * w, block amax (MXFP4: one shuffle joins the
//      two chunks of a 32-element block), the scale byte, the E2M1 codes of 16
//      elements in one 64-bit store, the scale byte(s) in each layout asked for;
//   5. slices of padding rows (tiled layout, rows M..128*ceil(M/128)) write
//      zeros; the owner of the last block of a row zeroes the k padding.
// Everything stays in registers; the only shared memory is the reduction.
#pragma once

#include "fp4q_device.cuh"
#include "fp4q_launch.h"

namespace fp4q {

constexpr int kFmtNV = 0;
constexpr int kFmtMX = 1;


__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void st_peer_f32(float* local_slot, uint32_t peer, float v) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(local_slot));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(peer));
  asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(remote), "f"(v) : "memory");
}

template <typename T, int FMT, int CPT>
__global__ void __launch_bounds__(max_threads_for_cpt(CPT))
fused_add_rmsnorm_fp4_kernel(const FusedParams p) {
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
    cluster_arrive_relaxed();   // matched by the wait before the DSMEM stores
  } else {
    row = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta + grp;
  }
  const bool row_ok = row < p.M;
  const int c_begin = rank * p.chunks_per_cta;
  const int c_end = c_begin + p.chunks_per_cta;

  const size_t row_off = static_cast<size_t>(row_ok ? row : 0) * static_cast<size_t>(p.H);
  const T* xrow = static_cast<const T*>(p.x) + row_off;
  T* rrow = static_cast<T*>(p.r) + row_off;

  // ---- 1. load x, r; h = rn(x + r); write h back -------------------------
  Chunk h[CPT];
  Chunk rr[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = c_begin + lane + k * tpr;
    if (row_ok && c < c_end) {
      h[k] = ld_stream_ro(xrow + c * 16);
      rr[k] = ld_stream_rw(rrow + c * 16);
    }
  }
  // even elements accumulate in .x, odd ones in .y (packed f32x2 FMA)
  float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = c_begin + lane + k * tpr;
    if (row_ok && c < c_end) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t u = Pair<T>::add(h[k].u[j], rr[k].u[j]);
        h[k].u[j] = u;
        const float2 f = Pair<T>::to_f32(u);
        ss2 = __ffma2_rn(f, f, ss2);   // squares of 8/11-bit significands are exact
      }
      st_stream(rrow + c * 16, h[k]);
    }
  }
  float ss = ss2.x + ss2.y;

  // ---- 2. sum of squares over the row ------------------------------------
  const int width = tpr < 32 ? tpr : 32;
  for (int o = width >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
  if (tpr > 32) {
    const int wpr = tpr >> 5;
    if ((tid & 31) == 0) warp_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int i = 0; i < wpr; ++i) tot += warp_part[grp * wpr + i];
    ss = tot;
  }
  if (p.cluster > 1) {
    cluster_wait_acquire();                      // every CTA of the cluster is running
    if (tid < p.cluster) st_peer_f32(&cluster_part[rank], static_cast<uint32_t>(tid), ss);
    cluster_arrive_release();
    cluster_wait_acquire();                      // all partials have landed here
    float tot = 0.0f;
    for (int i = 0; i < p.cluster; ++i) tot += cluster_part[i];
    ss = tot;
  }

  // ---- 3. reciprocal RMS ---------------------------------------------------
  const float ms = __fdiv_rn(ss, static_cast<float>(p.H));
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));

  // ---- 4. normalise, scale, quantize, store --------------------------------
  const float2 rstd2 = make_float2(rstd, rstd);
  const T* wvec = static_cast<const T*>(p.w);
  uint8_t* prow = p.packed + static_cast<size_t>(row_ok ? row : 0) * static_cast<size_t>(p.H / 2);
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = c_begin + lane + k * tpr;
    const bool ok = row_ok && c < c_end;
    float y[16];
    float amax = 0.0f;
    if (ok) {
      const Chunk wc = ld_cached_ro(wvec + c * 16);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 hf = Pair<T>::to_f32(h[k].u[j]);
        const float2 wf = Pair<T>::to_f32(wc.u[j]);
        const float2 yy = __fmul2_rn(__fmul2_rn(hf, rstd2), wf);   // (h * rstd) * w
        y[2 * j] = yy.x;
        y[2 * j + 1] = yy.y;
        amax = fmaxf(amax, fmaxf(fabsf(yy.x), fabsf(yy.y)));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = 0.0f;
    }
    if (FMT == kFmtMX) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    if (ok) {
      float v[16];
      float inv_s;
      const uint32_t code = (FMT == kFmtNV) ? nvfp4_scale(amax, inv_s) : mxfp4_scale(amax, inv_s);
      // v = y * (1/s); a zero NVFP4 scale has inv_s = 0 and gives +0 codes
      const float2 inv2 = make_float2(inv_s, inv_s);
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 vv = __fmul2_rn(make_float2(y[i], y[i + 1]), inv2);
        v[i] = vv.x;
        v[i + 1] = vv.y;
      }
      const uint64_t packed = static_cast<uint64_t>(e2m1_pack8(v)) |
                              (static_cast<uint64_t>(e2m1_pack8(v + 8)) << 32);
      st_u64(prow + static_cast<size_t>(c) * 8, packed);

      const bool owner = (FMT == kFmtNV) || ((c & 1) == 0);
      if (owner) {
        const int kb = (FMT == kFmtNV) ? c : (c >> 1);
        if (p.sf_rm) st_u8(p.sf_rm + static_cast<size_t>(row) * p.nb + kb, code);
        if (p.sf_tiled) {
          st_u8(p.sf_tiled + tiled_sf_offset(row, kb, p.nkt), code);
          if (kb == p.nb - 1) {
            for (int kk = p.nb; kk < 4 * p.nkt; ++kk)
              st_u8(p.sf_tiled + tiled_sf_offset(row, kk, p.nkt), 0u);
          }
        }
      }
    }
  }

  // ---- 5. padding rows of the tiled layout ---------------------------------
  if (p.sf_tiled && !row_ok && row < p.rows && rank == 0) {
    for (int g = lane; g < p.nkt; g += tpr) st_u32(p.sf_tiled + tiled_sf_offset(row, 4 * g, p.nkt), 0u);
  }
}

template <typename T, int FMT>
cudaError_t launch_fused_fmt(const FusedShape& s, const FusedParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(s.threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (s.cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  switch (s.cpt) {
    case 1: return cudaLaunchKernelEx(&cfg, fused_add_rmsnorm_fp4_kernel<T, FMT, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, fused_add_rmsnorm_fp4_kernel<T, FMT, 2>, p);
    case 3: return cudaLaunchKernelEx(&cfg, fused_add_rmsnorm_fp4_kernel<T, FMT, 3>, p);
    case 4: return cudaLaunchKernelEx(&cfg, fused_add_rmsnorm_fp4_kernel<T, FMT, 4>, p);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_fused_dtype(int fmt, const FusedShape& s, const FusedParams& p,
                               cudaStream_t stream) {
  return fmt == kFmtNV ? launch_fused_fmt<T, kFmtNV>(s, p, stream)
                       : launch_fused_fmt<T, kFmtMX>(s, p, stream);
}

}  // namespace fp4q
