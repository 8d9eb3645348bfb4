// fused_common.cuh - the per-row phases of the fused residual-add + RMSNorm +
// FP4 quantization (FlashInfer `add_rmsnorm_fp4quant.py`,
// `AddRMSNormFP4QuantKernel.kernel`, phases 2 and 3), shared by the persistent
// TMA kernel and the cluster kernel.
//
// Work decomposition.  A row of H elements is cut into 16-element chunks (32
// bytes of bf16/fp16: one NVFP4 block, half an MXFP4 block).  A "row slice" of
// `tpr` threads owns chunks c0, c0 + tpr, c0 + 2 tpr, ... (CPT of them, c0 =
// slice start + lane), so one 256-bit access per thread covers 1 KiB per warp.
// A thread keeps its chunks of h in registers between the two phases.
#pragma once

#include "fp4q_device.cuh"
#include "fp4q_launch.h"

namespace fp4q {

// Formats: NVFP4 (16-element blocks, E4M3 scales), MXFP4 (32, UE8M0), and
// 32-element blocks with E4M3 scales (FlashInfer `scale_format="e4m3"` on the
// block-32 branch).
constexpr int kFmtNV = 0;
constexpr int kFmtMX = 1;
constexpr int kFmtE4B32 = 2;
template <int FMT> struct Fmt {
  static constexpr bool kBlock32 = FMT != kFmtNV;   // a block is two chunks
  static constexpr bool kE4M3 = FMT != kFmtMX;      // E4M3 scale, global scale applies
};

// The global scale: one fp32 on the device (read once per thread), 1 if absent.
__device__ __forceinline__ float load_global_scale(const float* gs) {
  return gs ? __ldg(gs) : 1.0f;
}

// Phase 2, first half: h = rn(x + r) with the packed bf16x2 / f16x2 add (x
// arrives in h[], r in rr[]), h written back to the residual row at once, and
// this thread's partial sum of h^2 (exact squares from the mixed-precision
// FMA; two fp32 lanes: even / odd elements, chunk order).
template <typename T, int CPT>
__device__ __forceinline__ float add_and_write_back(const FusedParams& p, Chunk (&h)[CPT],
                                                    const Chunk (&rr)[CPT], T* rrow, int c0,
                                                    int tpr, int c_end, bool row_ok) {
  float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = c0 + k * tpr;
    if (row_ok && c < c_end) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t u = Pair<T>::add(h[k].u[j], rr[k].u[j]);
        h[k].u[j] = u;
        Pair<T>::sq_acc(u, ss2);
      }
      if (FP4Q_IN_RANGE(p, rrow + c * 16, 32, p.r, r_extent(p))) st_stream(rrow + c * 16, h[k]);
    }
  }
  return ss2.x + ss2.y;
}

// rstd = 1 / sqrt(ss / H + eps), each step correctly rounded.
__device__ __forceinline__ float row_rstd(float ss, int H, float eps) {
  const float ms = __fdiv_rn(ss, static_cast<float>(H));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// Phase 3 for one row slice: y = (h * w) * rstd (h * w exact in fp32, so y is
// one rounding of the product; FlashInfer's cluster branch multiplies in this
// order), block amax (32-element
// blocks: a shuffle with the neighbouring lane joins the two chunks), the
// scale byte, v = y * inv_s, E2M1 codes of 16 elements in one 64-bit store, and
// the scale byte in each layout asked for.  Every lane of the warp must call it
// (the shuffle is unconditional); lanes without a chunk contribute amax 0.
// EX is the general form (strided rows, optional y side output); the common
// dense instance carries none of that code.
template <typename T, int FMT, int CPT, bool EX>
__device__ __forceinline__ void quantize_and_store(const Chunk (&h)[CPT], float rstd, float gs,
                                                   const FusedParams& p, int64_t row, int c0,
                                                   int tpr, int c_end, bool row_ok) {
  const float2 rstd2 = make_float2(rstd, rstd);
  const T* wvec = static_cast<const T*>(p.w);
  uint8_t* prow = p.packed + static_cast<size_t>(row_ok ? row : 0) * static_cast<size_t>(p.H / 2);
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int c = c0 + k * tpr;
    const bool ok = row_ok && c < c_end;
    float y[16];
    float amax = 0.0f;
    if (ok) {
      Chunk wc = {};
      if (FP4Q_IN_RANGE(p, wvec + c * 16, 32, p.w, 2LL * p.H)) wc = ld_cached_ro(wvec + c * 16);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 yy = __fmul2_rn(Pair<T>::mul(h[k].u[j], wc.u[j]), rstd2);   // (h * w) * rstd
        y[2 * j] = yy.x;
        y[2 * j + 1] = yy.y;
        amax = max_abs3(amax, yy.x, yy.y);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = 0.0f;
    }
    if (Fmt<FMT>::kBlock32) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    if (EX && ok && p.y) {   // side output: y rounded to the storage type
      Chunk yc;
#pragma unroll
      for (int j = 0; j < 8; ++j) yc.u[j] = Pair<T>::from_f32(y[2 * j], y[2 * j + 1]);
      T* yp = static_cast<T*>(p.y) + static_cast<size_t>(row) * p.H + c * 16;
      if (FP4Q_IN_RANGE(p, yp, 32, p.y, 2LL * p.M * p.H)) st_stream(yp, yc);
    }
    if (ok) {
      float v[16];
      float inv_s;
      const uint32_t code = Fmt<FMT>::kE4M3 ? e4m3_block_scale(amax, gs, inv_s)
                                            : ue8m0_block_scale(amax, inv_s);
      // v = y * inv_s; a zero E4M3 scale (inv_s = 0) gives +0 codes
      if (inv_s > 0.0f) {
        const float2 inv2 = make_float2(inv_s, inv_s);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float2 vv = __fmul2_rn(make_float2(y[i], y[i + 1]), inv2);
          v[i] = vv.x;
          v[i + 1] = vv.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
      }
      const uint64_t packed = static_cast<uint64_t>(e2m1_pack8(v)) |
                              (static_cast<uint64_t>(e2m1_pack8(v + 8)) << 32);
      if (FP4Q_IN_RANGE(p, prow + static_cast<size_t>(c) * 8, 8, p.packed, packed_extent(p.M, p.H)))
        st_u64(prow + static_cast<size_t>(c) * 8, packed);

      const bool owner = !Fmt<FMT>::kBlock32 || ((c & 1) == 0);
      if (owner) {
        const int kb = Fmt<FMT>::kBlock32 ? (c >> 1) : c;
        uint8_t* rm = p.sf_rm + static_cast<size_t>(row) * p.nb + kb;
        if (p.sf_rm && FP4Q_IN_RANGE(p, rm, 1, p.sf_rm, static_cast<long long>(p.M) * p.nb))
          st_u8(rm, code);
        if (p.sf_tiled) {
          uint8_t* tl = p.sf_tiled + tiled_sf_offset(row, kb, p.nkt);
          if (FP4Q_IN_RANGE(p, tl, 1, p.sf_tiled, tiled_extent(p.M, p.nkt))) st_u8(tl, code);
          if (kb == p.nb - 1) {   // k padding of the last 4-block group
            for (int kk = p.nb; kk < 4 * p.nkt; ++kk) {
              uint8_t* pad = p.sf_tiled + tiled_sf_offset(row, kk, p.nkt);
              if (FP4Q_IN_RANGE(p, pad, 1, p.sf_tiled, tiled_extent(p.M, p.nkt))) st_u8(pad, 0u);
            }
          }
        }
      }
    }
  }
}

// A padding row of the tiled layout (M <= row < 128*ceil(M/128)): zero its
// nkt four-byte groups.
__device__ __forceinline__ void zero_tiled_row(const FusedParams& p, int64_t row, int lane,
                                               int tpr) {
  for (int g = lane; g < p.nkt; g += tpr) {
    uint8_t* q = p.sf_tiled + tiled_sf_offset(row, 4 * g, p.nkt);
    if (FP4Q_IN_RANGE(p, q, 4, p.sf_tiled, tiled_extent(p.M, p.nkt))) st_u32(q, 0u);
  }
}

// Marks a row whose inputs never arrived: every scale byte of the slice set
// to 0xFF (NaN in both E4M3 and UE8M0), so a consumer sees the failure.
template <int FMT>
__device__ __forceinline__ void mark_row_failed(const FusedParams& p, int64_t row, int c0,
                                                int tpr, int c_end) {
  if (row >= p.M) return;
  for (int c = c0; c < c_end; c += tpr) {
    if (Fmt<FMT>::kBlock32 && (c & 1)) continue;
    const int kb = Fmt<FMT>::kBlock32 ? (c >> 1) : c;
    uint8_t* rm = p.sf_rm + static_cast<size_t>(row) * p.nb + kb;
    if (p.sf_rm && FP4Q_IN_RANGE(p, rm, 1, p.sf_rm, static_cast<long long>(p.M) * p.nb))
      st_u8(rm, 0xFFu);
    uint8_t* tl = p.sf_tiled + tiled_sf_offset(row, kb, p.nkt);
    if (p.sf_tiled && FP4Q_IN_RANGE(p, tl, 1, p.sf_tiled, tiled_extent(p.M, p.nkt)))
      st_u8(tl, 0xFFu);
  }
}

}  // namespace fp4q
