// quantize.cu - standalone block quantization of a bf16/fp16 matrix to packed
// E2M1 codes plus scales, without the residual add and the normalisation (the
// producer the FlashRT `fp4-gemm` README lists as `quantize_fp4_sfa_bf16` /
// `quantize_fp4_sfa_fp16`; block scales as in the fused kernels).
//
// No value depends on anything but its own block, so this is a flat streaming
// kernel: a warp takes SEGS segments of 32 consecutive 16-element chunks of
// one row (one chunk per lane, 1 KiB per warp load) and issues all their
// 256-bit loads before using any.  Grid: x = groups of 8 row slots (one per
// warp), y = runs of SEGS segments along the row, so no thread divides; the
// grid covers every segment once (many short CTAs, balanced by the hardware
// scheduler); where SEGS does not divide the row's segments the last run is
// ragged and its missing segments are skipped.  Rows >= M (padding rows of
// the tiled scale layout) only write zero scale bytes.
#include "async_copy.cuh"
#include "fused_common.cuh"

namespace fp4q {
namespace {

template <typename T, int FMT>
__device__ __forceinline__ void quantize_chunk(const QuantParams& p, const Chunk& xc, bool have,
                                               int64_t row, int c, float gs) {
  float y[16];
  float amax = 0.0f;
  if (have) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 f = Pair<T>::to_f32(xc.u[j]);
      y[2 * j] = f.x;
      y[2 * j + 1] = f.y;
      amax = max_abs3(amax, f.x, f.y);
    }
  }
  // every lane takes part in the shuffle; lanes past the row then leave
  if (Fmt<FMT>::kBlock32) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
  if (c >= p.nchunk) return;
  const bool owner = !Fmt<FMT>::kBlock32 || ((c & 1) == 0);
  const int kb = Fmt<FMT>::kBlock32 ? (c >> 1) : c;
  uint32_t code = 0;                        // padding rows of the tiled layout keep code 0
  if (have) {
    float inv_s;
    code = Fmt<FMT>::kE4M3 ? e4m3_block_scale(amax, gs, inv_s) : ue8m0_block_scale(amax, inv_s);
    float v[16];
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
    uint8_t* pk = p.packed + row * static_cast<int64_t>(p.H / 2) + static_cast<int64_t>(c) * 8;
    if (FP4Q_IN_RANGE(p, pk, 8, p.packed, packed_extent(p.M, p.H))) st_u64(pk, packed);
  }
  if (owner) {
    uint8_t* rm = p.sf_rm + row * p.nb + kb;
    if (p.sf_rm && have && FP4Q_IN_RANGE(p, rm, 1, p.sf_rm, static_cast<long long>(p.M) * p.nb))
      st_u8(rm, code);
    if (p.sf_tiled) {
      uint8_t* tl = p.sf_tiled + tiled_sf_offset(row, kb, p.nkt);
      if (FP4Q_IN_RANGE(p, tl, 1, p.sf_tiled, tiled_extent(p.M, p.nkt))) st_u8(tl, code);
      if (kb == p.nb - 1) {                 // k padding of the last 4-block group
        for (int kk = p.nb; kk < 4 * p.nkt; ++kk) {
          uint8_t* pad = p.sf_tiled + tiled_sf_offset(row, kk, p.nkt);
          if (FP4Q_IN_RANGE(p, pad, 1, p.sf_tiled, tiled_extent(p.M, p.nkt))) st_u8(pad, 0u);
        }
      }
    }
  }
}

// Three or four segments per warp: capped at 64 registers (four CTAs per SM),
// which measured 7-9 % faster than the uncapped 73-82 (three CTAs per SM).
template <typename T, int FMT, int SEGS>
__global__ void __launch_bounds__(256, SEGS >= 3 ? 4 : 1) quantize_kernel(const QuantParams p) {
  const float gs = load_global_scale(p.gs);
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= p.rows) return;                          // whole warps leave together
  griddep_wait();                                     // input from the kernel before (PDL)
  const bool have_row = row < p.M;
  const T* xrow = static_cast<const T*>(p.x) + row * p.H;
  int c[SEGS];
  bool have[SEGS];
  Chunk xc[SEGS];
#pragma unroll
  for (int u = 0; u < SEGS; ++u) {                    // all loads first
    c[u] = (blockIdx.y * SEGS + u) * 32 + lane;
    have[u] = have_row && c[u] < p.nchunk;
    if (have[u] && FP4Q_IN_RANGE(p, xrow + c[u] * 16, 32, p.x, 2LL * p.M * p.H))
      xc[u] = p.evict_first ? ld_stream_ro_evict_first(xrow + c[u] * 16)
                            : ld_stream_ro(xrow + c[u] * 16);
  }
  griddep_launch_dependents();
#pragma unroll
  for (int u = 0; u < SEGS; ++u) quantize_chunk<T, FMT>(p, xc[u], have[u], row, c[u], gs);
}

// SEGS: 4 or 3 where it divides the row's segment count, else 4 with a
// ragged last run from 8 segments up (measured 2-11 % faster than runs of 2),
// else 2 or 1.
template <typename T, int FMT>
cudaError_t launch_q_fmt(const QuantParams& p, int pdl, cudaStream_t stream) {
  const int segs = (p.nchunk + 31) / 32;
  const int per = segs % 4 == 0 ? 4
                : segs % 3 == 0 ? 3
                : segs >= 8     ? 4
                : segs % 2 == 0 ? 2 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.rows + 7) / 8),
                     static_cast<unsigned>((segs + per - 1) / per));
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (per) {
    case 4: return cudaLaunchKernelEx(&cfg, quantize_kernel<T, FMT, 4>, p);
    case 3: return cudaLaunchKernelEx(&cfg, quantize_kernel<T, FMT, 3>, p);
    case 2: return cudaLaunchKernelEx(&cfg, quantize_kernel<T, FMT, 2>, p);
    default: return cudaLaunchKernelEx(&cfg, quantize_kernel<T, FMT, 1>, p);
  }
}

template <typename T>
cudaError_t launch_q(int fmt, const QuantParams& p, int pdl, cudaStream_t stream) {
  switch (fmt) {
    case kFmtNV: return launch_q_fmt<T, kFmtNV>(p, pdl, stream);
    case kFmtMX: return launch_q_fmt<T, kFmtMX>(p, pdl, stream);
    case kFmtE4B32: return launch_q_fmt<T, kFmtE4B32>(p, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_quantize(int dtype, int fmt, const QuantParams& p, int pdl,
                            cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  if ((p.rows + 7) / 8 > INT32_MAX || (p.nchunk + 31) / 32 > 65535)
    return cudaErrorInvalidConfiguration;
  // Inputs read with L2 evict-first for rows up to 8192 elements: measured
  // 6-9 % faster there (C3 / C4 shapes, 1536-wide rows), 1-2 % slower on
  // 17408- and 32768-wide rows.
  QuantParams q = p;
  q.evict_first = p.H <= 8192 ? 1 : 0;
  return dtype == 0 ? launch_q<__nv_bfloat16>(fmt, q, pdl, stream)
                     : launch_q<__half>(fmt, q, pdl, stream);
}

}  // namespace fp4q
