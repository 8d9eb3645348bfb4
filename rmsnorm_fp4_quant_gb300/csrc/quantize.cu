// quantize.cu - standalone block quantization of a bf16/fp16 matrix to packed
// E2M1 codes plus scales, without the residual add and the normalisation (the
// producer the FlashRT `fp4-gemm` README lists as `quantize_fp4_sfa_bf16` /
// `quantize_fp4_sfa_fp16`; block scales as in the fused kernels).
//
// No value depends on anything but its own block, so this is a flat streaming
// kernel: a work item is a segment of 32 consecutive 16-element chunks of one
// row (one chunk per lane, 1 KiB per warp load); each warp takes
// FP4Q_QUANT_SEGS items and issues all their 256-bit loads before using any.
// The grid covers every item once (many short CTAs; the hardware scheduler
// balances them), rows >= M (padding rows of the tiled scale layout) write
// only zero scale bytes.
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
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = 0.0f;
  }
  if (Fmt<FMT>::kBlock32) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
  if (row < 0) return;                      // lane past the last row slot
  const bool owner = !Fmt<FMT>::kBlock32 || ((c & 1) == 0);
  const int kb = Fmt<FMT>::kBlock32 ? (c >> 1) : c;
  if (row >= p.M) {                         // padding row of the tiled layout
    if (owner) {
      st_u8(p.sf_tiled + tiled_sf_offset(row, kb, p.nkt), 0u);
      if (kb == p.nb - 1)
        for (int kk = p.nb; kk < 4 * p.nkt; ++kk) st_u8(p.sf_tiled + tiled_sf_offset(row, kk, p.nkt), 0u);
    }
    return;
  }
  float inv_s;
  const uint32_t code = Fmt<FMT>::kE4M3 ? e4m3_block_scale(amax, gs, inv_s)
                                        : ue8m0_block_scale(amax, inv_s);
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
  st_u64(p.packed + row * static_cast<int64_t>(p.H / 2) + static_cast<int64_t>(c) * 8, packed);
  if (owner) {
    if (p.sf_rm) st_u8(p.sf_rm + row * p.nb + kb, code);
    if (p.sf_tiled) {
      st_u8(p.sf_tiled + tiled_sf_offset(row, kb, p.nkt), code);
      if (kb == p.nb - 1)
        for (int kk = p.nb; kk < 4 * p.nkt; ++kk) st_u8(p.sf_tiled + tiled_sf_offset(row, kk, p.nkt), 0u);
    }
  }
}

#ifndef FP4Q_QUANT_SEGS
#define FP4Q_QUANT_SEGS 2
#endif
constexpr int kSegsPerStep = FP4Q_QUANT_SEGS;   // row segments (32 chunks each) per warp

template <typename T, int FMT>
__global__ void __launch_bounds__(256) quantize_kernel(const QuantParams p) {
  const float gs = load_global_scale(p.gs);
  // work item = one 32-chunk segment of one row slot; lane l takes chunk 32*seg + l
  const int segs_per_row = (p.nchunk + 31) >> 5;
  const int64_t items = p.rows * static_cast<int64_t>(segs_per_row);
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const T* x = static_cast<const T*>(p.x);
  // one group of items per warp (the grid covers them all; no grid-stride tail);
  // all lanes of a warp take the same path (the block-32 shuffle needs them)
  for (int64_t base = warp * kSegsPerStep; base < items; base += nwarps * kSegsPerStep) {
    int64_t row[kSegsPerStep];
    int c[kSegsPerStep];
    bool have[kSegsPerStep];
    Chunk xc[kSegsPerStep];
#pragma unroll
    for (int u = 0; u < kSegsPerStep; ++u) {            // warp-uniform index math, then loads
      const int64_t it = base + u;
      const int64_t r = it < items ? it / segs_per_row : -1;
      row[u] = r;
      c[u] = r >= 0 ? static_cast<int>(it - r * segs_per_row) * 32 + lane : p.nchunk;
      if (c[u] >= p.nchunk) row[u] = -1;                // lane past the row's last chunk
      have[u] = row[u] >= 0 && row[u] < p.M;
      if (have[u]) xc[u] = ld_stream_ro(x + row[u] * p.H + c[u] * 16);
    }
#pragma unroll
    for (int u = 0; u < kSegsPerStep; ++u) quantize_chunk<T, FMT>(p, xc[u], have[u], row[u], c[u], gs);
  }
}

template <typename T>
cudaError_t launch_q(int fmt, const QuantParams& p, int64_t blocks, cudaStream_t stream) {
  const unsigned g = static_cast<unsigned>(blocks);
  switch (fmt) {
    case kFmtNV: quantize_kernel<T, kFmtNV><<<g, 256, 0, stream>>>(p); break;
    case kFmtMX: quantize_kernel<T, kFmtMX><<<g, 256, 0, stream>>>(p); break;
    case kFmtE4B32: quantize_kernel<T, kFmtE4B32><<<g, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(int dtype, int fmt, const QuantParams& p, int num_sms,
                            cudaStream_t stream) {
  const int64_t items = p.rows * static_cast<int64_t>((p.nchunk + 31) / 32);
  if (items == 0) return cudaSuccess;
  int64_t blocks = (items + 8 * kSegsPerStep - 1) / (8 * kSegsPerStep);   // 8 warps per block
  (void)num_sms;
  if (blocks > INT32_MAX) return cudaErrorInvalidConfiguration;
  return dtype == 0 ? launch_q<__nv_bfloat16>(fmt, p, blocks, stream)
                    : launch_q<__half>(fmt, p, blocks, stream);
}

}  // namespace fp4q
