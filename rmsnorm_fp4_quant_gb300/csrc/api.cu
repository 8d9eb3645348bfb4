// api.cu - the C ABI of libfp4q.so (declared in include/fp4q.h): argument
// checks, launch-shape choice and dispatch to the sm_103a kernels.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fp4q.h"
#include "fp4q_launch.h"

namespace fp4q {
cudaError_t launch_fused_bf16(int fmt, const FusedShape& s, const FusedParams& p, cudaStream_t st);
cudaError_t launch_fused_fp16(int fmt, const FusedShape& s, const FusedParams& p, cudaStream_t st);

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxChunksPerCta = 2048;   // 32768 elements held in registers by one CTA
constexpr int kMaxCluster = 8;           // portable cluster size

inline int block_of(fp4_format_t f) { return f == FP4_NVFP4 ? 16 : 32; }

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

int num_sms_current_device() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

// Threads per slice for `chunks` chunks at `cpt` chunks per thread: a power of
// two in [2, 32], or a multiple of 32 above.
int round_tpr(int chunks, int cpt) {
  int t = (chunks + cpt - 1) / cpt;
  if (t <= 32) {
    int p = 2;
    while (p < t) p <<= 1;
    return p;
  }
  return (t + 31) / 32 * 32;
}

}  // namespace

bool choose_fused_shape(int64_t M, int H, int fmt, int num_sms, FusedShape* out) {
  const int nchunk = H / 16;
  // Cluster size: enough CTAs per row that a slice fits one CTA's registers,
  // and, for short batches, enough CTAs to cover the SMs.
  // A slice must be a whole number of chunks (of chunk pairs for MXFP4).
  auto splits = [&](int c) {
    return nchunk % c == 0 && (fmt == 0 || ((nchunk / c) & 1) == 0);
  };
  int cluster = 1;
  while (nchunk / cluster > kMaxChunksPerCta) cluster <<= 1;
  if (cluster > kMaxCluster || !splits(cluster)) return false;
  while (cluster < kMaxCluster && M * cluster < num_sms && nchunk / (cluster * 2) >= 128 &&
         splits(cluster * 2))
    cluster <<= 1;
  const int per_cta = nchunk / cluster;

  // Chunks per thread: least idle lanes, then more chunks per thread.
  int best_cpt = 0, best_tpr = 0, best_waste = 1 << 30;
  for (int cpt = 4; cpt >= 1; --cpt) {
    const int tpr = round_tpr(per_cta, cpt);
    const int maxt = max_threads_for_cpt(cpt);
    if (tpr > maxt) continue;
    const int waste = tpr * cpt - per_cta;
    if (waste < best_waste) {
      best_waste = waste;
      best_cpt = cpt;
      best_tpr = tpr;
    }
  }
  if (best_cpt == 0) return false;

  int rows_per_cta = 1;
  if (cluster == 1) {
    rows_per_cta = best_tpr >= 256 ? 1 : 256 / best_tpr;
    // short batches: spread rows over the SMs first
    const int64_t per_sm = (M + num_sms - 1) / num_sms;
    if (per_sm < rows_per_cta) rows_per_cta = static_cast<int>(per_sm < 1 ? 1 : per_sm);
    // whole warps
    while ((best_tpr * rows_per_cta) % 32) ++rows_per_cta;
  }
  if ((best_tpr * rows_per_cta) % 32 != 0) return false;   // whole warps only
  out->cpt = best_cpt;
  out->tpr = best_tpr;
  out->cluster = cluster;
  out->chunks_per_cta = per_cta;
  out->rows_per_cta = rows_per_cta;
  out->threads = best_tpr * rows_per_cta;
  out->grid = 0;
  return true;
}

cudaError_t launch_fused(int dtype, int fmt, const FusedShape& s, const FusedParams& p,
                         cudaStream_t stream) {
  return dtype == 0 ? launch_fused_bf16(fmt, s, p, stream) : launch_fused_fp16(fmt, s, p, stream);
}

}  // namespace fp4q

using namespace fp4q;

extern "C" {

int64_t fp4_sf_size_bytes(int64_t M, int64_t H, fp4_format_t format, fp4_sf_layout_t layout) {
  if (M < 0 || H <= 0) return -1;
  if (format != FP4_NVFP4 && format != FP4_MXFP4) return -1;
  const int64_t b = block_of(format);
  if (H % b) return -1;
  const int64_t nb = H / b;
  switch (layout) {
    case FP4_SF_ROWMAJOR:
      return M * nb;
    case FP4_SF_SWIZZLED:
    case FP4_SF_BOTH:
      return ((M + 127) / 128) * ((nb + 3) / 4) * 512;
    default:
      return -1;
  }
}

const char* fp4_status_string(fp4_status_t s) {
  switch (s) {
    case FP4_OK: return "ok";
    case FP4_ERR_INVALID_ARG: return "invalid argument";
    case FP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FP4_ERR_MISALIGNED: return "misaligned pointer";
    case FP4_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int fp4_last_cuda_error(void) { return g_last_cuda_error; }

fp4_status_t fp4_add_rmsnorm_quant(const void* input, void* residual, const void* weight,
                                   float eps, int64_t M, int64_t H, fp4_dtype_t dtype,
                                   fp4_format_t format, fp4_sf_layout_t sf_layout,
                                   uint8_t* out_packed, uint8_t* out_sf,
                                   uint8_t* out_sf_rowmajor, fp4q_stream_t stream) {
  if (dtype != FP4_DT_BF16 && dtype != FP4_DT_FP16) return FP4_ERR_INVALID_ARG;
  if (format != FP4_NVFP4 && format != FP4_MXFP4) return FP4_ERR_INVALID_ARG;
  if (sf_layout != FP4_SF_ROWMAJOR && sf_layout != FP4_SF_SWIZZLED && sf_layout != FP4_SF_BOTH)
    return FP4_ERR_INVALID_ARG;
  if (M < 0 || H <= 0 || !(eps >= 0.0f)) return FP4_ERR_INVALID_ARG;
  const int b = block_of(format);
  if (H % b != 0 || H < 64 || H > FP4Q_MAX_H) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FP4_OK;
  if (M > INT32_MAX) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (!input || !residual || !weight || !out_packed || !out_sf) return FP4_ERR_INVALID_ARG;
  if (sf_layout == FP4_SF_BOTH && !out_sf_rowmajor) return FP4_ERR_INVALID_ARG;
  if (!aligned(input, 32) || !aligned(residual, 32) || !aligned(weight, 32) ||
      !aligned(out_packed, 8))
    return FP4_ERR_MISALIGNED;
  // padding of the tiled buffer is zeroed with 4-byte stores
  if (sf_layout != FP4_SF_ROWMAJOR && !aligned(out_sf, 4)) return FP4_ERR_MISALIGNED;
  const int64_t act_bytes = M * H * 2;
  if (overlap(input, act_bytes, residual, act_bytes)) return FP4_ERR_INVALID_ARG;
  const int64_t sf_bytes = fp4_sf_size_bytes(M, H, format, sf_layout);
  if (overlap(out_packed, M * H / 2, out_sf, sf_bytes) ||
      overlap(out_packed, M * H / 2, residual, act_bytes) ||
      overlap(out_sf, sf_bytes, residual, act_bytes))
    return FP4_ERR_INVALID_ARG;

  FusedShape shape;
  if (!choose_fused_shape(M, static_cast<int>(H), format == FP4_MXFP4 ? 1 : 0,
                          num_sms_current_device(), &shape))
    return FP4_ERR_UNSUPPORTED_SHAPE;

  FusedParams p;
  p.x = input;
  p.r = residual;
  p.w = weight;
  p.packed = out_packed;
  p.sf_tiled = (sf_layout == FP4_SF_ROWMAJOR) ? nullptr : out_sf;
  p.sf_rm = (sf_layout == FP4_SF_ROWMAJOR) ? out_sf
            : (sf_layout == FP4_SF_BOTH)   ? out_sf_rowmajor
                                           : nullptr;
  p.eps = eps;
  p.M = M;
  p.rows = p.sf_tiled ? (M + 127) / 128 * 128 : M;
  p.H = static_cast<int>(H);
  p.nchunk = static_cast<int>(H / 16);
  p.nb = static_cast<int>(H / b);
  p.nkt = (p.nb + 3) / 4;
  p.tpr = shape.tpr;
  p.rows_per_cta = shape.rows_per_cta;
  p.cluster = shape.cluster;
  p.chunks_per_cta = shape.chunks_per_cta;
  shape.grid = shape.cluster > 1 ? p.rows * shape.cluster
                                 : (p.rows + shape.rows_per_cta - 1) / shape.rows_per_cta;
  if (shape.grid > INT32_MAX) return FP4_ERR_UNSUPPORTED_SHAPE;

  cudaError_t err = launch_fused(dtype == FP4_DT_BF16 ? 0 : 1, format == FP4_MXFP4 ? 1 : 0, shape,
                                 p, reinterpret_cast<cudaStream_t>(stream));
  if (err == cudaSuccess) err = cudaGetLastError();
  if (err != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(err);
    return FP4_ERR_CUDA;
  }
  return FP4_OK;
}

fp4_status_t fp4_dequant(const uint8_t* packed, const uint8_t* sf, int64_t M, int64_t H,
                         fp4_format_t format, fp4_sf_layout_t sf_layout, float* out,
                         fp4q_stream_t stream) {
  if (format != FP4_NVFP4 && format != FP4_MXFP4) return FP4_ERR_INVALID_ARG;
  if (sf_layout != FP4_SF_ROWMAJOR && sf_layout != FP4_SF_SWIZZLED) return FP4_ERR_INVALID_ARG;
  if (M < 0 || H <= 0) return FP4_ERR_INVALID_ARG;
  const int b = block_of(format);
  if (H % b != 0 || H > INT32_MAX / 2) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FP4_OK;
  if (!packed || !sf || !out) return FP4_ERR_INVALID_ARG;
  if (!aligned(packed, 8) || !aligned(out, 16)) return FP4_ERR_MISALIGNED;
  DequantParams p;
  p.packed = packed;
  p.sf = sf;
  p.out = out;
  p.M = M;
  p.H = static_cast<int>(H);
  p.nchunk = static_cast<int>(H / 16);
  p.nb = static_cast<int>(H / b);
  p.nkt = (p.nb + 3) / 4;
  p.tiled = sf_layout == FP4_SF_SWIZZLED ? 1 : 0;
  const cudaError_t err =
      launch_dequant(format == FP4_MXFP4 ? 1 : 0, p, reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(err);
    return FP4_ERR_CUDA;
  }
  return FP4_OK;
}

}  // extern "C"
