// api.cu - the C ABI of libfp4q.so (declared in include/fp4q.h): argument
// checks, launch-shape choice and dispatch to the sm_103a kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/fp4q.h"
#include "fp4q_launch.h"
#include "fused_tma.cuh"

namespace fp4q {
cudaError_t launch_fused_bf16(int fmt, const FusedShape& s, const FusedParams& p, cudaStream_t st);
cudaError_t launch_fused_fp16(int fmt, const FusedShape& s, const FusedParams& p, cudaStream_t st);
int tma_ctas_per_sm_bf16(int fmt, int cpt, int threads, size_t smem);
int tma_ctas_per_sm_fp16(int fmt, int cpt, int threads, size_t smem);

// Tuning constants of the launch-shape choice (compile-time, overridable with -D).
#ifndef FP4Q_TMA_CTA_THREADS
#define FP4Q_TMA_CTA_THREADS 256        // target threads of a TMA-kernel CTA
#endif
#ifndef FP4Q_TMA_SMEM_PER_SM
#define FP4Q_TMA_SMEM_PER_SM (220 * 1024)   // shared memory the row rings may take per SM
#endif
#ifndef FP4Q_TMA_MAX_STAGES
#define FP4Q_TMA_MAX_STAGES 6
#endif
#ifndef FP4Q_TMA_CTAS_PER_SM
#define FP4Q_TMA_CTAS_PER_SM 2          // CTAs per SM aimed for when the ring allows
#endif
#ifndef FP4Q_TMA_MIN_H
#define FP4Q_TMA_MIN_H 20480            // rows at least this wide use the TMA kernel
#endif
#ifndef FP4Q_DIRECT_CTA_THREADS
#define FP4Q_DIRECT_CTA_THREADS 128     // target threads of a direct-kernel CTA
#endif
#ifndef FP4Q_WARP_ROWS
#define FP4Q_WARP_ROWS 1                // prefer a whole row in one warp when no lane idles
#endif

static_assert(kStatusTimeout == FP4_ERR_TIMEOUT, "device and host timeout status differ");

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxChunksPerCta = 2048;   // 32768 elements held in registers by one CTA
constexpr int kMaxCluster = 8;           // portable cluster size
constexpr size_t kMaxSmemPerCta = 227 * 1024;

inline int block_of(fp4_format_t f) { return f == FP4_NVFP4 ? 16 : 32; }
inline bool valid_format(fp4_format_t f) {
  return f == FP4_NVFP4 || f == FP4_MXFP4 || f == FP4_E4M3_B32;
}
inline bool valid_layout(fp4_sf_layout_t l) {
  return l == FP4_SF_ROWMAJOR || l == FP4_SF_SWIZZLED || l == FP4_SF_BOTH;
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

int num_sms_current_device() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev].load(std::memory_order_relaxed) == 0) {
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

// Chunks per thread and slice width for `chunks` chunks: fewest idle lanes,
// ties broken in the order 2, 1, 3, 4 (fewer registers first, then more
// work per thread).  min_tpr forces whole warps where the kernel needs them.
bool pick_cpt(int chunks, int min_tpr, int* cpt_out, int* tpr_out) {
  static const int order[4] = {2, 1, 3, 4};
  int best = -1, best_tpr = 0, best_waste = 1 << 30;
  if (FP4Q_WARP_ROWS && min_tpr <= 32) {
    // a row in one warp, no idle lane: the slice reduction is shuffles only
    for (int i = 0; i < 4; ++i) {
      const int cpt = order[i];
      const int tpr = round_tpr(chunks, cpt);
      if (tpr <= 32 && tpr >= min_tpr && tpr * cpt == chunks) {
        *cpt_out = cpt;
        *tpr_out = tpr;
        return true;
      }
    }
  }
  for (int i = 0; i < 4; ++i) {
    const int cpt = order[i];
    int tpr = round_tpr(chunks, cpt);
    if (tpr < min_tpr) tpr = min_tpr;
    if (tpr > max_threads_for_cpt(cpt)) continue;
    const int waste = tpr * cpt - chunks;
    if (waste < best_waste) {
      best_waste = waste;
      best = cpt;
      best_tpr = tpr;
    }
  }
  if (best < 0) return false;
  *cpt_out = best;
  *tpr_out = best_tpr;
  return true;
}

}  // namespace

bool choose_fused_shape(int64_t M, int64_t rows, int H, int fmt, int dtype, int num_sms,
                        FusedShape* out) {
  const int nchunk = H / 16;
  // A cluster slice must be a whole number of chunks (of chunk pairs for MXFP4).
  auto splits = [&](int c) {
    return nchunk % c == 0 && (fmt == 0 || ((nchunk / c) & 1) == 0);   // fmt != 0: 32-blocks
  };
  // Cluster size: enough CTAs per row that a slice fits one CTA's registers,
  // and, for batches shorter than the SM count, enough CTAs to cover the SMs.
  int cluster = 1;
  while (nchunk / cluster > kMaxChunksPerCta) cluster <<= 1;
  if (cluster > kMaxCluster || !splits(cluster)) return false;
  while (cluster < kMaxCluster && M * cluster < num_sms && nchunk / (cluster * 2) >= 128 &&
         splits(cluster * 2))
    cluster <<= 1;

  if (cluster > 1) {
    const int per_cta = nchunk / cluster;
    int cpt, tpr;
    if (!pick_cpt(per_cta, 32, &cpt, &tpr)) return false;
    out->path = kPathDirect;
    out->cpt = cpt;
    out->tpr = tpr;
    out->rows_per_cta = 1;
    out->cluster = cluster;
    out->chunks_per_cta = per_cta;
    out->stages = 0;
    out->threads = tpr;
    out->smem = 0;
    out->grid = rows * cluster;
    return true;
  }

  if (H < FP4Q_TMA_MIN_H) {
    // Register-resident rows, several row slices per CTA.
    int cpt, tpr;
    if (!pick_cpt(nchunk, 2, &cpt, &tpr)) return false;
    int R = tpr >= FP4Q_DIRECT_CTA_THREADS ? 1 : FP4Q_DIRECT_CTA_THREADS / tpr;
    // short batches: at least one CTA per SM before rows are stacked in a CTA
    if (M < static_cast<int64_t>(R) * num_sms) {
      const int64_t fit = M / num_sms;
      R = static_cast<int>(fit < 1 ? 1 : fit);
    }
    while ((tpr * R) % 32) ++R;                           // whole warps
    if (tpr * R > max_threads_for_cpt(cpt)) return false;
    out->path = kPathDirect;
    out->cpt = cpt;
    out->tpr = tpr;
    out->rows_per_cta = R;
    out->cluster = 1;
    out->chunks_per_cta = nchunk;
    out->stages = 0;
    out->threads = tpr * R;
    out->smem = 0;
    out->grid = (rows + R - 1) / R;
    return true;
  }

  // Persistent TMA kernel.
  int cpt, tpr;
  if (!pick_cpt(nchunk, 2, &cpt, &tpr)) return false;
  int R = tpr >= FP4Q_TMA_CTA_THREADS ? 1 : FP4Q_TMA_CTA_THREADS / tpr;
  // short batches: spread rows over the SMs before stacking them in a stage
  const int64_t per_sm = (M + num_sms - 1) / num_sms;
  if (per_sm < R) R = static_cast<int>(per_sm < 1 ? 1 : per_sm);
  while ((tpr * R) % 32) ++R;               // whole warps
  if (tpr * R > max_threads_for_cpt(cpt)) return false;
  const size_t stage = 4u * static_cast<size_t>(R) * H;
  const int want_ctas = stage * FP4Q_TMA_CTAS_PER_SM <= FP4Q_TMA_SMEM_PER_SM ? FP4Q_TMA_CTAS_PER_SM : 1;
  size_t budget = FP4Q_TMA_SMEM_PER_SM / want_ctas;
  if (budget > kMaxSmemPerCta - 1024) budget = kMaxSmemPerCta - 1024;
  int S = static_cast<int>(budget / stage);
  if (S > FP4Q_TMA_MAX_STAGES) S = FP4Q_TMA_MAX_STAGES;
  if (S < 1) S = 1;
  const size_t smem = tma_smem_bytes(S, R, H);
  if (smem > kMaxSmemPerCta) return false;
  const int per = dtype == 0 ? tma_ctas_per_sm_bf16(fmt, cpt, tpr * R, smem)
                             : tma_ctas_per_sm_fp16(fmt, cpt, tpr * R, smem);
  if (per <= 0) return false;
  const int64_t groups = (rows + R - 1) / R;
  int64_t grid = static_cast<int64_t>(per) * num_sms;
  if (grid > groups) grid = groups;
  out->path = kPathTma;
  out->cpt = cpt;
  out->tpr = tpr;
  out->rows_per_cta = R;
  out->cluster = 1;
  out->chunks_per_cta = nchunk;
  out->stages = S;
  out->threads = tpr * R;
  out->smem = smem;
  out->grid = grid;
  return true;
}

cudaError_t launch_fused(int dtype, int fmt, const FusedShape& s, const FusedParams& p,
                         cudaStream_t stream) {
  return dtype == 0 ? launch_fused_bf16(fmt, s, p, stream) : launch_fused_fp16(fmt, s, p, stream);
}

int record_cuda_error(cudaError_t err) {
  if (err != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(err);
    return FP4_ERR_CUDA;
  }
  return FP4_OK;
}

int sm_count_current_device() { return num_sms_current_device(); }

#ifdef FP4Q_DEBUG_CHECKS
namespace {
std::mutex g_debug_mu;
DebugKnobs g_debug = {kWaitLimitCycles, 0, 0, -1, -1, nullptr};
}  // namespace

DebugKnobs debug_knobs() {
  std::lock_guard<std::mutex> lock(g_debug_mu);
  return g_debug;
}
#endif

}  // namespace fp4q

using namespace fp4q;

extern "C" {

int64_t fp4_sf_size_bytes(int64_t M, int64_t H, fp4_format_t format, fp4_sf_layout_t layout) {
  if (M < 0 || H <= 0) return -1;
  if (!valid_format(format)) return -1;
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
    case FP4_ERR_TIMEOUT: return "a kernel gave up on a bounded wait (timeout)";
    default: return "unknown status";
  }
}

int fp4_last_cuda_error(void) { return g_last_cuda_error; }

fp4_status_t fp4_launch_shape(int64_t M, int64_t H, fp4_dtype_t dtype, fp4_format_t format,
                              fp4_sf_layout_t sf_layout, int64_t out[8]) {
  if (!out) return FP4_ERR_INVALID_ARG;
  if (dtype != FP4_DT_BF16 && dtype != FP4_DT_FP16) return FP4_ERR_INVALID_ARG;
  if (!valid_format(format) || !valid_layout(sf_layout)) return FP4_ERR_INVALID_ARG;
  if (M <= 0 || H <= 0) return FP4_ERR_INVALID_ARG;
  const int b = block_of(format);
  if (H % b != 0 || H < 64 || H > FP4Q_MAX_H || M > INT32_MAX) return FP4_ERR_UNSUPPORTED_SHAPE;
  const int64_t rows = sf_layout == FP4_SF_ROWMAJOR ? M : (M + 127) / 128 * 128;
  FusedShape s;
  if (!choose_fused_shape(M, rows, static_cast<int>(H), static_cast<int>(format),
                          dtype == FP4_DT_BF16 ? 0 : 1, num_sms_current_device(), &s))
    return FP4_ERR_UNSUPPORTED_SHAPE;
  out[0] = s.path;
  out[1] = s.cpt;
  out[2] = s.tpr;
  out[3] = s.rows_per_cta;
  out[4] = s.cluster;
  out[5] = s.stages;
  out[6] = s.threads;
  out[7] = s.grid;
  return FP4_OK;
}

static fp4_status_t record_cuda_status(cudaError_t err) {
  return static_cast<fp4_status_t>(record_cuda_error(err));
}

// A buffer the call touches, for the overlap checks.
struct Extent {
  const void* p;
  int64_t bytes;
};

// True if any two of the non-null extents overlap.
static bool any_overlap(const Extent* e, int n) {
  for (int i = 0; i < n; ++i)
    for (int j = i + 1; j < n; ++j)
      if (e[i].p && e[j].p && overlap(e[i].p, e[i].bytes, e[j].p, e[j].bytes)) return true;
  return false;
}

// Output-side checks shared by the fused op and the standalone quantize:
// presence and alignment of the outputs.
static fp4_status_t check_outputs(fp4_sf_layout_t sf_layout, const uint8_t* out_packed,
                                  const uint8_t* out_sf, const uint8_t* out_sf_rowmajor) {
  if (!out_packed || !out_sf) return FP4_ERR_INVALID_ARG;
  if (sf_layout == FP4_SF_BOTH && !out_sf_rowmajor) return FP4_ERR_INVALID_ARG;
  if (!aligned(out_packed, 8)) return FP4_ERR_MISALIGNED;
  // padding of the tiled buffer is zeroed with 4-byte stores
  if (sf_layout != FP4_SF_ROWMAJOR && !aligned(out_sf, 4)) return FP4_ERR_MISALIGNED;
  return FP4_OK;
}

static fp4_status_t fused_call(const void* input, int64_t x_stride, void* residual,
                               int64_t r_stride, const void* weight, const float* global_scale,
                               float eps, int64_t M, int64_t H, fp4_dtype_t dtype,
                               fp4_format_t format, fp4_sf_layout_t sf_layout,
                               uint8_t* out_packed, uint8_t* out_sf, uint8_t* out_sf_rowmajor,
                               void* out_y, int32_t* status, int pdl, fp4q_stream_t stream) {
  if (dtype != FP4_DT_BF16 && dtype != FP4_DT_FP16) return FP4_ERR_INVALID_ARG;
  if (!valid_format(format) || !valid_layout(sf_layout)) return FP4_ERR_INVALID_ARG;
  if (M < 0 || H <= 0 || !(eps >= 0.0f)) return FP4_ERR_INVALID_ARG;
  if (x_stride == 0) x_stride = H;
  if (r_stride == 0) r_stride = H;
  if (x_stride < H || r_stride < H) return FP4_ERR_INVALID_ARG;
  const int b = block_of(format);
  if (H % b != 0 || H < 64 || H > FP4Q_MAX_H) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FP4_OK;
  if (M > INT32_MAX) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (!input || !residual || !weight) return FP4_ERR_INVALID_ARG;
  // rows start on 32-byte boundaries (256-bit accesses, bulk copies)
  if (!aligned(input, 32) || !aligned(residual, 32) || !aligned(weight, 32) ||
      !aligned(global_scale, 4) || !aligned(out_y, 32) || !aligned(status, 4) ||
      x_stride % 16 || r_stride % 16)
    return FP4_ERR_MISALIGNED;
  const fp4_status_t st = check_outputs(sf_layout, out_packed, out_sf, out_sf_rowmajor);
  if (st != FP4_OK) return st;
  // Nothing the call writes may overlap anything else it reads or writes.
  // The input and the weight are only read, so they may share memory with
  // each other (and the global scale with either).
  const int64_t x_bytes = ((M - 1) * x_stride + H) * 2;
  const int64_t r_bytes = ((M - 1) * r_stride + H) * 2;
  const int64_t nb = H / b;
  const Extent writes[] = {{residual, r_bytes},
                           {out_packed, M * H / 2},
                           {out_sf, fp4_sf_size_bytes(M, H, format, sf_layout)},
                           {sf_layout == FP4_SF_BOTH ? out_sf_rowmajor : nullptr, M * nb},
                           {out_y, M * H * 2},
                           {status, 4}};
  constexpr int kWrites = sizeof(writes) / sizeof(writes[0]);
  if (any_overlap(writes, kWrites)) return FP4_ERR_INVALID_ARG;
  const Extent reads[] = {{input, x_bytes}, {weight, H * 2}, {global_scale, 4}};
  for (const Extent& w : writes)
    for (const Extent& r : reads)
      if (w.p && r.p && overlap(w.p, w.bytes, r.p, r.bytes)) return FP4_ERR_INVALID_ARG;

  FusedShape shape;
  const int64_t rows = sf_layout == FP4_SF_ROWMAJOR ? M : (M + 127) / 128 * 128;
  if (!choose_fused_shape(M, rows, static_cast<int>(H), static_cast<int>(format),
                          dtype == FP4_DT_BF16 ? 0 : 1, num_sms_current_device(), &shape))
    return FP4_ERR_UNSUPPORTED_SHAPE;
  if (shape.grid > INT32_MAX) return FP4_ERR_UNSUPPORTED_SHAPE;
  // the TMA ring copies a stage's rows in one piece: strided rows need one row per stage
  if (shape.path == kPathTma && shape.rows_per_cta > 1 && (x_stride != H || r_stride != H))
    return FP4_ERR_UNSUPPORTED_SHAPE;

  FusedParams p{};
  p.x = input;
  p.r = residual;
  p.w = weight;
  p.packed = out_packed;
  p.sf_tiled = (sf_layout == FP4_SF_ROWMAJOR) ? nullptr : out_sf;
  p.sf_rm = (sf_layout == FP4_SF_ROWMAJOR) ? out_sf
            : (sf_layout == FP4_SF_BOTH)   ? out_sf_rowmajor
                                           : nullptr;
  p.gs = global_scale;
  p.y = out_y;
  p.status = status;
  p.x_stride = x_stride;
  p.r_stride = r_stride;
  p.eps = eps;
  p.M = M;
  p.rows = rows;
  p.H = static_cast<int>(H);
  p.nchunk = static_cast<int>(H / 16);
  p.nb = static_cast<int>(H / b);
  p.nkt = (p.nb + 3) / 4;
  p.tpr = shape.tpr;
  p.rows_per_cta = shape.rows_per_cta;
  p.cluster = shape.cluster;
  p.chunks_per_cta = shape.chunks_per_cta;
  p.stages = shape.stages;
  p.groups = (rows + shape.rows_per_cta - 1) / shape.rows_per_cta;
  FP4Q_SET_DEBUG(p);

  shape.pdl = pdl ? 1 : 0;
  // cudaLaunchKernelEx reports this launch's own errors; the thread's sticky
  // last error (which may belong to the caller) is left alone
  return record_cuda_status(launch_fused(dtype == FP4_DT_BF16 ? 0 : 1, static_cast<int>(format),
                                         shape, p, reinterpret_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_add_rmsnorm_quant(const void* input, void* residual, const void* weight,
                                   float eps, int64_t M, int64_t H, fp4_dtype_t dtype,
                                   fp4_format_t format, fp4_sf_layout_t sf_layout,
                                   uint8_t* out_packed, uint8_t* out_sf,
                                   uint8_t* out_sf_rowmajor, fp4q_stream_t stream) {
  return fused_call(input, H, residual, H, weight, nullptr, eps, M, H, dtype, format, sf_layout,
                    out_packed, out_sf, out_sf_rowmajor, nullptr, nullptr, 0, stream);
}

fp4_status_t fp4_add_rmsnorm_quant_gs(const void* input, void* residual, const void* weight,
                                      const float* global_scale, float eps, int64_t M,
                                      int64_t H, fp4_dtype_t dtype, fp4_format_t format,
                                      fp4_sf_layout_t sf_layout, uint8_t* out_packed,
                                      uint8_t* out_sf, uint8_t* out_sf_rowmajor,
                                      fp4q_stream_t stream) {
  return fused_call(input, H, residual, H, weight, global_scale, eps, M, H, dtype, format,
                    sf_layout, out_packed, out_sf, out_sf_rowmajor, nullptr, nullptr, 0, stream);
}

fp4_status_t fp4_add_rmsnorm_quant_ex(const void* input, int64_t input_row_stride,
                                      void* residual, int64_t residual_row_stride,
                                      const void* weight, const float* global_scale, float eps,
                                      int64_t M, int64_t H, fp4_dtype_t dtype,
                                      fp4_format_t format, fp4_sf_layout_t sf_layout,
                                      uint8_t* out_packed, uint8_t* out_sf,
                                      uint8_t* out_sf_rowmajor, void* out_y, int32_t* status,
                                      int pdl, fp4q_stream_t stream) {
  return fused_call(input, input_row_stride, residual, residual_row_stride, weight, global_scale,
                    eps, M, H, dtype, format, sf_layout, out_packed, out_sf, out_sf_rowmajor,
                    out_y, status, pdl, stream);
}

fp4_status_t fp4_quantize(const void* input, const float* global_scale, int64_t M, int64_t H,
                          fp4_dtype_t dtype, fp4_format_t format, fp4_sf_layout_t sf_layout,
                          uint8_t* out_packed, uint8_t* out_sf, uint8_t* out_sf_rowmajor, int pdl,
                          fp4q_stream_t stream) {
  if (dtype != FP4_DT_BF16 && dtype != FP4_DT_FP16) return FP4_ERR_INVALID_ARG;
  if (!valid_format(format) || !valid_layout(sf_layout)) return FP4_ERR_INVALID_ARG;
  if (M < 0 || H <= 0) return FP4_ERR_INVALID_ARG;
  const int b = block_of(format);
  if (H % b != 0 || H > INT32_MAX / 2) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FP4_OK;
  if (!input) return FP4_ERR_INVALID_ARG;
  if (!aligned(input, 32) || !aligned(global_scale, 4)) return FP4_ERR_MISALIGNED;
  const fp4_status_t st = check_outputs(sf_layout, out_packed, out_sf, out_sf_rowmajor);
  if (st != FP4_OK) return st;
  const Extent writes[] = {{out_packed, M * H / 2},
                           {out_sf, fp4_sf_size_bytes(M, H, format, sf_layout)},
                           {sf_layout == FP4_SF_BOTH ? out_sf_rowmajor : nullptr, M * (H / b)}};
  if (any_overlap(writes, 3)) return FP4_ERR_INVALID_ARG;
  for (const Extent& w : writes)
    if (w.p && (overlap(w.p, w.bytes, input, M * H * 2) ||
                (global_scale && overlap(w.p, w.bytes, global_scale, 4))))
      return FP4_ERR_INVALID_ARG;
  QuantParams p{};
  p.x = input;
  p.packed = out_packed;
  p.sf_tiled = (sf_layout == FP4_SF_ROWMAJOR) ? nullptr : out_sf;
  p.sf_rm = (sf_layout == FP4_SF_ROWMAJOR) ? out_sf
            : (sf_layout == FP4_SF_BOTH)   ? out_sf_rowmajor
                                           : nullptr;
  p.gs = global_scale;
  p.M = M;
  p.rows = sf_layout == FP4_SF_ROWMAJOR ? M : (M + 127) / 128 * 128;
  p.H = static_cast<int>(H);
  p.nchunk = static_cast<int>(H / 16);
  p.nb = static_cast<int>(H / b);
  p.nkt = (p.nb + 3) / 4;
  FP4Q_SET_DEBUG(p);
  return record_cuda_status(launch_quantize(dtype == FP4_DT_BF16 ? 0 : 1, static_cast<int>(format), p,
                                            pdl, reinterpret_cast<cudaStream_t>(stream)));
}

int fp4_debug_build(void) {
#ifdef FP4Q_DEBUG_CHECKS
  return 1;
#else
  return 0;
#endif
}

fp4_status_t fp4_debug_configure(int64_t wait_limit_cycles, int64_t shrink_bytes, int drop_kernel,
                                 int drop_cta, int drop_iter, uint32_t* violations) {
#ifdef FP4Q_DEBUG_CHECKS
  if (wait_limit_cycles <= 0 || shrink_bytes < 0 || drop_kernel < 0 || drop_kernel > 2)
    return FP4_ERR_INVALID_ARG;
  if (violations && !aligned(violations, 4)) return FP4_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_debug_mu);
  g_debug = DebugKnobs{wait_limit_cycles, shrink_bytes, drop_kernel, drop_cta, drop_iter,
                       reinterpret_cast<unsigned int*>(violations)};
  return FP4_OK;
#else
  (void)wait_limit_cycles; (void)shrink_bytes; (void)drop_kernel; (void)drop_cta;
  (void)drop_iter; (void)violations;
  return FP4_ERR_INVALID_ARG;   // the knobs exist in the debug build only
#endif
}

fp4_status_t fp4_read_device_status(const int32_t* status, fp4q_stream_t stream) {
  if (!status || !aligned(status, 4)) return FP4_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  int32_t v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda_status(e);
  return v == FP4_OK || v == FP4_ERR_TIMEOUT ? static_cast<fp4_status_t>(v) : FP4_ERR_INVALID_ARG;
}

fp4_status_t fp4_dequant(const uint8_t* packed, const uint8_t* sf, int64_t M, int64_t H,
                         fp4_format_t format, fp4_sf_layout_t sf_layout, float* out,
                         fp4q_stream_t stream) {
  if (!valid_format(format)) return FP4_ERR_INVALID_ARG;
  if (sf_layout != FP4_SF_ROWMAJOR && sf_layout != FP4_SF_SWIZZLED) return FP4_ERR_INVALID_ARG;
  if (M < 0 || H <= 0) return FP4_ERR_INVALID_ARG;
  const int b = block_of(format);
  if (H % b != 0 || H > INT32_MAX / 2) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FP4_OK;
  if (!packed || !sf || !out) return FP4_ERR_INVALID_ARG;
  if (!aligned(packed, 8) || !aligned(out, 16)) return FP4_ERR_MISALIGNED;
  DequantParams p{};
  p.packed = packed;
  p.sf = sf;
  p.out = out;
  p.M = M;
  p.H = static_cast<int>(H);
  p.nchunk = static_cast<int>(H / 16);
  p.nb = static_cast<int>(H / b);
  p.nkt = (p.nb + 3) / 4;
  p.tiled = sf_layout == FP4_SF_SWIZZLED ? 1 : 0;
  return record_cuda_status(
      launch_dequant(static_cast<int>(format), p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
