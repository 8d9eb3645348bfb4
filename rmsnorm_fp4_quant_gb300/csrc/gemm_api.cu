// gemm_api.cu - the C entry point of the NVFP4 GEMM (declared in
// include/fp4q.h): argument checks and the choice of tile schedule; the
// kernels are in gemm_nvfp4.cu.
#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>

#include "../../include/fp4q.h"
#include "fp4q_launch.h"
#include "gemm_launch.h"

// Tuning constants of the schedule choice (compile-time, overridable with -D).
#ifndef FP4Q_GEMM_STAGES
#define FP4Q_GEMM_STAGES 3              // GEMM shared-memory ring depth (2 CTAs per SM at 3)
#endif
#ifndef FP4Q_GEMM_VARIANT
#define FP4Q_GEMM_VARIANT 0             // the GEMM schedule of the automatic choice
#endif
#ifndef FP4Q_GEMM_PSTAGES_128
#define FP4Q_GEMM_PSTAGES_128 3         // ring depth of the persistent 128-wide schedule
#endif                                  // (2 CTAs per SM at 3)
#ifndef FP4Q_GEMM_PSTAGES_256
#define FP4Q_GEMM_PSTAGES_256 4         // ring depth of the persistent 256-wide schedule
#endif

using namespace fp4q;

namespace {

// The schedule of an M x N x K product: `variant` if given (>= 0), else the
// automatic choice.  Measured on the decode shapes: with up to 6 K blocks a
// single CTA per tile holding them all in flight is faster than a split; with
// 24 the split wins by a third.  Measured on an 8192 x 7168 x 7168 product:
// with more tiles than two CTAs per SM take at once, persistent CTAs that load
// the next tile during the epilogue run 2.5 % (NVFP4) to 2.7 % (MXFP4) faster
// than one CTA per tile.
int choose_variant(int64_t M, int64_t N, int64_t K, bool fp4_out, int variant, int sms) {
  if (variant >= 0) return variant;
  const int64_t tiles128 = ((N + 127) / 128) * ((M + 127) / 128);
  const int64_t num_kb = (K + 255) / 256;
  if (tiles128 * 2 <= sms && num_kb > 6 && !fp4_out) return 4;
  // many tiles: the 256-wide persistent schedule (8192 x 7168 x 7168: 202 us
  // against 219 us for the 128-wide one, NVFP4; 201 against 206 us, MXFP4)
  if (tiles128 > 2 * static_cast<int64_t>(sms)) return 3;
  return FP4Q_GEMM_VARIANT;
}

// Every form: NVFP4 (mx = false) or MXFP4 operands; epilogue kEpiPlain /
// kEpiGelu into `out` (bf16), or kEpiGeluFp4 into out_packed + out_sf.
fp4_status_t gemm_call(bool mx, int epilogue, const uint8_t* a_packed, const uint8_t* b_packed,
                       const uint8_t* sfa, const uint8_t* sfb, float alpha, const void* bias,
                       const void* residual, int64_t M, int64_t N, int64_t K, void* out,
                       uint8_t* out_packed, uint8_t* out_sf, int variant, int pdl,
                       int32_t* status, fp4q_stream_t stream) {
  const bool fp4_out = epilogue == kEpiGeluFp4;
  if (M < 0 || N < 0 || K <= 0) return FP4_ERR_INVALID_ARG;
  if (variant < -1 || variant > 4) return FP4_ERR_INVALID_ARG;
  if (pdl < 0 || pdl > 2) return FP4_ERR_INVALID_ARG;
  if (fp4_out && variant == 4) return FP4_ERR_INVALID_ARG;   // split K stores 8-column groups
  if (K % 32 != 0 || N % (fp4_out ? 16 : 8) != 0) return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX - 128 || N > INT32_MAX - 128 || K > INT32_MAX / 2)
    return FP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return FP4_OK;
  if (!a_packed || !b_packed || !sfa || !sfb) return FP4_ERR_INVALID_ARG;
  if (fp4_out ? (!out_packed || !out_sf) : !out) return FP4_ERR_INVALID_ARG;
  for (const void* ptr : {static_cast<const void*>(a_packed), static_cast<const void*>(b_packed),
                          static_cast<const void*>(sfa), static_cast<const void*>(sfb),
                          static_cast<const void*>(out), bias, residual,
                          static_cast<const void*>(out_packed)})
    if (!abi_aligned(ptr, 16)) return FP4_ERR_MISALIGNED;
  if (fp4_out) {
    const int64_t pk = M * N / 2;
    const int64_t sfo = fp4_sf_size_bytes(M, N, FP4_NVFP4, FP4_SF_SWIZZLED);
    const void* ins[4] = {a_packed, b_packed, sfa, sfb};
    const int64_t in_bytes[4] = {M * K / 2, N * K / 2,
                                 fp4_sf_size_bytes(M, K, FP4_NVFP4, FP4_SF_SWIZZLED),
                                 fp4_sf_size_bytes(N, K, FP4_NVFP4, FP4_SF_SWIZZLED)};
    if (abi_overlap(out_packed, pk, out_sf, sfo)) return FP4_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
      if (abi_overlap(out_packed, pk, ins[i], in_bytes[i]) ||
          abi_overlap(out_sf, sfo, ins[i], in_bytes[i]))
        return FP4_ERR_INVALID_ARG;
    if (bias && (abi_overlap(out_packed, pk, bias, N * 2) || abi_overlap(out_sf, sfo, bias, N * 2)))
      return FP4_ERR_INVALID_ARG;
  }
  const int64_t out_bytes = fp4_out ? 0 : M * N * 2;
  const fp4_format_t fmt = mx ? FP4_MXFP4 : FP4_NVFP4;
  const int64_t sfa_bytes = fp4_sf_size_bytes(M, K, fmt, FP4_SF_SWIZZLED);
  const int64_t sfb_bytes = fp4_sf_size_bytes(N, K, fmt, FP4_SF_SWIZZLED);
  if (abi_overlap(out, out_bytes, a_packed, M * K / 2) ||
      abi_overlap(out, out_bytes, b_packed, N * K / 2) ||
      abi_overlap(out, out_bytes, sfa, sfa_bytes) || abi_overlap(out, out_bytes, sfb, sfb_bytes) ||
      (bias && abi_overlap(out, out_bytes, bias, N * 2)))
    return FP4_ERR_INVALID_ARG;
  // the residual may be the output itself (each element is read, then written,
  // by the same thread), but not partly overlap it
  if (residual && residual != out && abi_overlap(out, out_bytes, residual, out_bytes))
    return FP4_ERR_INVALID_ARG;
  if (status) {   // the status word overlaps nothing else the call touches
    if (!abi_aligned(status, 4)) return FP4_ERR_MISALIGNED;
    const void* bufs[9] = {a_packed, b_packed, sfa, sfb, bias, residual, out, out_packed, out_sf};
    const int64_t sizes[9] = {M * K / 2, N * K / 2, sfa_bytes, sfb_bytes, N * 2, M * N * 2,
                              out_bytes, fp4_out ? M * N / 2 : 0,
                              fp4_out ? fp4_sf_size_bytes(M, N, FP4_NVFP4, FP4_SF_SWIZZLED) : 0};
    for (int i = 0; i < 9; ++i)
      if (bufs[i] && abi_overlap(status, 4, bufs[i], sizes[i])) return FP4_ERR_INVALID_ARG;
  }
  GemmParams p{};
  p.sfa = sfa;
  p.sfb = sfb;
  p.bias = static_cast<const uint16_t*>(bias);
  p.residual = static_cast<const uint16_t*>(residual);
  p.out = static_cast<uint16_t*>(out);
  p.out_packed = out_packed;
  p.out_sf = out_sf;
  p.status = reinterpret_cast<int*>(status);
  p.epilogue = epilogue;
  p.out_nkt = static_cast<int>((N / 16 + 3) / 4);
  p.rows_out = static_cast<int>(fp4_out ? (M + 127) / 128 * 128 : M);
  p.alpha = alpha;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  // few output tiles (short, wide products such as decode steps): split the K
  // loop of each tile over a cluster of CTAs so that most SMs take part
  const int sms = sm_count_current_device();
  const int64_t tiles128 = ((N + 127) / 128) * ((M + 127) / 128);
  const int num_kb = static_cast<int>((K + 255) / 256);
  const int v = choose_variant(M, N, K, fp4_out, variant, sms);
  const int bn = (v == 1 || v == 3) ? 256 : 128;
  const bool persistent = v == 2 || v == 3;
  p.stages = !persistent ? FP4Q_GEMM_STAGES : bn == 128 ? FP4Q_GEMM_PSTAGES_128
                                                        : FP4Q_GEMM_PSTAGES_256;
  p.split = 1;
  p.b_static = pdl == 2 ? 1 : 0;
  if (v == 4) {
    int64_t sk = tiles128 > 0 ? sms / tiles128 : 1;
    if (sk > 16) sk = 16;
    if (sk > num_kb) sk = num_kb;
    p.split = sk < 2 ? 2 : static_cast<int>(sk);
    if (p.split > num_kb) p.split = 1;
  }
  // a single wave of one-tile CTAs: let each CTA have all (up to 6) of its K
  // blocks in flight at once instead of sharing its SM with a second CTA
  if (!persistent && bn == 128) {
    const int64_t ctas = tiles128 * p.split;
    const int kb_per_cta = (num_kb + p.split - 1) / p.split;
    if (ctas <= sms && kb_per_cta > p.stages) p.stages = kb_per_cta < 6 ? kb_per_cta : 6;
  }
  p.nkt = 0;        // filled by the launcher
  p.num_kb = 0;
  p.tmem_cols = 0;
  FP4Q_SET_DEBUG(p);
  cudaError_t e = launch_gemm_nvfp4(a_packed, b_packed, p, bn, persistent, mx, pdl,
                                    reinterpret_cast<cudaStream_t>(stream));
  // a cluster of this many CTAs may not fit: halve it until one does
  while (e == cudaErrorInvalidConfiguration && p.split > 2) {
    p.split /= 2;
    e = launch_gemm_nvfp4(a_packed, b_packed, p, bn, persistent, mx, pdl,
                          reinterpret_cast<cudaStream_t>(stream));
  }
  return static_cast<fp4_status_t>(record_cuda_error(e));
}

}  // namespace

extern "C" {

fp4_status_t fp4_gemm_nvfp4_bf16(const uint8_t* a_packed, const uint8_t* b_packed,
                                 const uint8_t* sfa, const uint8_t* sfb, float alpha,
                                 const void* bias, const void* residual, int64_t M, int64_t N,
                                 int64_t K, void* out, int variant, int pdl,
                                 fp4q_stream_t stream) {
  return gemm_call(false, kEpiPlain, a_packed, b_packed, sfa, sfb, alpha, bias, residual, M, N,
                   K, out, nullptr, nullptr, variant, pdl, nullptr, stream);
}

fp4_status_t fp4_gemm_mxfp4_bf16(const uint8_t* a_packed, const uint8_t* b_packed,
                                 const uint8_t* sfa, const uint8_t* sfb, float alpha,
                                 const void* bias, const void* residual, int64_t M, int64_t N,
                                 int64_t K, void* out, int variant, int pdl,
                                 fp4q_stream_t stream) {
  return gemm_call(true, kEpiPlain, a_packed, b_packed, sfa, sfb, alpha, bias, residual, M, N, K,
                   out, nullptr, nullptr, variant, pdl, nullptr, stream);
}

fp4_status_t fp4_gemm_nvfp4_gelu_bf16(const uint8_t* a_packed, const uint8_t* b_packed,
                                      const uint8_t* sfa, const uint8_t* sfb, float alpha,
                                      const void* bias, int64_t M, int64_t N, int64_t K,
                                      void* out, int variant, int pdl, fp4q_stream_t stream) {
  return gemm_call(false, kEpiGelu, a_packed, b_packed, sfa, sfb, alpha, bias, nullptr, M, N, K,
                   out, nullptr, nullptr, variant, pdl, nullptr, stream);
}

fp4_status_t fp4_gemm_nvfp4_gelu_nvfp4(const uint8_t* a_packed, const uint8_t* b_packed,
                                       const uint8_t* sfa, const uint8_t* sfb, float alpha,
                                       const void* bias, int64_t M, int64_t N, int64_t K,
                                       uint8_t* out_packed, uint8_t* out_sf, int variant,
                                       int pdl, fp4q_stream_t stream) {
  return gemm_call(false, kEpiGeluFp4, a_packed, b_packed, sfa, sfb, alpha, bias, nullptr, M, N,
                   K, nullptr, out_packed, out_sf, variant, pdl, nullptr, stream);
}

fp4_status_t fp4_gemm_ex(const uint8_t* a_packed, const uint8_t* b_packed, const uint8_t* sfa,
                         const uint8_t* sfb, fp4_format_t format, fp4_epilogue_t epilogue,
                         float alpha, const void* bias, const void* residual, int64_t M,
                         int64_t N, int64_t K, void* out, uint8_t* out_packed, uint8_t* out_sf,
                         int variant, int pdl, int32_t* status, fp4q_stream_t stream) {
  if (format != FP4_NVFP4 && format != FP4_MXFP4) return FP4_ERR_INVALID_ARG;
  const bool mx = format == FP4_MXFP4;
  switch (epilogue) {
    case FP4_EPI_BF16:
      return gemm_call(mx, kEpiPlain, a_packed, b_packed, sfa, sfb, alpha, bias, residual, M, N,
                       K, out, nullptr, nullptr, variant, pdl, status, stream);
    case FP4_EPI_GELU_BF16:
      if (residual) return FP4_ERR_INVALID_ARG;
      return gemm_call(mx, kEpiGelu, a_packed, b_packed, sfa, sfb, alpha, bias, nullptr, M, N, K,
                       out, nullptr, nullptr, variant, pdl, status, stream);
    case FP4_EPI_GELU_NVFP4:
      if (mx || residual) return FP4_ERR_INVALID_ARG;
      return gemm_call(false, kEpiGeluFp4, a_packed, b_packed, sfa, sfb, alpha, bias, nullptr, M,
                       N, K, nullptr, out_packed, out_sf, variant, pdl, status, stream);
    default:
      return FP4_ERR_INVALID_ARG;
  }
}

int fp4_gemm_variant(int64_t M, int64_t N, int64_t K, fp4_format_t format, int fp4_out,
                     int variant) {
  if (format != FP4_NVFP4 && format != FP4_MXFP4) return -1;
  const bool mx = format == FP4_MXFP4;
  if (M < 0 || N < 0 || K <= 0 || variant < -1 || variant > 4) return -1;
  if (fp4_out && (mx || variant == 4)) return -1;
  if (K % 32 != 0 || N % (fp4_out ? 16 : 8) != 0) return -1;
  if (M > INT32_MAX - 128 || N > INT32_MAX - 128 || K > INT32_MAX / 2) return -1;
  return choose_variant(M, N, K, fp4_out != 0, variant, sm_count_current_device());
}

}  // extern "C"
