/*
 * fp4q.h - C ABI of the GB300 (sm_103a) fused residual-add + RMSNorm +
 * block-scaled FP4 quantization library (libfp4q.so).
 *
 * The operation is the one on the FlashInfer page `add_rmsnorm_fp4quant.py`
 * (module docstring; `AddRMSNormFP4QuantKernel.kernel` phases 1-3;
 * `add_rmsnorm_fp4quant` Parameters / Returns / Notes).  Per row m of an
 * M x H batch, with b = 16 (NVFP4) or 32 (MXFP4), nb = H / b:
 *
 *   h        = round_dtype(float(input) + float(residual))   -> residual (in place)
 *   rstd     = 1 / sqrt(sum(h^2) / H + eps)                   (fp32, each op rounded)
 *   y        = (h * weight) * rstd                            (fp32: h * weight is exact,
 *                                                              so y is rounded once)
 *   per block of b elements (amax = max |y| over the block):
 *     NVFP4: scale = E4M3 nearest-even of min(amax / 6, 448)
 *     MXFP4: scale = UE8M0, the power of two at or above amax / 6
 *     code  = E2M1 nearest-even of y * rn(1 / scale) on {0,.5,1,1.5,2,3,4,6},
 *             saturating, sign in bit 3 (the page's kernel scales by the
 *             reciprocal of the decoded scale); a zero scale gives zero codes
 *   out_packed[m, j] = code[2j] | code[2j+1] << 4
 *
 * Scale layouts (same page, `is_sf_swizzled_layout`, `output_both_sf_layouts`):
 *   row-major : sf[m * nb + k]
 *   tiled     : sf[(m/128)*nkt*512 + (k/4)*512 + (m%32)*16 + ((m%128)/32)*4 + k%4],
 *               nkt = ceil(nb / 4), buffer = ceil(M/128) * nkt * 512 bytes, every
 *               padding byte (rows >= M, k >= nb) written 0.  This is the scale
 *               layout the FlashRT `fp4-gemm` README (Tensor Contract) names as
 *               the CUTLASS SFA input of its NVFP4 GEMM.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing and keeps no state between calls.
 *   - Tensors are dense row-major (row stride = H elements / H/2 bytes).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream);
 *     argument errors are detected on the host before anything is launched.
 *   - Status codes, never exceptions or aborts.
 */
#ifndef FP4Q_H_
#define FP4Q_H_

#include <stdint.h>

/* Only the entry points below are exported from libfp4q.so (built with hidden
 * visibility). */
#if defined(__GNUC__)
#define FP4Q_API __attribute__((visibility("default")))
#else
#define FP4Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t / CUstream. */
typedef struct CUstream_st* fp4q_stream_t;

typedef enum { FP4_DT_BF16 = 0, FP4_DT_FP16 = 1 } fp4_dtype_t;

/* NVFP4: 16-element blocks, E4M3 scale bytes.  MXFP4: 32-element blocks,
 * UE8M0 scale bytes.  E4M3_B32: 32-element blocks with E4M3 scale bytes
 * (FlashInfer page, `block_size` / `scale_format`: "e4m3" on the block-32
 * branch).  A global scale applies to the two E4M3 formats only. */
typedef enum { FP4_NVFP4 = 0, FP4_MXFP4 = 1, FP4_E4M3_B32 = 2 } fp4_format_t;

typedef enum {
  FP4_SF_ROWMAJOR = 0, /* (M, nb) bytes                                  */
  FP4_SF_SWIZZLED = 1, /* 128x4 tiled, padded to whole tiles             */
  FP4_SF_BOTH = 2      /* tiled into out_sf AND row-major into out_sf_rowmajor */
} fp4_sf_layout_t;

typedef enum {
  FP4_OK = 0,
  FP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, negative size, overlap */
  FP4_ERR_UNSUPPORTED_SHAPE = 2, /* H % b != 0, H < 64, or H above the maximum     */
  FP4_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment rule below       */
  FP4_ERR_CUDA = 4,              /* the CUDA runtime reported an error on launch    */
  FP4_ERR_TIMEOUT = 5            /* a kernel gave up on a bounded wait (device status word) */
} fp4_status_t;

/*
 * Device status word.  The kernels that wait on asynchronous copies (the
 * wide-row fused kernel, which streams rows through a shared-memory ring
 * filled by the copy engine, and every GEMM schedule) bound each wait at about
 * one second of clock cycles.  A CTA whose wait runs out does not hang or
 * trap: it stops, marks what it could not compute and returns, and the
 * context stays usable.  The calls that take an optional `status` (a DEVICE
 * pointer to one int32_t owned by the caller) then store FP4_ERR_TIMEOUT
 * there.  The library never writes anything else to it and never clears it:
 * zero it before the call, synchronise, and read it (fp4_read_device_status
 * does the last two).  What a timed-out call leaves behind:
 *   fused op: every scale byte of the rows the CTA did not finish is 0xFF
 *             (NaN in E4M3 and in UE8M0); their codes, residual rows and y
 *             rows are unspecified (the residual row may be the old value);
 *   GEMM:     the output tiles of the CTA are NaN (bf16 out), or their scale
 *             bytes 0xFF (NVFP4 out).
 * The host-side return value of the call itself only reports what is known
 * at launch (FP4_OK once the launch succeeded).
 */

/* Largest supported H: one CTA holds up to 32768 elements of a row in
 * registers and a thread-block cluster of up to 8 CTAs shares one row.  Above
 * 32768, H / 16 must split evenly over the cluster (over chunk pairs for MXFP4). */
#define FP4Q_MAX_H 262144

/*
 * fp4_add_rmsnorm_quant - the fused op (FlashInfer page, `add_rmsnorm_fp4quant`).
 *
 *   input           [M, H] dtype, read only.                      32-byte aligned.
 *   residual        [M, H] dtype, read then overwritten with h.   32-byte aligned.
 *   weight          [H]    dtype, read only.                      32-byte aligned.
 *   eps             added to the mean of squares (fp32).
 *   M               rows, >= 0 (M == 0: nothing is launched, FP4_OK).
 *   H               hidden size: multiple of the block size, 64 <= H <= FP4Q_MAX_H.
 *   out_packed      [M, H/2] bytes, two E2M1 codes per byte.       8-byte aligned.
 *   out_sf          row-major scales (FP4_SF_ROWMAJOR) or the tiled buffer
 *                   (FP4_SF_SWIZZLED / FP4_SF_BOTH, 4-byte aligned); size from
 *                   fp4_sf_size_bytes.
 *   out_sf_rowmajor row-major scales for FP4_SF_BOTH, else ignored (may be NULL).
 *
 * input must not overlap residual; outputs must not overlap inputs or each
 * other.  Global scale is 1 (the page's default when none is given).
 */
FP4Q_API fp4_status_t fp4_add_rmsnorm_quant(const void* input, void* residual, const void* weight,
                                            float eps, int64_t M, int64_t H, fp4_dtype_t dtype,
                                            fp4_format_t format, fp4_sf_layout_t sf_layout,
                                            uint8_t* out_packed, uint8_t* out_sf,
                                            uint8_t* out_sf_rowmajor, fp4q_stream_t stream);

/*
 * fp4_add_rmsnorm_quant_gs - fp4_add_rmsnorm_quant with a device-resident
 * global scale (FlashInfer page, `global_scale`; read on the device, so a
 * captured CUDA graph picks up a new value).  global_scale: DEVICE pointer to
 * one positive finite fp32, or NULL for 1.  For the E4M3 formats each block
 * scale becomes E4M3(min(gs * amax / 6, 448)) and codes round from
 * y * rn(rn(1 / scale) * gs) (so dequantised values are y * gs: a consumer divides by gs,
 * e.g. gs = 448 * 6 / max|y| fills the E4M3 range); UE8M0 scales ignore it.
 * All other arguments as fp4_add_rmsnorm_quant.
 */
FP4Q_API fp4_status_t fp4_add_rmsnorm_quant_gs(const void* input, void* residual, const void* weight,
                                               const float* global_scale, float eps, int64_t M,
                                               int64_t H, fp4_dtype_t dtype, fp4_format_t format,
                                               fp4_sf_layout_t sf_layout, uint8_t* out_packed,
                                               uint8_t* out_sf, uint8_t* out_sf_rowmajor,
                                               fp4q_stream_t stream);

/*
 * fp4_add_rmsnorm_quant_ex - the general form of the fused op: strided rows,
 * an optional y output, a device status word and programmatic dependent
 * launch (API variants of the FlashInfer page's `add_rmsnorm_fp4quant`,
 * which views 3-D input as 2-D rows).
 *
 *   input_row_stride, residual_row_stride  elements between consecutive rows
 *                  (0 = H); >= H and a multiple of 16 (rows start 32-byte
 *                  aligned).  Outputs stay dense.
 *   out_y          [M, H] dtype, dense, 32-byte aligned, or NULL: receives y =
 *                  (h * w) * rstd rounded to the storage dtype (the value the
 *                  codes quantize), for consumers that want it unquantized.
 *   global_scale   as in fp4_add_rmsnorm_quant_gs (NULL = 1).
 *   status         DEVICE int32_t, 4-byte aligned, or NULL: receives
 *                  FP4_ERR_TIMEOUT if a bounded wait ran out (see "Device
 *                  status word" above); left untouched otherwise.
 *   pdl            nonzero: launched as a programmatic dependent of the kernel
 *                  before it on `stream` (e.g. the GEMM that produced `input`),
 *                  so the launch overlaps that kernel's tail; the kernel waits
 *                  for its results before reading anything.  Every kernel of
 *                  this library lets its own dependents launch once its CTAs
 *                  have issued their loads.
 * Everything else as fp4_add_rmsnorm_quant; the outputs, y and status must
 * not overlap the inputs or each other.
 */
FP4Q_API fp4_status_t fp4_add_rmsnorm_quant_ex(const void* input, int64_t input_row_stride,
                                               void* residual, int64_t residual_row_stride,
                                               const void* weight, const float* global_scale, float eps,
                                               int64_t M, int64_t H, fp4_dtype_t dtype,
                                               fp4_format_t format, fp4_sf_layout_t sf_layout,
                                               uint8_t* out_packed, uint8_t* out_sf,
                                               uint8_t* out_sf_rowmajor, void* out_y,
                                               int32_t* status, int pdl, fp4q_stream_t stream);

/*
 * fp4_quantize - block quantization of `input` [M, H] itself, without the
 * residual add and the normalisation: the standalone producer of packed E2M1
 * plus scales (FlashRT `fp4-gemm` README, `quantize_fp4_sfa_bf16` /
 * `quantize_fp4_sfa_fp16`).  The same layouts serve as the GEMM's A-operand
 * scales (rows = M) or B-operand scales (rows = N).  input 32-byte aligned,
 * H a multiple of the block size (>= 16); global_scale as in
 * fp4_add_rmsnorm_quant_gs; outputs as fp4_add_rmsnorm_quant; pdl as in
 * fp4_add_rmsnorm_quant_ex (launched as a programmatic dependent of the
 * kernel before it on `stream`, e.g. the kernel that produced `input`).
 */
FP4Q_API fp4_status_t fp4_quantize(const void* input, const float* global_scale, int64_t M, int64_t H,
                                   fp4_dtype_t dtype, fp4_format_t format, fp4_sf_layout_t sf_layout,
                                   uint8_t* out_packed, uint8_t* out_sf, uint8_t* out_sf_rowmajor,
                                   int pdl, fp4q_stream_t stream);

/*
 * fp4_dequant - validation helper: out[m, i] = E2M1 value of code (m, i) times
 * its block scale, fp32 (exact).  Mirrors the dequantise-and-compare method of
 * the FlashRT `fp4-gemm` README (Validation; `dequantize_fp4_sfa_fp16`).
 *
 *   packed    [M, H/2] bytes.                      8-byte aligned.
 *   sf        scales in `sf_layout` (FP4_SF_ROWMAJOR or FP4_SF_SWIZZLED).
 *   out       [M, H] fp32.                         16-byte aligned.
 * H must be a multiple of the block size (>= 16); M >= 0.
 */
FP4Q_API fp4_status_t fp4_dequant(const uint8_t* packed, const uint8_t* sf, int64_t M, int64_t H,
                                  fp4_format_t format, fp4_sf_layout_t sf_layout, float* out,
                                  fp4q_stream_t stream);

/*
 * fp4_sf_size_bytes - bytes of ONE scale buffer in `layout` (FlashInfer page,
 * output allocation; FlashRT README `sfa_size_bytes`): row-major M * (H/b);
 * tiled ceil(M/128) * ceil((H/b)/4) * 512.  FP4_SF_BOTH returns the tiled size
 * (the size of out_sf).  Returns -1 on bad arguments.  Host only; no GPU needed.
 */
FP4Q_API int64_t fp4_sf_size_bytes(int64_t M, int64_t H, fp4_format_t format, fp4_sf_layout_t layout);

/*
 * fp4_launch_shape - the launch the library would make for fp4_add_rmsnorm_quant
 * with these sizes on the current device (diagnostics; launches nothing).
 * Fills out[8] = {kernel (0 = persistent TMA-ring kernel, 1 = register-resident
 * kernel), chunks per thread, threads per row slice, row slices per CTA,
 * CTAs per cluster, shared-memory ring stages, threads per CTA, CTAs}.
 * Returns FP4_OK, or the status fp4_add_rmsnorm_quant would return for the sizes.
 */
FP4Q_API fp4_status_t fp4_launch_shape(int64_t M, int64_t H, fp4_dtype_t dtype, fp4_format_t format,
                                       fp4_sf_layout_t sf_layout, int64_t out[8]);

/*
 * fp4_gemm_variant - the schedule (the `variant` numbers of
 * fp4_gemm_nvfp4_bf16 below) the GEMM entry points would run for an
 * M x N x K product of `format` operands (FP4_NVFP4 or FP4_MXFP4); fp4_out
 * nonzero for fp4_gemm_nvfp4_gelu_nvfp4.  `variant` -1 asks for the
 * automatic choice; any other accepted value is returned as given.  Returns
 * -1 for sizes or a variant the GEMM would reject.  Host only (diagnostics;
 * launches nothing): the choice depends on the current device's SM count,
 * taken as 152 when no device is visible.
 */
FP4Q_API int fp4_gemm_variant(int64_t M, int64_t N, int64_t K, fp4_format_t format, int fp4_out,
                              int variant);

/*
 * fp4_gemm_nvfp4_bf16 - the consumer of the packed codes and tiled scales:
 * out = bf16(alpha * deq(A) @ deq(B)^T (+ bias) (+ residual)) on the tensor
 * cores (FlashRT `fp4-gemm` README: Tensor Contract; `nvfp4_gemm_bf16`,
 * `nvfp4_gemm_bias_bf16`, `nvfp4_gemm_residual_bf16`,
 * `nvfp4_gemm_bias_residual_bf16`), deq = E2M1 value times its E4M3 block
 * scale (16 elements per block), accumulation in fp32.
 *
 *   a_packed  [M, K/2] bytes: rows of A, two E2M1 codes per byte (element 2j in
 *             the low nibble), e.g. out_packed of the fused op or fp4_quantize.
 *   b_packed  [N, K/2] bytes: rows of B (the weight, one row per output column).
 *   sfa, sfb  NVFP4 scales of A (M rows) and of B (N rows) in the 128x4 tiled
 *             layout (FP4_SF_SWIZZLED), fp4_sf_size_bytes(M or N, K, ...) bytes.
 *   alpha     fp32 multiplier of the product (e.g. 1 / (gs_a * gs_b) for
 *             operands quantized with global scales).
 *   bias      [N] bf16 or NULL, added after alpha.
 *   residual  [M, N] bf16 or NULL, added last; may be `out` itself.
 *   out       [M, N] bf16, row-major.
 *   variant   tile schedule (the README's `variant`; fp4_gemm_variant reports
 *             the automatic choice): -1 automatic; one CTA per output tile with
 *             0 = 128 x 128 tiles (two CTAs per SM) or 1 = 128 x 256 tiles;
 *             persistent CTAs walking the tiles, one accumulator each, loading
 *             the next tile while the epilogue drains the last, with
 *             2 = 128 x 128 (two CTAs per SM) or 3 = 128 x 256 (one per SM;
 *             automatic when the output has more 128 x 128 tiles than twice
 *             the SMs); 4 = 128 x 128 tiles with the K loop of each tile split
 *             over a thread-block cluster of up to 16 CTAs (partial tiles
 *             summed in rank order through distributed shared memory;
 *             automatic when the output has at most half as many 128 x 128
 *             tiles as SMs and K > 1536, e.g. the M = 41 decode product with
 *             K = 6144).
 *   pdl       1: launched as a programmatic dependent of the previous kernel
 *             on `stream`, so its prologue overlaps that kernel's tail (it
 *             waits for that kernel's results before reading anything).
 *             2: the same, and the caller states that the previous kernel
 *             writes neither b_packed nor sfb (weights, as in a decode step
 *             after the fused op): the one-CTA-per-tile and split-K schedules
 *             then start B's first ring of copies before the wait.  0: none.
 *             Other values: FP4_ERR_INVALID_ARG.
 * K must be a multiple of 32 (a packed row a whole number of 16-byte units;
 * the FlashRT contract's K % 16 otherwise) and N of 8; every pointer 16-byte
 * aligned; out must not overlap the inputs (except residual == out).  When K
 * is not a multiple of 64, the last K = 64 step reads the k-padding scales of
 * the tiled layout against zero codes: they must be finite (this library's
 * producers write them as 0).  A tile whose inputs never arrive (a bounded
 * wait runs out) is written as NaN.
 */
FP4Q_API fp4_status_t fp4_gemm_nvfp4_bf16(const uint8_t* a_packed, const uint8_t* b_packed,
                                          const uint8_t* sfa, const uint8_t* sfb, float alpha,
                                          const void* bias, const void* residual, int64_t M, int64_t N,
                                          int64_t K, void* out, int variant, int pdl,
                                          fp4q_stream_t stream);

/*
 * fp4_gemm_mxfp4_bf16 - the same product for MXFP4 operands: E2M1 codes with
 * one UE8M0 scale per 32 elements (the fused op's and fp4_quantize's MXFP4
 * output, tiled layout, fp4_sf_size_bytes(M or N, K, FP4_MXFP4, ...) bytes).
 * Not on the FlashRT page (its GEMM is NVFP4 only): the consumer of this
 * library's own MXFP4 producer.  Arguments, checks and variants as
 * fp4_gemm_nvfp4_bf16 (every variant).
 */
FP4Q_API fp4_status_t fp4_gemm_mxfp4_bf16(const uint8_t* a_packed, const uint8_t* b_packed,
                                          const uint8_t* sfa, const uint8_t* sfb, float alpha,
                                          const void* bias, const void* residual, int64_t M,
                                          int64_t N, int64_t K, void* out, int variant, int pdl,
                                          fp4q_stream_t stream);

/*
 * fp4_gemm_nvfp4_gelu_bf16 - out = bf16(GELU(alpha * deq(A) @ deq(B)^T + bias))
 * (FlashRT `fp4-gemm` README, `nvfp4_gemm_bias_gelu_bf16`; GELU is the exact
 * x * Phi(x), computed with erff; bias may be NULL).  Arguments as
 * fp4_gemm_nvfp4_bf16 without the residual.
 */
FP4Q_API fp4_status_t fp4_gemm_nvfp4_gelu_bf16(const uint8_t* a_packed, const uint8_t* b_packed,
                                               const uint8_t* sfa, const uint8_t* sfb,
                                               float alpha, const void* bias, int64_t M,
                                               int64_t N, int64_t K, void* out, int variant,
                                               int pdl, fp4q_stream_t stream);

/*
 * fp4_gemm_nvfp4_gelu_nvfp4 - the same GELU values, rounded to fp32 and
 * quantized in the epilogue to NVFP4 for the next GEMM (README,
 * `nvfp4_gemm_bias_gelu_nvfp4`: "packed FP4 plus CUTLASS SFA"): the
 * producer's rules (E4M3 scale of amax / 6 per 16 values, codes of
 * v * rn(1/s), no global scale).
 *   out_packed  [M, N/2] bytes, 16-byte aligned.
 *   out_sf      tiled scales of the M x N output (fp4_sf_size_bytes(M, N,
 *               FP4_NVFP4, FP4_SF_SWIZZLED) bytes), padding rows and k padding
 *               written 0.
 * N must be a multiple of 16; variant 4 (split K) is not available
 * (FP4_ERR_INVALID_ARG); outputs must not overlap the inputs or each other.
 */
FP4Q_API fp4_status_t fp4_gemm_nvfp4_gelu_nvfp4(const uint8_t* a_packed,
                                                const uint8_t* b_packed, const uint8_t* sfa,
                                                const uint8_t* sfb, float alpha,
                                                const void* bias, int64_t M, int64_t N,
                                                int64_t K, uint8_t* out_packed,
                                                uint8_t* out_sf, int variant, int pdl,
                                                fp4q_stream_t stream);

/* Output of the general GEMM entry point fp4_gemm_ex. */
typedef enum {
  FP4_EPI_BF16 = 0,        /* alpha * product (+ bias) (+ residual) -> bf16 out   */
  FP4_EPI_GELU_BF16 = 1,   /* GELU(alpha * product (+ bias)) -> bf16 out          */
  FP4_EPI_GELU_NVFP4 = 2   /* GELU(...) -> NVFP4 codes + tiled scales (out_packed, out_sf) */
} fp4_epilogue_t;

/*
 * fp4_gemm_ex - the general form of the four GEMM entry points above: operand
 * `format` (FP4_NVFP4 or FP4_MXFP4; FP4_EPI_GELU_NVFP4 takes NVFP4 only), the
 * `epilogue`, and a device `status` word (DEVICE int32_t, 4-byte aligned, or
 * NULL) that receives FP4_ERR_TIMEOUT when a CTA's bounded wait ran out (its
 * tiles are then NaN, or 0xFF scale bytes for NVFP4 output; see "Device status
 * word").  `residual` is used by FP4_EPI_BF16 only; `out` by the bf16
 * epilogues, `out_packed` / `out_sf` by FP4_EPI_GELU_NVFP4.  Every other
 * argument, check and variant as fp4_gemm_nvfp4_bf16 /
 * fp4_gemm_nvfp4_gelu_nvfp4; the four named entry points are this call with
 * status = NULL.
 */
FP4Q_API fp4_status_t fp4_gemm_ex(const uint8_t* a_packed, const uint8_t* b_packed,
                                  const uint8_t* sfa, const uint8_t* sfb, fp4_format_t format,
                                  fp4_epilogue_t epilogue, float alpha, const void* bias,
                                  const void* residual, int64_t M, int64_t N, int64_t K, void* out,
                                  uint8_t* out_packed, uint8_t* out_sf, int variant, int pdl,
                                  int32_t* status, fp4q_stream_t stream);

/*
 * fp4_read_device_status - synchronises `stream`, then copies the device
 * status word back and returns it as a status: FP4_OK (0) or FP4_ERR_TIMEOUT;
 * FP4_ERR_INVALID_ARG for a NULL or misaligned pointer or a value that is no
 * status; FP4_ERR_CUDA if the synchronisation or the copy failed.  Blocks the
 * calling thread; not for use inside stream capture.
 */
FP4Q_API fp4_status_t fp4_read_device_status(const int32_t* status, fp4q_stream_t stream);

/*
 * Debug build.  `python -m rmsnorm_fp4_quant_gb300.build --debug` also builds
 * libfp4q_debug.so: the same entry points compiled with checks of every
 * global address a kernel computes against the extent of its buffer (an
 * access outside it is counted and skipped, never made), and with a fault
 * injector for the bounded waits.  The default libfp4q.so carries neither.
 *
 * fp4_debug_build - 1 in the debug build, 0 in the default one.
 *
 * fp4_debug_configure - process-wide knobs of the debug build, applied to
 * every later launch (FP4_ERR_INVALID_ARG in the default build):
 *   wait_limit_cycles  clock cycles each bounded wait allows (> 0; about one
 *                      second, 2e9, unless changed);
 *   shrink_bytes       bytes taken off every buffer extent the checks use
 *                      (>= 0; 0 for the real extents), so a test can see the
 *                      checks catch the accesses near the end of a buffer;
 *   drop_kernel        0 none, 1 the wide-row fused kernel, 2 the GEMM: CTA
 *                      `drop_cta` arrives on a stage's barrier expecting the
 *                      bytes of a copy it then never issues, at ring iteration
 *                      (fused) or K-block count (GEMM) `drop_iter`, so that
 *                      the wait on that stage runs out with nothing in flight
 *                      for it and the kernel's timeout path runs;
 *   violations         DEVICE uint32_t counter (4-byte aligned) that the
 *                      checks increment, or NULL (not counted).
 * These knobs are for tests; no default build reads them.
 */
FP4Q_API int fp4_debug_build(void);
FP4Q_API fp4_status_t fp4_debug_configure(int64_t wait_limit_cycles, int64_t shrink_bytes,
                                          int drop_kernel, int drop_cta, int drop_iter,
                                          uint32_t* violations);

/* Static, NUL-terminated description of a status code. */
FP4Q_API const char* fp4_status_string(fp4_status_t status);

/* cudaError_t value behind the last FP4_ERR_CUDA returned on this thread (0 if none). */
FP4Q_API int fp4_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FP4Q_H_ */
