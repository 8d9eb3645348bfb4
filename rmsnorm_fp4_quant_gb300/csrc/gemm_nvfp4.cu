// gemm_nvfp4.cu - the consumer of the packed codes and tiled scales: an NVFP4 x
// NVFP4 -> bf16 GEMM on the sm_103a tensor cores (FlashRT `fp4-gemm` README:
// Tensor Contract, `nvfp4_gemm_bf16` and its bias / residual epilogues).
//
//   out[m, n] = bf16( alpha * sum_k deq(A)[m, k] * deq(B)[n, k]  (+ bias[n])  (+ residual[m, n]) )
//
// A is [M, K/2] bytes and B is [N, K/2] bytes of E2M1 codes (both K-major, as
// the producer writes them); sfa / sfb are their 128x4 tiled E4M3 scale
// buffers.  One CTA computes one 128 x 128 output tile; the fp32 accumulator
// lives in tensor memory (128 lanes = rows, 128 columns).
//
//   warp 0, one lane   producer.  Per K block of 256 elements: the A and B
//                      tiles (128 rows x 128 bytes each) by TMA with the
//                      128-byte swizzle, and 2 KiB of each scale buffer by a
//                      bulk copy - the four 512-byte scale tiles of this K
//                      block, contiguous in the 128x4 layout - into a ring of
//                      S stages, completion counted on full[s].
//   warp 1, one lane   MMA issuer.  Copies the stage's eight scale tiles into
//                      tensor memory (tcgen05.cp 32x128b, repeated over the four
//                      lane quarters: a 512-byte tile is exactly the image of
//                      128 rows x 4 scales the block-scaled MMA reads), issues
//                      four K = 64 MMAs of kind mxf4nvf4 with one E4M3 scale per
//                      16 elements, and commits the stage back (empty[s]).
//   all four warps     epilogue.  Warp w owns accumulator lanes 32w..32w+31 (one
//                      output row per thread): 32 columns at a time from tensor
//                      memory, alpha, bias and residual in fp32, one rounding to
//                      bf16, 16-byte stores.
//
// Two CTAs fit an SM (S = 3 stages: 108 KiB of shared memory and 256 tensor-
// memory columns each), so one CTA's epilogue overlaps the other's main loop.
//
// Every mbarrier wait is bounded.  A producer or MMA wait that runs out marks
// the CTA failed: the producer waits (bounded) for its copies in flight, the
// MMA issuer still commits so the epilogue wait ends once its MMAs are done,
// the tile is written as NaN, and tensor memory is freed before the exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp4q_launch.h"
#include "tcgen05.cuh"

namespace fp4q {

namespace {

constexpr int kBM = 128;                    // output rows per CTA (MMA M)
constexpr int kBN = 128;                    // output columns per CTA (MMA N)
constexpr int kBKBytes = 128;               // K block: 256 E2M1 codes = one swizzle row
constexpr int kMmaKBytes = 32;              // K = 64 codes per MMA
constexpr uint32_t kTileBytes = kBM * kBKBytes;   // 16 KiB, A and B alike
constexpr uint32_t kSfTileBytes = 512;            // 128 rows x 4 scales
constexpr uint32_t kSfBytes = 4 * kSfTileBytes;   // scales of one K block
constexpr uint32_t kStageBytes = 2 * kTileBytes + 2 * kSfBytes;
constexpr uint32_t kAccCols = kBN;          // fp32 accumulator columns
constexpr uint32_t kSfColsPerStage = 32;    // 16 for A's four tiles, 16 for B's

// Instruction descriptor of the block-scaled MMA: E2M1 A and B (format 1 at
// bits 7-9 and 10-12), both K-major, N >> 3 at bits 17-22, E4M3 scales (bit 23
// clear), M >> 7 at bits 27-28, dense K = 64.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) |
                            (static_cast<uint32_t>(kBM >> 7) << 27);

__host__ __device__ constexpr uint32_t tmem_cols_for(int stages) {
  // accumulator + per-stage scale columns, rounded up to a power of two
  return (kAccCols + kSfColsPerStage * stages) <= 256 ? 256u : 512u;
}

__host__ __device__ constexpr size_t gemm_smem_bytes(int stages) {
  // 1 KiB of alignment slack (the 128-byte swizzle wants 1 KiB-aligned tiles),
  // the ring, 2S + 1 mbarriers, the tensor-memory address and a failure flag
  return 1024 + static_cast<size_t>(stages) * kStageBytes + (2 * stages + 1) * 8 + 8;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__global__ void __launch_bounds__(128, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmap_a,
                  const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  uint8_t* sA = smem;
  uint8_t* sB = sA + static_cast<size_t>(S) * kTileBytes;
  uint8_t* sSFA = sB + static_cast<size_t>(S) * kTileBytes;
  uint8_t* sSFB = sSFA + static_cast<size_t>(S) * kSfBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + static_cast<size_t>(S) * kSfBytes);
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* failed = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x;
  const int m_tile = blockIdx.y;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *failed = 0;
    mbar_init_fence();
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  // A and its scales may come from the kernel before this one (PDL); tensor
  // memory is taken only after it, since that kernel may still hold some
  griddep_wait();
  if (warp == 0) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- producer ----
    const uint8_t* sfa_k = p.sfa + static_cast<size_t>(m_tile) * p.nkt * kSfTileBytes;
    const uint8_t* sfb_k = p.sfb + static_cast<size_t>(n_tile) * p.nkt * kSfTileBytes;
    int kb = 0;
    for (; kb < p.num_kb; ++kb) {
      const int s = kb % S;
      if (kb >= S && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((kb / S - 1) & 1))) {
        *failed = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[s], kStageBytes);
      tma_load_2d(sA + static_cast<size_t>(s) * kTileBytes, &tmap_a, kb * kBKBytes, m_tile * kBM,
                  &full[s]);
      tma_load_2d(sB + static_cast<size_t>(s) * kTileBytes, &tmap_b, kb * kBKBytes, n_tile * kBN,
                  &full[s]);
      bulk_g2s(sSFA + static_cast<size_t>(s) * kSfBytes, sfa_k + static_cast<size_t>(kb) * kSfBytes,
               kSfBytes, &full[s]);
      bulk_g2s(sSFB + static_cast<size_t>(s) * kSfBytes, sfb_k + static_cast<size_t>(kb) * kSfBytes,
               kSfBytes, &full[s]);
    }
    if (kb < p.num_kb) {   // gave up: let the copies already issued land first
      for (int j = kb > S ? kb - S : 0; j < kb; ++j)
        mbar_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1));
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    for (int kb = 0; kb < p.num_kb; ++kb) {
      const int s = kb % S;
      if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((kb / S) & 1))) {
        *failed = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t sfa_t = tmem + kAccCols + static_cast<uint32_t>(s) * kSfColsPerStage;
      const uint32_t sfb_t = sfa_t + 16;
      const uint32_t a_s = smem_addr(sA + static_cast<size_t>(s) * kTileBytes);
      const uint32_t b_s = smem_addr(sB + static_cast<size_t>(s) * kTileBytes);
      const uint32_t sfa_s = smem_addr(sSFA + static_cast<size_t>(s) * kSfBytes);
      const uint32_t sfb_s = smem_addr(sSFB + static_cast<size_t>(s) * kSfBytes);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // a scale tile: 32 rows of 16 bytes, 8-row groups 128 bytes apart
        tmem_copy_32x128b_x4(sfa_t + 4 * j, smem_desc(sfa_s + j * kSfTileBytes, 0, 128, kSwizzleNone));
        tmem_copy_32x128b_x4(sfb_t + 4 * j, smem_desc(sfb_s + j * kSfTileBytes, 0, 128, kSwizzleNone));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // K-major, 128-byte swizzle: 8-row groups 1024 bytes apart; the K step
        // advances the start address inside the swizzle row
        const uint64_t adesc = smem_desc(a_s + j * kMmaKBytes, 0, 1024, kSwizzle128B);
        const uint64_t bdesc = smem_desc(b_s + j * kMmaKBytes, 0, 1024, kSwizzle128B);
        mma_mxf4nvf4(tmem, adesc, bdesc, kIdesc, sfa_t + 4 * j, sfb_t + 4 * j,
                     (kb | j) != 0 ? 1u : 0u);
      }
      tc_commit(&empty[s]);   // the stage is free once these MMAs have read it
    }
    tc_commit(accum);         // every MMA issued above has completed
  }
  __syncthreads();            // roles done; a failure flag is visible to all

  // ---- epilogue ----
  const bool acc_ok = mbar_wait_bounded(accum, 0);
  tc_fence_after_sync();
  const bool bad = !acc_ok || *failed != 0;
  griddep_launch_dependents();

  const int row = m_tile * kBM + warp * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const float nan = __int_as_float(0x7fc00000);
#pragma unroll 1
  for (int c = 0; c < kBN; c += 32) {
    uint32_t r[32];
    tmem_load_32cols(lane_base + static_cast<uint32_t>(c), r);   // whole warp, unconditionally
    if (row >= p.M) continue;
    const int n0 = n_tile * kBN + c;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + 8 * q;
      if (n >= p.N) break;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = bad ? nan : __uint_as_float(r[8 * q + i]) * p.alpha;
      if (p.bias) {
        const uint4 b = *reinterpret_cast<const uint4*>(p.bias + n);
        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = bf16x2_to_float2(bw[i]);
          v[2 * i] += f.x;
          v[2 * i + 1] += f.y;
        }
      }
      const size_t off = static_cast<size_t>(row) * static_cast<size_t>(p.N) + n;
      if (p.residual) {
        const uint4 rr = *reinterpret_cast<const uint4*>(p.residual + off);
        const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = bf16x2_to_float2(rw[i]);
          v[2 * i] += f.x;
          v[2 * i + 1] += f.y;
        }
      }
      uint4 o;
      o.x = bf16x2_bits(v[0], v[1]);
      o.y = bf16x2_bits(v[2], v[3]);
      o.z = bf16x2_bits(v[4], v[5]);
      o.w = bf16x2_bits(v[6], v[7]);
      *reinterpret_cast<uint4*>(p.out + off) = o;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [rows, K/2] bytes, row-major: boxes of 128 rows x 128 bytes, 128-byte swizzle,
// rows past the end read as zero.
bool make_operand_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t k_bytes) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(kBM)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t gemm_nvfp4_smem_bytes(int stages) { return gemm_smem_bytes(stages); }

cudaError_t launch_gemm_nvfp4(const uint8_t* a, const uint8_t* b, GemmParams p, int pdl,
                              cudaStream_t stream) {
  if (p.stages < 2 || p.stages > 6) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_operand_map(&ta, a, p.M, p.K / 2) || !make_operand_map(&tb, b, p.N, p.K / 2))
    return cudaErrorInvalidValue;
  p.tmem_cols = tmem_cols_for(p.stages);
  p.nkt = p.K / 64;
  p.num_kb = p.K / (2 * kBKBytes);
  const size_t smem = gemm_smem_bytes(p.stages);
  static size_t raised[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || raised[dev] < smem) {
    e = cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) raised[dev] = smem;
  }
  // resident CTAs must not ask for more than the SM's 512 tensor-memory columns
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_nvfp4_kernel, 128, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1 || per_sm * p.tmem_cols > 512) return cudaErrorInvalidConfiguration;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.N + kBN - 1) / kBN),
                     static_cast<unsigned>((p.M + kBM - 1) / kBM), 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_nvfp4_kernel, ta, tb, p);
}

}  // namespace fp4q
