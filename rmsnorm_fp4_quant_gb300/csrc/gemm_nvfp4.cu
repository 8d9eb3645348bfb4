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
//   warps 0 and 2,     producers.  Per K block of 256 elements: the A and B
//   one lane each      tiles (128 rows x 128 bytes each) by TMA with the
//                      128-byte swizzle, and 2 KiB of each scale buffer by a
//                      bulk copy - the four 512-byte scale tiles of this K
//                      block, contiguous in the 128x4 layout - into a ring of
//                      S stages, the operand tiles counted on full[s], the
//                      scales on sf_full[s].  Warp 0 loads A and its scales,
//                      warp 2 B and its scales, each arriving once per stage
//                      on each barrier (two threads issue a stage's copies in
//                      about half the time one takes: 4 % on a large product).
//   warps 3 and 4,     scale movers.  As soon as a stage's scales have landed
//   one lane each      (sf_full[s], before its operand tiles), copy its eight
//                      scale tiles into the stage's tensor-memory slot
//                      (tcgen05.cp 32x128b, repeated over the four lane
//                      quarters: a 512-byte tile is exactly the image of 128
//                      rows x 4 scales the block-scaled MMA reads), even tiles
//                      by one and odd by the other, each committing to
//                      sf_ready[s], so the copies of stage s + 1 run while
//                      stage s multiplies.  Issuing a copy holds its thread for
//                      tens of cycles, hence two.
//   warp 1, one lane   MMA issuer.  Once the stage's scales are in tensor
//                      memory, issues four K = 64 MMAs of kind mxf4nvf4 with
//                      one E4M3 scale per 16 elements, and commits the stage
//                      back (empty[s]).
//   warps 0..3         epilogue.  Warp w owns accumulator lanes 32w..32w+31 (one
//                      output row per thread), read 32 columns at a time from
//                      tensor memory into the drained ring as fp32; then all
//                      five warps write the tile out row by row (consecutive
//                      threads on consecutive 16-byte pieces) with alpha, bias
//                      and residual in fp32 and one rounding to bf16.
//
// Two CTAs fit an SM (S = 3 stages: 108 KiB of shared memory and 256 tensor-
// memory columns each), so one CTA's epilogue overlaps the other's main loop.
//
// Every mbarrier wait is bounded.  A producer or MMA wait that runs out marks
// the CTA failed: the producer waits (bounded) for its copies in flight, the
// MMA issuer still commits so the epilogue wait ends once its MMAs are done,
// the tile is written as NaN, the caller's status word (if any) receives the
// timeout status, and tensor memory is freed before the exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "fp4q_device.cuh"
#include "fp4q_launch.h"
#include "gemm_launch.h"
#include "tcgen05.cuh"

namespace fp4q {

namespace {

constexpr int kBM = 128;                    // output rows per CTA (MMA M)
constexpr int kBKBytes = 128;               // K block: 256 E2M1 codes = one swizzle row
constexpr int kMmaKBytes = 32;              // K = 64 codes per MMA
constexpr uint32_t kTileBytesA = kBM * kBKBytes;  // 16 KiB
constexpr uint32_t kSfTileBytes = 512;            // 128 rows x 4 scales

// Per output-tile width BN (the MMA's N: 128 or 256 columns) and scale format:
// NVFP4 (E4M3 scale per 16 codes, four 512-byte scale tiles per K block, one
// per MMA) or MXFP4 (UE8M0 per 32 codes, two tiles per K block, each holding
// the scales of two MMAs: bytes 0-1 and 2-3 of a row's 4-byte group).
template <int BN, bool MX = false>
struct Cfg {
  static constexpr uint32_t kTileBytesB = BN * kBKBytes;
  static constexpr int kSfTilesB = BN / 128;              // 128-row scale tiles of B
  static constexpr int kSfAtoms = MX ? 2 : 4;             // scale tiles per 128 rows per K block
  static constexpr uint32_t kSfBytesA = kSfAtoms * kSfTileBytes;
  static constexpr uint32_t kSfBytesB = kSfTilesB * kSfBytesA;
  static constexpr uint32_t kStageBytes = kTileBytesA + kTileBytesB + kSfBytesA + kSfBytesB;
  static constexpr uint32_t kAccCols = BN;                // fp32 accumulator columns
  static constexpr uint32_t kSfColsA = 4 * kSfAtoms;      // tensor-memory columns per stage
  static constexpr uint32_t kSfColsB = 4 * kSfAtoms * kSfTilesB;
  static constexpr uint32_t kSfColsPerStage = kSfColsA + kSfColsB;
  // Instruction descriptor of the block-scaled MMA: E2M1 A and B (format 1 at
  // bits 7-9 and 10-12), both K-major, N >> 3 at bits 17-22, scale type at bit
  // 23 (0 = E4M3, 1 = UE8M0), M >> 7 at bits 27-28, dense K = 64; the scale
  // byte pair of an MXFP4 step is chosen at bits 4-5 (B) and 29-30 (A).
  static constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) |
                                     (static_cast<uint32_t>(BN >> 3) << 17) |
                                     ((MX ? 1u : 0u) << 23) |
                                     (static_cast<uint32_t>(kBM >> 7) << 27);
  // K step j (of 4 per K block): its scale tile and instruction descriptor
  __host__ __device__ static constexpr int atom(int j) { return MX ? j / 2 : j; }
  __host__ __device__ static constexpr uint32_t idesc(int j) {
    return MX ? kIdesc | (static_cast<uint32_t>((j & 1) * 2) << 4) |
                    (static_cast<uint32_t>((j & 1) * 2) << 29)
              : kIdesc;
  }
  static constexpr uint32_t tmem_cols(int stages) {
    // accumulator + per-stage scale columns, rounded up to a power of two
    return (kAccCols + kSfColsPerStage * stages) <= 256 ? 256u : 512u;
  }
  static constexpr size_t smem_bytes(int stages) {
    // 1 KiB of alignment slack (the 128-byte swizzle wants 1 KiB-aligned
    // tiles), the ring, 4S + 3 mbarriers, the tensor-memory address, a flag
    return 1024 + static_cast<size_t>(stages) * kStageBytes + (4 * stages + 3) * 8 + 8;
  }
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// x * Phi(x) with the exact normal CDF (CUDA's erff).
__device__ __forceinline__ float gelu_exact(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

// alpha * acc + bias (fp32) for 8 columns starting at n, GELU when asked.
__device__ __forceinline__ void epilogue_values(const GemmParams& p, const float (&acc)[8], int n,
                                                bool bad, float (&v)[8]) {
  const float nan = __int_as_float(0x7fc00000);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = bad ? nan : acc[i] * p.alpha;
  if (p.bias && FP4Q_IN_RANGE(p, p.bias + n, 16, p.bias, 2LL * p.N)) {
    const uint4 b = *reinterpret_cast<const uint4*>(p.bias + n);
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_float2(bw[i]);
      v[2 * i] += f.x;
      v[2 * i + 1] += f.y;
    }
  }
  if (p.epilogue != kEpiPlain) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = gelu_exact(v[i]);
  }
}

// Epilogue of 8 accumulator values of one output row at column n (N % 8 == 0,
// so a group is all in or all out): alpha, bias, GELU or residual in fp32,
// one rounding to bf16, one 16-byte store.  `bad` stores NaN.
__device__ __forceinline__ void store8(const GemmParams& p, const float (&acc)[8], int row, int n,
                                       bool bad) {
  if (n >= p.N) return;
  float v[8];
  epilogue_values(p, acc, n, bad, v);
  const size_t off = static_cast<size_t>(row) * static_cast<size_t>(p.N) + n;
  const long long out_bytes = 2LL * p.M * p.N;
  if (p.residual && FP4Q_IN_RANGE(p, p.residual + off, 16, p.residual, out_bytes)) {
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
  if (FP4Q_IN_RANGE(p, p.out + off, 16, p.out, out_bytes)) *reinterpret_cast<uint4*>(p.out + off) = o;
}

// FP4 output of 16 values (one NVFP4 block) of one row at column n: the
// producer's rules (E4M3 scale of amax / 6, codes of v * rn(1/s)), codes to
// the packed output, the scale byte to the tiled scale buffer (k padding of
// the row's last group zeroed by the last block).  `row_valid` false writes
// the zero scale byte of a padding row; `bad` (the tile's inputs never
// arrived) writes the scale byte 0xFF (NaN in E4M3) and zero codes.
__device__ __forceinline__ void store_fp4_block16(const GemmParams& p, const float (&v)[16],
                                                  int row, int n, bool row_valid, bool bad) {
  const int kb = n >> 4;
  uint32_t code = 0;
  if (row_valid && bad) {
    code = 0xFFu;
    uint8_t* pk = p.out_packed + static_cast<size_t>(row) * static_cast<size_t>(p.N / 2) + n / 2;
    if (FP4Q_IN_RANGE(p, pk, 8, p.out_packed, packed_extent(p.M, p.N))) st_u64(pk, 0ull);
  } else if (row_valid) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) amax = max_abs3(amax, v[i], v[i + 1]);
    float inv_s;
    code = e4m3_block_scale(amax, 1.0f, inv_s);
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = inv_s > 0.0f ? v[i] * inv_s : 0.0f;
    const uint64_t packed = static_cast<uint64_t>(e2m1_pack8(q)) |
                            (static_cast<uint64_t>(e2m1_pack8(q + 8)) << 32);
    uint8_t* pk = p.out_packed + static_cast<size_t>(row) * static_cast<size_t>(p.N / 2) + n / 2;
    if (FP4Q_IN_RANGE(p, pk, 8, p.out_packed, packed_extent(p.M, p.N))) st_u64(pk, packed);
  }
  uint8_t* sfp = p.out_sf + tiled_sf_offset(row, kb, p.out_nkt);
  if (FP4Q_IN_RANGE(p, sfp, 1, p.out_sf, tiled_extent(p.M, p.out_nkt))) st_u8(sfp, code);
  if (kb == p.N / 16 - 1) {
    for (int kk = kb + 1; kk < 4 * p.out_nkt; ++kk) {
      uint8_t* pad = p.out_sf + tiled_sf_offset(row, kk, p.out_nkt);
      if (FP4Q_IN_RANGE(p, pad, 1, p.out_sf, tiled_extent(p.M, p.out_nkt))) st_u8(pad, 0u);
    }
  }
}

// 32 accumulator columns (raw fp32 bits from tensor memory) of one row.  Rows
// past M (the last row tile's padding) only write zero scale bytes, and only
// in the FP4-output epilogue.
__device__ __forceinline__ void store_columns32(const GemmParams& p, const uint32_t (&r)[32],
                                                int row, int n0, bool bad) {
  if (p.epilogue == kEpiGeluFp4) {
    const bool row_valid = row < p.M;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = n0 + 16 * h;
      if (n >= p.N) break;
      float v[16];
      if (row_valid) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float acc[8], out8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = __uint_as_float(r[16 * h + 8 * q + i]);
          epilogue_values(p, acc, n + 8 * q, bad, out8);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[8 * q + i] = out8[i];
        }
      }
      store_fp4_block16(p, v, row, n, row_valid, bad);
    }
    return;
  }
  if (row >= p.M) return;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __uint_as_float(r[8 * q + i]);
    store8(p, acc, row, n0 + 8 * q, bad);
  }
}

// SPLIT: split-K over a thread-block cluster of p.split CTAs along x, all on
// the same output tile; CTA rank q takes K blocks [q * nkb / split, (q + 1) *
// nkb / split), writes its fp32 partial tile into its own shared memory (the
// drained ring), and after a cluster barrier every rank sums a share of the
// tile over the ranks' partials in rank order (distributed shared memory
// loads), so the result does not depend on timing.  A second cluster barrier
// keeps each partial alive until every peer has read it.  For short, wide
// products (few output tiles) this spreads the K loop over many SMs.
//
// RAG: K % 256 != 0, so the last K block is ragged: only its K = 64 steps and
// scale tiles that exist are issued (codes past K read as zero, so a half
// step meets the tiled layout's k-padding scales).  A separate instance, so
// the full-block loops of every other product stay as they are.
// Threads of the one-tile kernel: four warps (roles, then the epilogue, one
// tensor-memory lane quarter each) and a fifth, the second scale mover.
constexpr int kTileThreads = 160;

template <int BN, bool SPLIT, bool MX, bool RAG>
__global__ void __launch_bounds__(kTileThreads, 1)
gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmap_a,
                  const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  using C = Cfg<BN, MX>;
  static_assert(!SPLIT || BN == 128, "the split partial tile must fit the drained ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  uint8_t* sA = smem;
  uint8_t* sB = sA + static_cast<size_t>(S) * kTileBytesA;
  uint8_t* sSFA = sB + static_cast<size_t>(S) * C::kTileBytesB;
  uint8_t* sSFB = sSFA + static_cast<size_t>(S) * C::kSfBytesA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + static_cast<size_t>(S) * C::kSfBytesB);
  uint64_t* empty = full + S;
  uint64_t* accum = empty + S;
  uint64_t* sf_ready = accum + 1;     // the stage's scales are in tensor memory
  uint64_t* sf_done = sf_ready + S;   // every scale copy has completed
  uint64_t* sf_full = sf_done + 1;    // the stage's scale bytes have landed
  uint64_t* recv_bar = sf_full + S;   // split K: the peers' partial rows have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recv_bar + 1);
  volatile int* failed = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = SPLIT ? p.split : 1;
  const int n_tile = SPLIT ? static_cast<int>(blockIdx.x) / split : static_cast<int>(blockIdx.x);
  const int rank = SPLIT ? static_cast<int>(cluster_ctarank()) : 0;
  const int m_tile = blockIdx.y;
  const int kb0 = SPLIT ? rank * p.num_kb / split : 0;
  const int kb1 = SPLIT ? (rank + 1) * p.num_kb / split : p.num_kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);   // one arrival per producer
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 2);  // one commit per scale mover
      mbar_init(&sf_full[s], 2);   // one arrival per producer
    }
    mbar_init(sf_done, 2);
    mbar_init(accum, 1);
    mbar_init(recv_bar, 1);
    *failed = 0;
    mbar_init_fence();
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  // B's 128-row scale tiles of this column tile that exist (the last column
  // tile may cover fewer rows than BN)
  const int b_tile0 = n_tile * C::kSfTilesB;
  const int b_tiles_total = (p.N + 127) / 128;
  const int b_tiles = b_tiles_total - b_tile0 < C::kSfTilesB ? b_tiles_total - b_tile0
                                                              : C::kSfTilesB;
  // block i's B tile and its scales into ring slot s (the B producer)
  auto issue_b = [&](int i, int s) {
    const int kb = kb0 + i;
    uint32_t sf_bytes = C::kSfBytesA;
    if constexpr (RAG) {
      if (kb == p.num_kb - 1)     // fewer scale tiles in the ragged last block
        sf_bytes = static_cast<uint32_t>(p.sf_tiles_last) * kSfTileBytes;
    }
    mbar_arrive_expect_tx(&sf_full[s], static_cast<uint32_t>(b_tiles) * sf_bytes);
    mbar_arrive_expect_tx(&full[s], C::kTileBytesB);
    for (int t = 0; t < b_tiles; ++t) {
      const uint8_t* src = p.sfb + (static_cast<size_t>(b_tile0 + t) * p.nkt) * kSfTileBytes +
                           static_cast<size_t>(kb) * C::kSfBytesA;
      if (FP4Q_IN_RANGE(p, src, sf_bytes, p.sfb, tiled_extent(p.N, p.nkt)))
        bulk_g2s(sSFB + static_cast<size_t>(s) * C::kSfBytesB + t * C::kSfBytesA, src,
                 sf_bytes, &sf_full[s]);
    }
    tma_load_2d(sB + static_cast<size_t>(s) * C::kTileBytesB, &tmap_b, kb * kBKBytes,
                n_tile * BN, &full[s]);
  };
  // When the caller states that the kernel before this one writes neither B
  // nor its scales (pdl = 2: weights), B's first ring of copies leaves before
  // the dependency wait and streams in during that kernel's tail.
  const int b_early = p.b_static ? (kb1 - kb0 < S ? kb1 - kb0 : S) : 0;
  if (b_early > 0) {
    __syncthreads();            // the barriers above are initialised
    if (warp == 2 && lane == 0)
      for (int i = 0; i < b_early; ++i) issue_b(i, i);
  }
  // A and its scales may come from the kernel before this one (PDL); tensor
  // memory is taken only after it, since that kernel may still hold some
  griddep_wait();
  if (warp == 0) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int issued = 0;    // K blocks a producer thread issued copies for

  if ((warp == 0 || warp == 2) && lane == 0) {
    // ---- producers: warp 0 A and its scales, warp 2 B and its scales ----
    const bool load_a = warp == 0;
    const uint8_t* sfa_k = p.sfa + static_cast<size_t>(m_tile) * p.nkt * kSfTileBytes;
    int i = 0;    // K blocks issued
    int s = 0;    // ring slot of block i; ph = (i / S) & 1, by counters (no division per block)
    uint32_t ph = 0;
    for (; i < kb1 - kb0; ++i) {
      const int kb = kb0 + i;
      if (i >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u, FP4Q_WAIT_LIMIT(p))) {
        *failed = 1;
        break;
      }
      if (!load_a) {
        if (i >= b_early) issue_b(i, s);   // the first b_early blocks left before the wait
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
        continue;
      }
      uint32_t sf_bytes = C::kSfBytesA;
      if constexpr (RAG) {
        if (kb == p.num_kb - 1)     // fewer scale tiles in the ragged last block
          sf_bytes = static_cast<uint32_t>(p.sf_tiles_last) * kSfTileBytes;
      }
      // the scales land on their own barrier, so the scale movers copy them
      // into tensor memory while the operand tiles are still arriving
      mbar_arrive_expect_tx(&sf_full[s], sf_bytes);
      mbar_arrive_expect_tx(&full[s], kTileBytesA);
      const uint8_t* src = sfa_k + static_cast<size_t>(kb) * C::kSfBytesA;
      if (FP4Q_IN_RANGE(p, src, sf_bytes, p.sfa, tiled_extent(p.M, p.nkt)))
        bulk_g2s(sSFA + static_cast<size_t>(s) * C::kSfBytesA, src, sf_bytes, &sf_full[s]);
      // debug build: one CTA never issues one A tile (fault injection)
      if (!FP4Q_DROP(p, 2, static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x), i))
        tma_load_2d(sA + static_cast<size_t>(s) * kTileBytesA, &tmap_a, kb * kBKBytes,
                    m_tile * kBM, &full[s]);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    issued = i;
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < kb1 - kb0; ++i) {
      // the operand tiles (full[s]) and the scales in tensor memory (sf_ready[s])
      if (!mbar_wait_bounded(&sf_ready[s], ph, FP4Q_WAIT_LIMIT(p)) ||
          !mbar_wait_bounded(&full[s], ph, FP4Q_WAIT_LIMIT(p))) {
        *failed = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t sfa_t = tmem + C::kAccCols + static_cast<uint32_t>(s) * C::kSfColsPerStage;
      const uint32_t sfb_t = sfa_t + C::kSfColsA;
      const uint32_t a_s = smem_addr(sA + static_cast<size_t>(s) * kTileBytesA);
      const uint32_t b_s = smem_addr(sB + static_cast<size_t>(s) * C::kTileBytesB);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if constexpr (RAG) {
          if (kb0 + i == p.num_kb - 1 && j >= p.mma_last) break;
        }
        // K-major, 128-byte swizzle: 8-row groups 1024 bytes apart; the K step
        // advances the start address inside the swizzle row
        const uint64_t adesc = smem_desc(a_s + j * kMmaKBytes, 0, 1024, kSwizzle128B);
        const uint64_t bdesc = smem_desc(b_s + j * kMmaKBytes, 0, 1024, kSwizzle128B);
        mma_fp4_block_scaled<MX>(tmem, adesc, bdesc, C::idesc(j), sfa_t + 4 * C::atom(j),
                                 sfb_t + 4 * C::kSfTilesB * C::atom(j), (i | j) != 0 ? 1u : 0u);
      }
      tc_commit(&empty[s]);   // the stage is free once these MMAs have read it
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    tc_commit(accum);         // every MMA issued above has completed
  } else if ((warp == 3 || warp == 4) && lane == 0) {
    // ---- scale movers: even scale tiles by warp 3, odd by warp 4 ----
    // Slot s is free for stage i: sf_full[s] of stage i means the producers
    // refilled the stage, which waited for the MMAs of stage i - S.
    const int mover = warp - 3;
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < kb1 - kb0; ++i) {
      if (!mbar_wait_bounded(&sf_full[s], ph, FP4Q_WAIT_LIMIT(p))) {
        *failed = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t sfa_t = tmem + C::kAccCols + static_cast<uint32_t>(s) * C::kSfColsPerStage;
      const uint32_t sfb_t = sfa_t + C::kSfColsA;
      const uint32_t sfa_s = smem_addr(sSFA + static_cast<size_t>(s) * C::kSfBytesA);
      const uint32_t sfb_s = smem_addr(sSFB + static_cast<size_t>(s) * C::kSfBytesB);
#pragma unroll
      for (int q = 0; q < C::kSfAtoms; ++q) {
        if (q % 2 != mover) continue;
        if constexpr (RAG) {
          if (kb0 + i == p.num_kb - 1 && q >= p.sf_tiles_last) break;
        }
        // a scale tile: 32 rows of 16 bytes, 8-row groups 128 bytes apart.
        // Tile q: A's at column 4q; B's 128-row tiles side by side from
        // 4 * kSfTilesB * q
        tmem_copy_32x128b_x4(sfa_t + 4 * q, smem_desc(sfa_s + q * kSfTileBytes, 0, 128, kSwizzleNone));
#pragma unroll
        for (int t = 0; t < C::kSfTilesB; ++t)
          tmem_copy_32x128b_x4(sfb_t + 4 * (C::kSfTilesB * q + t),
                               smem_desc(sfb_s + t * C::kSfBytesA + q * kSfTileBytes, 0, 128,
                                         kSwizzleNone));
      }
      tc_commit(&sf_ready[s]);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    tc_commit(sf_done);       // no copy may still be running when tensor memory is freed
    mbar_wait_bounded(sf_done, 0, FP4Q_WAIT_LIMIT(p));
  }
  __syncthreads();            // roles done; a failure flag is visible to all
  if (*failed != 0 && (warp == 0 || warp == 2) && lane == 0) {
    // A failed CTA may have stopped consuming stages it still has copies in
    // flight for: each producer waits (bounded) for the last S stages it
    // filled - earlier ones were consumed by MMAs, so their copies landed -
    // before anything here can end the CTA.
    for (int j = issued > S ? issued - S : 0; j < issued; ++j) {
      mbar_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1), FP4Q_WAIT_LIMIT(p));
      mbar_wait_bounded(&sf_full[j % S], static_cast<uint32_t>((j / S) & 1), FP4Q_WAIT_LIMIT(p));
    }
  }

  // ---- epilogue ----
  const bool acc_ok = mbar_wait_bounded(accum, 0, FP4Q_WAIT_LIMIT(p));
  tc_fence_after_sync();
  const bool bad = !acc_ok || *failed != 0;
  if (bad && threadIdx.x == 0 && p.status) atomicExch(p.status, kStatusTimeout);
  griddep_launch_dependents();

  // warps 0..3 drain the accumulator, warp w its lanes 32w..32w+31
  const int row = m_tile * kBM + warp * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  // The tile in fp32 in the drained ring, rows 16 bytes apart beyond BN
  // floats (a warp's row-per-lane float4 stores then take the minimum four
  // shared-memory wavefronts), so that it leaves in row order: a thread per
  // row storing its own 16-byte pieces scattered a warp's stores over 32 rows
  // and held each warp about 1100 cycles per 32 columns.
  constexpr int kStride = BN + 4;
  constexpr int kChunks = BN / 8;     // 8-column pieces of a row
  float* part = reinterpret_cast<float*>(smem);
  const int local_row = warp * 32 + lane;
  const int rows_valid = p.M - m_tile * kBM < kBM ? p.M - m_tile * kBM : kBM;
  if constexpr (!SPLIT) {
    if (p.epilogue == kEpiGeluFp4) {
      // NVFP4 output: a thread quantizes its own row's 16-element blocks
#pragma unroll 1
      for (int c = 0; c < BN && warp < 4; c += 32) {
        uint32_t r[32];
        tmem_load_32cols(lane_base + static_cast<uint32_t>(c), r);   // whole warp, unconditionally
        if (row >= p.rows_out) continue;
        store_columns32(p, r, row, n_tile * BN + c, bad);
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < BN && warp < 4; c += 32) {
        uint32_t r[32];
        tmem_load_32cols(lane_base + static_cast<uint32_t>(c), r);   // whole warp, unconditionally
        if (local_row >= rows_valid) continue;
        float4* dst = reinterpret_cast<float4*>(part + local_row * kStride + c);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                               __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
      }
      __syncthreads();
      // consecutive threads take consecutive 8-column pieces of a row
      for (int it = static_cast<int>(threadIdx.x); it < rows_valid * kChunks; it += kTileThreads) {
        const int rl = it / kChunks;
        const int ch = it - rl * kChunks;
        const float4 lo = *reinterpret_cast<const float4*>(part + rl * kStride + ch * 8);
        const float4 hi = *reinterpret_cast<const float4*>(part + rl * kStride + ch * 8 + 4);
        const float acc[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        store8(p, acc, m_tile * kBM + rl, n_tile * BN + ch * 8, bad);
      }
    }
  } else {
    // Partial tile -> own shared memory (NaN if this CTA's inputs never
    // arrived, so every sum it enters is NaN).  Rank q owns rows
    // [q * rows_valid / split, (q + 1) * rows_valid / split) of the tile: after
    // a cluster barrier every rank bulk-copies (TMA engine, shared to shared)
    // the rows each other rank owns into that rank's receive slot for it, and
    // each owner sums its rows over the ranks in rank order - the same sum on
    // every run.  Reading the peers' partials with per-thread remote loads
    // instead took about 230 cycles per load, one after another.
    const float nan = __int_as_float(0x7fc00000);
#pragma unroll 1
    for (int c = 0; c < BN && warp < 4; c += 32) {
      uint32_t r[32];
      tmem_load_32cols(lane_base + static_cast<uint32_t>(c), r);
      if (local_row >= rows_valid) continue;
      float4* dst = reinterpret_cast<float4*>(part + local_row * kStride + c);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = bad ? make_float4(nan, nan, nan, nan)
                     : make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                   __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
    }
    if (bad && threadIdx.x == 0) *failed = 1;
    constexpr uint32_t kRowBytes = kStride * sizeof(float);
    const int slot_rows = (rows_valid + split - 1) / split;
    float* recv = part + kBM * kStride;       // slot q: the rows from rank q
    const int my0 = rank * rows_valid / split;
    const int my1 = (rank + 1) * rows_valid / split;
    if (threadIdx.x == 0)
      mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((split - 1) * (my1 - my0)) * kRowBytes);
    fence_proxy_async_smem();   // the partial, written above, is read by the copies below
    cluster_arrive_release();   // every rank's partial and receive barrier are ready
    cluster_wait_acquire();
    // lane 0 of each warp issues the copies to every fifth peer (issuing one
    // holds its thread about 200 cycles)
    if (lane == 0) {
      for (int q = warp; q < split; q += kTileThreads / 32) {
        const int r0 = q * rows_valid / split;
        const int r1 = (q + 1) * rows_valid / split;
        if (q == rank || r1 <= r0) continue;
        bulk_s2cluster(peer_smem_addr(smem_addr(recv + rank * slot_rows * kStride),
                                      static_cast<uint32_t>(q)),
                       smem_addr(part + r0 * kStride), static_cast<uint32_t>(r1 - r0) * kRowBytes,
                       peer_smem_addr(smem_addr(recv_bar), static_cast<uint32_t>(q)));
      }
    }
    const bool got = mbar_wait_bounded(recv_bar, 0, FP4Q_WAIT_LIMIT(p));
    if (!got && threadIdx.x == 0) *failed = 1;
    // This CTA's incoming copies have landed.  Once every rank has arrived
    // here, every copy out of this CTA's partial has landed too: the wait for
    // that, before the CTA may end, comes after the sums below.  Nothing is
    // read on the strength of this arrival (the copies' completion is already
    // a fact), so it needs no release.
    cluster_arrive_relaxed();
    const int items = (my1 - my0) * kChunks;
    for (int it = static_cast<int>(threadIdx.x); it < items; it += kTileThreads) {
      const int rl = it / kChunks;          // row within the owned rows
      const int ch = it - rl * kChunks;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // rank order; four ranks' loads issued before their adds
      for (int q0 = 0; q0 < split; q0 += 4) {
        float4 lo[4], hi[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q0 + u < split ? q0 + u : split - 1;
          const float* src = q == rank ? part + (my0 + rl) * kStride + ch * 8
                                       : recv + (q * slot_rows + rl) * kStride + ch * 8;
          lo[u] = *reinterpret_cast<const float4*>(src);
          hi[u] = *reinterpret_cast<const float4*>(src + 4);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (q0 + u >= split) break;
          acc[0] += lo[u].x; acc[1] += lo[u].y; acc[2] += lo[u].z; acc[3] += lo[u].w;
          acc[4] += hi[u].x; acc[5] += hi[u].y; acc[6] += hi[u].z; acc[7] += hi[u].w;
        }
      }
      store8(p, acc, m_tile * kBM + my0 + rl, n_tile * BN + ch * 8, !got);
    }
    cluster_wait_acquire();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *failed != 0 && p.status) atomicExch(p.status, kStatusTimeout);
  if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

// Persistent form: resident CTAs (two per SM for 128-wide tiles, one for
// 256-wide) walk the output tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...
// (row tile t / n_tiles, column tile t % n_tiles, so CTAs running together
// share A's row panel).  Nine warps (thirteen for 256-wide tiles):
//   warps 0 and 6,    producers (A and its scales / B and its scales): one
//   one lane each     continuous stream of K blocks over all the CTA's tiles
//                     through the S-stage operand ring (never drains between
//                     tiles);
//   warp 1            tensor-memory allocation; one lane issues the MMAs;
//   warps 2..5        epilogue, lane quarter = warp % 4 (and, for 256-wide
//                     tiles, warps 8..11 draining the other half of the columns);
//   warp 7 and the    scale movers, one lane each: a K block's scale tiles
//   last warp         into its tensor-memory slot (even tiles by one, odd by
//                     the other), each committing to sf_ready[ss].
// The scales have a ring of their own, SS = S + lead slots in shared and
// tensor memory, and a producer issues K block it + lead's scales together
// with block it's operands: the scale copy into tensor memory, which
// completes only behind the MMAs already in the tensor pipe, then lands
// while the block before is multiplied instead of after it.  Both rings are
// freed by the same event - the MMAs of block it - S have completed (empty[s])
// - since block it + lead - SS = it - S.  lead = 1 where shared and tensor
// memory hold the extra slot at the CTA's occupancy, else 0.
// While the epilogue reads a tile's accumulator out (acc_empty), the
// producers already fill the ring with the next tile's K blocks, so a new
// tile never waits for a CTA launch or a first load; with two CTAs per SM the
// other CTA's MMAs run meanwhile.
#ifndef FP4Q_GEMM_EPI8
#define FP4Q_GEMM_EPI8 1     // 256-wide persistent tiles drained by eight epilogue warps
#endif
#ifndef FP4Q_GEMM_SF_LEAD
#define FP4Q_GEMM_SF_LEAD 1  // K blocks the persistent scale ring runs ahead (0 or 1)
#endif

template <int BN, bool MX>
struct PCfg {
  // Epilogue warps: four (one per tensor-memory lane quarter), or eight for
  // 256-wide tiles (two per quarter, each draining half of the columns), so
  // the single accumulator is handed back to the MMAs sooner (8192 x 7168 x
  // 7168: 260.5 -> 241.9 us for the 256-wide schedule).
  static constexpr int kEpiWarps = (BN == 256 && FP4Q_GEMM_EPI8) ? 8 : 4;
  // Two scale movers: issuing a tensor-memory copy holds its thread for tens
  // of cycles, and one thread's eight (twelve for 256-wide tiles) per K block
  // trailed the MMAs (8192 x 7168 x 7168, 256-wide: 256.5 -> 218.8 us).
  static constexpr int kMovers = 2;
  static constexpr int kMover2Warp = 4 + kEpiWarps;   // after the epilogue warps
  static constexpr int kThreads = 32 * (kMover2Warp + 1);
  // One accumulator: a 128-wide tile then needs 128 + SS * 32 <= 256 tensor-
  // memory columns, so two CTAs share an SM and one's epilogue overlaps the
  // other's MMAs (measured faster than one CTA per SM with two accumulators
  // and six stages: 238 against 315 us on an 8192 x 7168 x 7168 product).
  static constexpr int kAcc = 1;
  static constexpr int kCtasPerSm = BN == 128 ? 2 : 1;
  static constexpr uint32_t kSfCol = kAcc * BN;     // the scale slots after the accumulators
  static constexpr uint32_t tmem_cols(int sf_stages) {
    return (kSfCol + Cfg<BN, MX>::kSfColsPerStage * sf_stages) <= 256 ? 256u : 512u;
  }
  static constexpr size_t smem_bytes(int stages, int sf_stages) {
    using C = Cfg<BN, MX>;
    return 1024 + static_cast<size_t>(stages) * (kTileBytesA + C::kTileBytesB) +
           static_cast<size_t>(sf_stages) * (C::kSfBytesA + C::kSfBytesB) +
           (2 * stages + 2 * sf_stages + 2 * kAcc + 2) * 8 + 8;
  }
  // The scale ring's lead: 1 if the extra slot still fits kCtasPerSm CTAs in
  // an SM's shared memory (228 KiB, 1 KiB of it reserved per CTA) and tensor
  // memory (512 columns), else 0.
  static constexpr int sf_lead(int stages) {
    return FP4Q_GEMM_SF_LEAD > 0 &&
                   kCtasPerSm * (smem_bytes(stages, stages + 1) + 1024) <= 228 * 1024 &&
                   kCtasPerSm * tmem_cols(stages + 1) <= 512 &&
                   kSfCol + Cfg<BN, MX>::kSfColsPerStage * (stages + 1) <= 512
               ? 1
               : 0;
  }
};

template <int BN, bool MX, bool RAG>
__global__ void __launch_bounds__(PCfg<BN, MX>::kThreads, PCfg<BN, MX>::kCtasPerSm)
gemm_nvfp4_persistent_kernel(const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  using C = Cfg<BN, MX>;
  using P = PCfg<BN, MX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  const int SS = p.sf_stages;     // S or S + 1
  const int lead = SS - S;
  uint8_t* sA = smem;
  uint8_t* sB = sA + static_cast<size_t>(S) * kTileBytesA;
  uint8_t* sSFA = sB + static_cast<size_t>(S) * C::kTileBytesB;
  uint8_t* sSFB = sSFA + static_cast<size_t>(SS) * C::kSfBytesA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + static_cast<size_t>(SS) * C::kSfBytesB);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + P::kAcc;
  uint64_t* mma_done = acc_empty + P::kAcc;
  uint64_t* sf_ready = mma_done + 1;  // a scale slot's tiles are in tensor memory
  uint64_t* sf_done = sf_ready + SS;
  uint64_t* sf_full = sf_done + 1;    // a scale slot's bytes have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_full + SS);
  volatile int* failed = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles = n_tiles * ((p.M + kBM - 1) / kBM);
  const int G = gridDim.x;
  const int my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / G + 1 : 0;
  const int total = my_tiles * p.num_kb;    // K blocks over all of this CTA's tiles

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);      // one arrival per producer
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < SS; ++s) {
      mbar_init(&sf_ready[s], P::kMovers);   // one commit per mover
      mbar_init(&sf_full[s], 2);
    }
    mbar_init(sf_done, P::kMovers);
    for (int a = 0; a < P::kAcc; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], P::kEpiWarps);   // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    *failed = 0;
    mbar_init_fence();
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  griddep_wait();
  if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int issued = 0;      // K blocks whose operand copies a producer thread issued
  int issued_sf = 0;   // K blocks whose scale copies it issued

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ---- producers: warp 0 A and its scales, warp 6 B and its scales ----
    // Ring slots, phases and block coordinates advance by counters: this
    // thread's issue rate bounds the ring, and a division by a runtime value
    // per K block cost it more than its copies.
    const bool load_a = warp == 0;
    const int b_tiles_total = (p.N + 127) / 128;
    struct Pos {         // a K block: its tile's coordinates and its index in the K loop
      int t, m_tile, n_tile, kb;
    };
    auto at_tile = [&](int t, Pos& q) {
      q.t = t;
      q.m_tile = t / n_tiles;
      q.n_tile = t - q.m_tile * n_tiles;
      q.kb = 0;
    };
    auto advance = [&](Pos& q) {
      if (++q.kb == p.num_kb) at_tile(q.t + G, q);
    };
    // block q's scales into scale slot ss
    auto issue_scales = [&](const Pos& q, int ss) {
      uint32_t sf_bytes = C::kSfBytesA;
      if constexpr (RAG) {
        if (q.kb == p.num_kb - 1)   // fewer scale tiles in the ragged last block
          sf_bytes = static_cast<uint32_t>(p.sf_tiles_last) * kSfTileBytes;
      }
      if (load_a) {
        mbar_arrive_expect_tx(&sf_full[ss], sf_bytes);
        const uint8_t* src = p.sfa + static_cast<size_t>(q.m_tile) * p.nkt * kSfTileBytes +
                             static_cast<size_t>(q.kb) * C::kSfBytesA;
        if (FP4Q_IN_RANGE(p, src, sf_bytes, p.sfa, tiled_extent(p.M, p.nkt)))
          bulk_g2s(sSFA + static_cast<size_t>(ss) * C::kSfBytesA, src, sf_bytes, &sf_full[ss]);
      } else {
        // B's 128-row scale tiles of this column tile that exist
        const int b_tile0 = q.n_tile * C::kSfTilesB;
        const int b_tiles = b_tiles_total - b_tile0 < C::kSfTilesB ? b_tiles_total - b_tile0
                                                                    : C::kSfTilesB;
        mbar_arrive_expect_tx(&sf_full[ss], static_cast<uint32_t>(b_tiles) * sf_bytes);
        for (int u = 0; u < b_tiles; ++u) {
          const uint8_t* src = p.sfb + static_cast<size_t>(b_tile0 + u) * p.nkt * kSfTileBytes +
                               static_cast<size_t>(q.kb) * C::kSfBytesA;
          if (FP4Q_IN_RANGE(p, src, sf_bytes, p.sfb, tiled_extent(p.N, p.nkt)))
            bulk_g2s(sSFB + static_cast<size_t>(ss) * C::kSfBytesB + u * C::kSfBytesA, src,
                     sf_bytes, &sf_full[ss]);
        }
      }
    };
    Pos op, sc;              // block it, and block it + lead (its scales go out with it)
    at_tile(blockIdx.x, op);
    sc = op;
    int ss = 0;              // scale slot of block it + lead
    // blocks 0 .. lead-1: their scale slots start free
    for (; issued_sf < lead && issued_sf < total; ++issued_sf) {
      issue_scales(sc, ss);
      advance(sc);
      if (++ss == SS) ss = 0;
    }
    int it = 0, s = 0;
    uint32_t ph = 0;         // it = round * S + s, ph = round & 1
    for (; it < total; ++it) {
      // the MMAs of block it - S have completed: operand slot s and scale
      // slot (it + lead) % SS (last used by that same block) are free
      if (it >= S && !mbar_wait_bounded(&empty[s], ph ^ 1u, FP4Q_WAIT_LIMIT(p))) {
        *failed = 1;
        break;
      }
      if (it + lead < total) {
        issue_scales(sc, ss);
        issued_sf = it + lead + 1;
        advance(sc);
        if (++ss == SS) ss = 0;
      }
      mbar_arrive_expect_tx(&full[s], load_a ? kTileBytesA : C::kTileBytesB);
      if (load_a) {
        // debug build: one CTA never issues one A tile (fault injection)
        if (!FP4Q_DROP(p, 2, static_cast<int>(blockIdx.x), it))
          tma_load_2d(sA + static_cast<size_t>(s) * kTileBytesA, &tmap_a, op.kb * kBKBytes,
                      op.m_tile * kBM, &full[s]);
      } else {
        tma_load_2d(sB + static_cast<size_t>(s) * C::kTileBytesB, &tmap_b, op.kb * kBKBytes,
                    op.n_tile * BN, &full[s]);
      }
      advance(op);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
    issued = it;
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    int it = 0;
    int s = 0, ss = 0;         // operand and scale slots of block it
    uint32_t ph = 0, sph = 0;  // their phases
    bool ok = true;
    for (int i = 0; i < my_tiles && ok; ++i) {
      const int a = i % P::kAcc;
      // the epilogue has read this accumulator out (first use: passes at once)
      if (!mbar_wait_bounded(&acc_empty[a], static_cast<uint32_t>(((i / P::kAcc) & 1) ^ 1),
                             FP4Q_WAIT_LIMIT(p))) {
        *failed = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d_t = tmem + static_cast<uint32_t>(a * BN);
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        if (!mbar_wait_bounded(&sf_ready[ss], sph, FP4Q_WAIT_LIMIT(p)) ||
            !mbar_wait_bounded(&full[s], ph, FP4Q_WAIT_LIMIT(p))) {
          *failed = 1;
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sfa_t = tmem + P::kSfCol + static_cast<uint32_t>(ss) * C::kSfColsPerStage;
        const uint32_t sfb_t = sfa_t + C::kSfColsA;
        const uint32_t a_s = smem_addr(sA + static_cast<size_t>(s) * kTileBytesA);
        const uint32_t b_s = smem_addr(sB + static_cast<size_t>(s) * C::kTileBytesB);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (RAG) {
            if (kb == p.num_kb - 1 && j >= p.mma_last) break;
          }
          const uint64_t adesc = smem_desc(a_s + j * kMmaKBytes, 0, 1024, kSwizzle128B);
          const uint64_t bdesc = smem_desc(b_s + j * kMmaKBytes, 0, 1024, kSwizzle128B);
          mma_fp4_block_scaled<MX>(d_t, adesc, bdesc, C::idesc(j), sfa_t + 4 * C::atom(j),
                                   sfb_t + 4 * C::kSfTilesB * C::atom(j), (kb | j) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
        if (++ss == SS) {
          ss = 0;
          sph ^= 1u;
        }
      }
      // this tile's MMAs are done.  Not after a failure: the epilogue's own
      // wait then runs out and marks the tile, so it never depends on seeing
      // the failure flag through the asynchronous arrive
      if (!ok) break;
      tc_commit(&acc_full[a]);
    }
    // tensor memory is freed below only after every MMA issued here has completed
    tc_commit(mma_done);
    mbar_wait_bounded(mma_done, 0, FP4Q_WAIT_LIMIT(p));
  } else if ((warp == 7 || warp == P::kMover2Warp) && lane == 0) {
    // ---- scale movers: block j's scale tiles into tensor-memory slot j % SS.
    // The slot is free: sf_full of block j means a producer saw the MMAs of
    // block j - SS (its last reader) complete before issuing these bytes.
    const int mover = warp == 7 ? 0 : 1;
    int ss = 0, kb = 0;
    uint32_t sph = 0;
    for (int j = 0; j < total; ++j) {
      if (!mbar_wait_bounded(&sf_full[ss], sph, FP4Q_WAIT_LIMIT(p))) {
        *failed = 1;
        break;
      }
      tc_fence_after_sync();
      const uint32_t sfa_t = tmem + P::kSfCol + static_cast<uint32_t>(ss) * C::kSfColsPerStage;
      const uint32_t sfb_t = sfa_t + C::kSfColsA;
      const uint32_t sfa_s = smem_addr(sSFA + static_cast<size_t>(ss) * C::kSfBytesA);
      const uint32_t sfb_s = smem_addr(sSFB + static_cast<size_t>(ss) * C::kSfBytesB);
#pragma unroll
      for (int q = 0; q < C::kSfAtoms; ++q) {
        if (q % P::kMovers != mover) continue;
        if constexpr (RAG) {
          if (kb == p.num_kb - 1 && q >= p.sf_tiles_last) break;
        }
        // scale tile q: 32 rows of 16 bytes, 8-row groups 128 bytes apart
        tmem_copy_32x128b_x4(sfa_t + 4 * q,
                             smem_desc(sfa_s + q * kSfTileBytes, 0, 128, kSwizzleNone));
#pragma unroll
        for (int u = 0; u < C::kSfTilesB; ++u)
          tmem_copy_32x128b_x4(sfb_t + 4 * (C::kSfTilesB * q + u),
                               smem_desc(sfb_s + u * C::kSfBytesA + q * kSfTileBytes, 0, 128,
                                         kSwizzleNone));
      }
      tc_commit(&sf_ready[ss]);
      if (++ss == SS) {
        ss = 0;
        sph ^= 1u;
      }
      if (++kb == p.num_kb) kb = 0;
    }
    tc_commit(sf_done);
    mbar_wait_bounded(sf_done, 0, FP4Q_WAIT_LIMIT(p));
  } else if ((warp >= 2 && warp <= 5) || (warp >= 8 && warp < P::kMover2Warp)) {
    // ---- epilogue: warps 2..5 (and 8..11) ----
    const int quarter = warp & 3;
    constexpr int kCols = BN / (P::kEpiWarps / 4);    // columns each warp drains
    const int c_lo = warp >= 8 ? kCols : 0;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // 256-wide tiles (one CTA per SM) have the registers to hold a warp's
    // kCols bf16 results; the 128-wide schedule is capped for two CTAs per SM
    constexpr bool kEarlyRelease = BN == 256;
    bool ok = true;
    for (int i = 0; i < my_tiles; ++i) {
      const int t = blockIdx.x + i * G;
      const int m_tile = t / n_tiles, n_tile = t - (t / n_tiles) * n_tiles;
      const int a = i % P::kAcc;
      const int row = m_tile * kBM + quarter * 32 + lane;
      if (ok) ok = mbar_wait_bounded(&acc_full[a], static_cast<uint32_t>((i / P::kAcc) & 1), FP4Q_WAIT_LIMIT(p));
      ok = __all_sync(0xffffffffu, ok);   // the tensor-memory loads below are warp-wide
      if (!ok && lane == 0) *failed = 1;
      tc_fence_after_sync();
      if (i == my_tiles - 1) griddep_launch_dependents();
      const bool bad = !ok || *failed != 0;
      if (kEarlyRelease && ok && p.residual == nullptr && p.epilogue != kEpiGeluFp4) {
        // bf16 output without a residual: the warp's columns become bf16
        // pairs in registers first and the accumulator is handed back to the
        // MMAs before any store.  (Storing first held the next tile's MMAs
        // about 9300 cycles per tile, 30 % of the tile: a thread per row
        // storing its own 16-byte pieces is slow.)
        uint32_t out2[kCols / 2];
        const int n0 = n_tile * BN + c_lo;
#pragma unroll
        for (int q = 0; q < kCols / 32; ++q) {
          uint32_t r[32];
          tmem_load_32cols(tmem + lane_off + static_cast<uint32_t>(a * BN + c_lo + 32 * q), r);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int n = n0 + 32 * q + 8 * g;
            float acc[8], v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __uint_as_float(r[8 * g + e]);
            if (n < p.N) {
              epilogue_values(p, acc, n, bad, v);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) out2[16 * q + 4 * g + e] = bf16x2_bits(v[2 * e], v[2 * e + 1]);
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
        if (row < p.rows_out) {
#pragma unroll
          for (int q = 0; q < kCols / 8; ++q) {
            const int n = n0 + 8 * q;
            if (n >= p.N) break;
            uint16_t* dst = p.out + static_cast<size_t>(row) * static_cast<size_t>(p.N) + n;
            if (FP4Q_IN_RANGE(p, dst, 16, p.out, 2LL * p.M * p.N))
              *reinterpret_cast<uint4*>(dst) =
                  make_uint4(out2[4 * q], out2[4 * q + 1], out2[4 * q + 2], out2[4 * q + 3]);
          }
        }
      } else if (ok) {
        // residual (added in fp32 before the one rounding) or NVFP4 output
#pragma unroll 1
        for (int c = c_lo; c < c_lo + kCols; c += 32) {
          uint32_t r[32];
          tmem_load_32cols(tmem + lane_off + static_cast<uint32_t>(a * BN + c), r);
          if (row < p.rows_out) store_columns32(p, r, row, n_tile * BN + c, bad);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
      } else if (row < p.rows_out) {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) r[c] = 0;
        for (int c = c_lo; c < c_lo + kCols; c += 32)
          store_columns32(p, r, row, n_tile * BN + c, true);
      }
    }
  }
  __syncthreads();            // every role done; a failure flag is visible to all
  if (*failed != 0 && (warp == 0 || warp == 6) && lane == 0) {
    // as in the one-tile kernel: the last S operand blocks and the last SS
    // scale blocks each producer issued have landed before the CTA ends
    // (earlier ones were consumed, so their copies completed)
    for (int j = issued > S ? issued - S : 0; j < issued; ++j)
      mbar_wait_bounded(&full[j % S], static_cast<uint32_t>((j / S) & 1), FP4Q_WAIT_LIMIT(p));
    for (int j = issued_sf > SS ? issued_sf - SS : 0; j < issued_sf; ++j)
      mbar_wait_bounded(&sf_full[j % SS], static_cast<uint32_t>((j / SS) & 1), FP4Q_WAIT_LIMIT(p));
  }
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *failed != 0 && p.status) atomicExch(p.status, kStatusTimeout);
  if (warp == 1) tmem_dealloc(tmem, p.tmem_cols);
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

// [rows, K/2] bytes, row-major: boxes of box_rows rows x 128 bytes, 128-byte
// swizzle, rows past the end read as zero.
bool encode_operand_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t k_bytes,
                        int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Recently encoded operand maps of this host thread: a model calls the GEMM on
// the same weight and activation buffers again and again, so the descriptor
// of a (buffer, shape) is encoded once.
bool operand_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t k_bytes,
                 int box_rows) {
  struct Entry {
    const uint8_t* base;
    int64_t rows, k_bytes;
    int box_rows;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  thread_local Entry cache[kEntries] = {};
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i) {
    const Entry& e = cache[i];
    if (e.base == base && e.rows == rows && e.k_bytes == k_bytes && e.box_rows == box_rows) {
      *map = e.map;
      return true;
    }
  }
  if (!encode_operand_map(map, base, rows, k_bytes, box_rows)) return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.base = base;
  e.rows = rows;
  e.k_bytes = k_bytes;
  e.box_rows = box_rows;
  e.map = *map;
  return true;
}

// Per device and ring depth, what a kernel instance needs before its launch,
// found once: its dynamic shared memory (raised as far as needed to keep the
// CTAs an SM can hold within its 512 tensor-memory columns: a third CTA's
// allocation would wait for one of the others to exit) and whether it fits.
struct Prep {
  size_t smem = 0;   // 0: not prepared yet
  cudaError_t err = cudaSuccess;
  uint32_t cluster_fits = 0;    // bit c: a cluster of c CTAs fits (tested lazily)
  uint32_t cluster_tested = 0;
};

// One table per kernel instance: an entry per device and ring depth, and the
// largest dynamic shared-memory limit set on the instance per device (the
// limit is a property of the kernel, so it is only ever raised: lowering it
// for a shallower ring would break a deeper one prepared earlier).
struct PrepTable {
  Prep entry[64][9];
  size_t attr[64] = {};
};

std::mutex& prep_mutex() {
  static std::mutex mu;
  return mu;
}

template <typename Kernel>
cudaError_t prepare(PrepTable& table, Kernel kernel, int threads, size_t smem_need,
                    uint32_t tmem_cols, int stages, Prep** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || stages < 0 || stages > 8) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(prep_mutex());
  Prep& pr = table.entry[dev][stages];
  *out = &pr;
  if (pr.smem != 0 || pr.err != cudaSuccess) return pr.err;
  size_t smem = smem_need;
  const int max_ctas = static_cast<int>(512 / tmem_cols);
  int per_sm = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (smem > table.attr[dev]) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) break;
      table.attr[dev] = smem;
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess) break;
    if (per_sm <= max_ctas) break;
    smem = (228 * 1024) / (max_ctas + 1) + 1;
  }
  if (e == cudaSuccess && (per_sm < 1 || per_sm > max_ctas)) e = cudaErrorInvalidConfiguration;
  pr.err = e;
  if (e == cudaSuccess) pr.smem = smem;
  return e;
}

template <typename Kernel>
bool cluster_fits(Prep* pr, Kernel kernel, cudaLaunchConfig_t cfg, int split) {
  std::lock_guard<std::mutex> lock(prep_mutex());
  const uint32_t bit = 1u << split;
  if (pr->cluster_tested & bit) return (pr->cluster_fits & bit) != 0;
  bool ok = true;
  if (split > 8)
    ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
         cudaSuccess;
  if (ok) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(split);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    ok = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) == cudaSuccess && clusters >= 1;
  }
  pr->cluster_tested |= bit;
  if (ok) pr->cluster_fits |= bit;
  return ok;
}

// K blocks of 256 codes, the last one ragged when K % 256 != 0: its K = 64
// steps and its scale tiles (one per step for NVFP4, one per two for MXFP4).
void set_k_blocks(GemmParams& p, bool mx) {
  p.nkt = (p.K + (mx ? 127 : 63)) / (mx ? 128 : 64);   // ceil(K / (4 * block))
  p.num_kb = (p.K + 255) / 256;
  const int rem = p.K - (p.num_kb - 1) * 256;          // 32..256 codes in the last block
  p.mma_last = (rem + 63) / 64;
  p.sf_tiles_last = mx ? (rem + 127) / 128 : p.mma_last;
}

template <int BN, bool SPLIT, bool MX, bool RAG>
cudaError_t launch_bn(const uint8_t* a, const uint8_t* b, GemmParams p, int pdl,
                      cudaStream_t stream) {
  using C = Cfg<BN, MX>;
  auto kernel = gemm_nvfp4_kernel<BN, SPLIT, MX, RAG>;
  CUtensorMap ta, tb;
  if (!operand_map(&ta, a, p.M, p.K / 2, kBM) || !operand_map(&tb, b, p.N, p.K / 2, BN))
    return cudaErrorInvalidValue;
  // The epilogue stages the fp32 tile (128 rows of BN + 4 floats) in the
  // drained operand ring; split K also receives there the rows each peer
  // sends (a slot of ceil(rows / split) rows per rank).  A deeper ring makes
  // the room where the default one is too small.
  const int64_t tile_rows = p.M < kBM ? p.M : kBM;
  const size_t stage_floats =
      static_cast<size_t>(kBM) * (BN + 4) +
      (SPLIT ? static_cast<size_t>(p.split) * ((tile_rows + p.split - 1) / p.split) * (BN + 4) : 0);
  while (static_cast<size_t>(p.stages) * (kTileBytesA + C::kTileBytesB) <
             stage_floats * sizeof(float) && p.stages < 6)
    ++p.stages;
  if (static_cast<size_t>(p.stages) * (kTileBytesA + C::kTileBytesB) < stage_floats * sizeof(float))
    return cudaErrorInvalidValue;
  p.tmem_cols = C::tmem_cols(p.stages);
  set_k_blocks(p, MX);
  const size_t smem_need = C::smem_bytes(p.stages);
  if (smem_need > 227 * 1024) return cudaErrorInvalidValue;
  static PrepTable table;
  Prep* pr = nullptr;
  cudaError_t e = prepare(table, kernel, kTileThreads, smem_need, p.tmem_cols, p.stages, &pr);
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.N + BN - 1) / BN) * (SPLIT ? p.split : 1),
                     static_cast<unsigned>((p.M + kBM - 1) / kBM), 1);
  cfg.blockDim = dim3(kTileThreads, 1, 1);
  cfg.dynamicSmemBytes = pr->smem;
  cfg.stream = stream;
  if (SPLIT && !cluster_fits(pr, kernel, cfg, p.split)) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (SPLIT) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(p.split);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, p);
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev].load(std::memory_order_relaxed) == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached[dev] = n;
  }
  return cached[dev];
}

template <int BN, bool MX, bool RAG>
cudaError_t launch_persistent(const uint8_t* a, const uint8_t* b, GemmParams p, int pdl,
                              cudaStream_t stream) {
  using C = Cfg<BN, MX>;
  using P = PCfg<BN, MX>;
  auto kernel = gemm_nvfp4_persistent_kernel<BN, MX, RAG>;
  CUtensorMap ta, tb;
  if (!operand_map(&ta, a, p.M, p.K / 2, kBM) || !operand_map(&tb, b, p.N, p.K / 2, BN))
    return cudaErrorInvalidValue;
  p.sf_stages = p.stages + P::sf_lead(p.stages);
  if (P::kSfCol + C::kSfColsPerStage * static_cast<uint32_t>(p.sf_stages) > 512)
    return cudaErrorInvalidValue;   // accumulators and scale slots must fit tensor memory
  p.tmem_cols = P::tmem_cols(p.sf_stages);
  set_k_blocks(p, MX);
  const size_t smem_need = P::smem_bytes(p.stages, p.sf_stages);
  if (smem_need > 227 * 1024) return cudaErrorInvalidValue;
  static PrepTable table;
  Prep* pr = nullptr;
  // as many CTAs per SM as tensor memory holds: two 128-wide, one 256-wide
  cudaError_t e = prepare(table, kernel, P::kThreads, smem_need, p.tmem_cols, p.stages, &pr);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  if (sms < 1) return cudaErrorInvalidDevice;
  const int64_t tiles = static_cast<int64_t>((p.N + BN - 1) / BN) * ((p.M + kBM - 1) / kBM);
  const int64_t resident = static_cast<int64_t>(sms) * static_cast<int64_t>(512 / p.tmem_cols);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles < resident ? tiles : resident), 1, 1);
  cfg.blockDim = dim3(P::kThreads, 1, 1);
  cfg.dynamicSmemBytes = pr->smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, p);
}

// One dispatch per operand format, ring shape and K raggedness.
template <bool RAG>
cudaError_t launch_k(const uint8_t* a, const uint8_t* b, const GemmParams& p, int bn,
                     bool persistent, bool mx, int pdl, cudaStream_t stream) {
  if (mx) {
    if (persistent) {
      if (p.split > 1) return cudaErrorInvalidValue;
      if (bn == 128) return launch_persistent<128, true, RAG>(a, b, p, pdl, stream);
      if (bn == 256) return launch_persistent<256, true, RAG>(a, b, p, pdl, stream);
      return cudaErrorInvalidValue;
    }
    if (p.split > 1)
      return bn == 128 && p.split <= 16 ? launch_bn<128, true, true, RAG>(a, b, p, pdl, stream)
                                        : cudaErrorInvalidValue;
    if (bn == 128) return launch_bn<128, false, true, RAG>(a, b, p, pdl, stream);
    if (bn == 256) return launch_bn<256, false, true, RAG>(a, b, p, pdl, stream);
    return cudaErrorInvalidValue;
  }
  if (p.split > 1) {
    if (bn != 128 || persistent || p.split > 16) return cudaErrorInvalidValue;
    return launch_bn<128, true, false, RAG>(a, b, p, pdl, stream);
  }
  if (!persistent) {
    if (bn == 128) return launch_bn<128, false, false, RAG>(a, b, p, pdl, stream);
    if (bn == 256) return launch_bn<256, false, false, RAG>(a, b, p, pdl, stream);
  } else {
    if (bn == 128) return launch_persistent<128, false, RAG>(a, b, p, pdl, stream);
    if (bn == 256) return launch_persistent<256, false, RAG>(a, b, p, pdl, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm_nvfp4(const uint8_t* a, const uint8_t* b, GemmParams p, int bn,
                              bool persistent, bool mx, int pdl, cudaStream_t stream) {
  if (p.stages < 2 || p.stages > 8) return cudaErrorInvalidValue;
  return p.K % 256 != 0 ? launch_k<true>(a, b, p, bn, persistent, mx, pdl, stream)
                        : launch_k<false>(a, b, p, bn, persistent, mx, pdl, stream);
}

}  // namespace fp4q
