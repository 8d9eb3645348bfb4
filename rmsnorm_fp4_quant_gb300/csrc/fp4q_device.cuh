// fp4q_device.cuh - device building blocks for the sm_103a kernels:
// 256-bit global accesses, bf16/fp16 pair conversion, the E4M3 / UE8M0 scale
// rules and E2M1 code packing, and the 128x4 tiled scale offset.
//
// Rounding rules (FlashInfer `add_rmsnorm_fp4quant.py`, Notes and kernel phase
// 3; the helper bodies it imports are not on the page, so the rule is stated
// here): E4M3 scale = nearest-even of min(amax/6, 448); UE8M0 scale = the power
// of two at or above amax/6; E2M1 code = nearest-even on {0,.5,1,1.5,2,3,4,6},
// saturating, sign kept.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace fp4q {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// 256-bit global memory accesses (sm_100+ vector width).  One thread moves one
// 16-element chunk of a bf16/fp16 row, so a warp covers 1 KiB contiguously.
// ---------------------------------------------------------------------------
struct Chunk { uint32_t u[8]; };   // 16 x 16-bit elements, element 2j in the low half of u[j]

// Streaming read of data this kernel never writes (the input).
__device__ __forceinline__ Chunk ld_stream_ro(const void* p) {
  Chunk c;
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3]),
                 "=r"(c.u[4]), "=r"(c.u[5]), "=r"(c.u[6]), "=r"(c.u[7])
               : "l"(p));
  return c;
}

// Streaming read that should also leave L2 first (evict-first): the
// standalone quantize reads each input byte once and writes far less, so
// its input should not push out lines still being written back.
__device__ __forceinline__ Chunk ld_stream_ro_evict_first(const void* p) {
  Chunk c;
  asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3]),
                 "=r"(c.u[4]), "=r"(c.u[5]), "=r"(c.u[6]), "=r"(c.u[7])
               : "l"(p));
  return c;
}

// Streaming read of data the same thread overwrites later (the residual):
// coherent load, no L1 allocation.
__device__ __forceinline__ Chunk ld_stream_rw(const void* p) {
  Chunk c;
  asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3]),
                 "=r"(c.u[4]), "=r"(c.u[5]), "=r"(c.u[6]), "=r"(c.u[7])
               : "l"(p));
  return c;
}

// Re-used read (the weight): cached in L1 so every row of a CTA hits.
__device__ __forceinline__ Chunk ld_cached_ro(const void* p) {
  Chunk c;
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(c.u[0]), "=r"(c.u[1]), "=r"(c.u[2]), "=r"(c.u[3]),
                 "=r"(c.u[4]), "=r"(c.u[5]), "=r"(c.u[6]), "=r"(c.u[7])
               : "l"(p));
  return c;
}

__device__ __forceinline__ void st_stream(void* p, const Chunk& c) {
  asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "l"(p), "r"(c.u[0]), "r"(c.u[1]), "r"(c.u[2]), "r"(c.u[3]),
                  "r"(c.u[4]), "r"(c.u[5]), "r"(c.u[6]), "r"(c.u[7])
               : "memory");
}

__device__ __forceinline__ void st_u64(void* p, uint64_t v) {
  asm volatile("st.global.L1::no_allocate.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_u32(void* p, uint32_t v) {
  asm volatile("st.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_u8(void* p, uint32_t v) {
  asm volatile("st.global.b8 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// 16-bit storage types: unpack a pair to fp32 (exact), round a pair of fp32 to
// the type, add two pairs, multiply two pairs into fp32, accumulate squares.
// ---------------------------------------------------------------------------
template <typename T> struct Pair;

// add() is the packed add.rn of the storage type: the exact sum rounded once
// to nearest-even in that type, which is what rounding the fp32 sum gives
// (fp32 carries more than 2p + 2 bits for p = 8 and 11).
// mul() gives the two fp32 products of two pairs with the mixed-precision FMA
// (16-bit sources, fp32 result, addend -0 so a zero product keeps its sign):
// a product of two 8- or 11-bit significands is exact in fp32.  sq_acc()
// accumulates the squares of a pair the same way, into two fp32 lanes.
#define FP4Q_PAIR_OPS(T16, ADD, MIXED)                                                        \
  static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {                   \
    uint32_t d;                                                                               \
    asm(ADD " %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));                                       \
    return d;                                                                                 \
  }                                                                                           \
  static __device__ __forceinline__ float2 mul(uint32_t a, uint32_t b) {                     \
    float2 r;                                                                                 \
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"                                                 \
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"                                  \
        MIXED " %0, al, bl, 0f80000000;\n\t" MIXED " %1, ah, bh, 0f80000000;\n\t}"            \
        : "=f"(r.x), "=f"(r.y) : "r"(a), "r"(b));                                             \
    return r;                                                                                 \
  }                                                                                           \
  static __device__ __forceinline__ void sq_acc(uint32_t a, float2& acc) {                   \
    asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"                               \
        MIXED " %0, al, al, %0;\n\t" MIXED " %1, ah, ah, %1;\n\t}"                              \
        : "+f"(acc.x), "+f"(acc.y) : "r"(a));                                                 \
  }

template <> struct Pair<__nv_bfloat16> {
  static __device__ __forceinline__ float2 to_f32(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static __device__ __forceinline__ uint32_t from_f32(float lo, float hi) {   // nearest-even
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  FP4Q_PAIR_OPS(__nv_bfloat16, "add.rn.bf16x2", "fma.rn.f32.bf16")
};

template <> struct Pair<__half> {
  static __device__ __forceinline__ float2 to_f32(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    return __half22float2(v);
  }
  static __device__ __forceinline__ uint32_t from_f32(float lo, float hi) {   // nearest-even
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  FP4Q_PAIR_OPS(__half, "add.rn.f16x2", "fma.rn.f32.f16")
};
#undef FP4Q_PAIR_OPS

// max(m, |a|, |b|) with the three-input float max of sm_100+.
__device__ __forceinline__ float max_abs3(float m, float a, float b) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
  return d;
}

// ---------------------------------------------------------------------------
// Block scales (FlashInfer kernel phase 3: the block scale is decoded and its
// reciprocal scales y before E2M1 rounding).  Both return the scale byte and
// inv_s, the nearest fp32 to 1/s that the element loop multiplies by.
// ---------------------------------------------------------------------------

// amax / 6 correctly rounded.  For a in [2^-125, FLT_MAX] the product with
// rn(1/6), corrected once by its fma remainder (Markstein's correction step),
// equals the correctly rounded quotient; tests/test_div6_gpu.py checks this
// against CUDA's __fdiv_rn for every float in that range.  Below it the
// quotient is subnormal and CUDA's division is used.
__device__ __forceinline__ float div6_rn(float a) {
  if (a >= __uint_as_float(0x01000000u) && a <= __uint_as_float(0x7F7FFFFFu)) {
    const float c6 = __uint_as_float(0x3E2AAAABu);   // rn(1/6)
    const float q = __fmul_rn(a, c6);
    return __fmaf_rn(__fmaf_rn(-q, 6.0f, a), c6, q);
  }
  return __fdiv_rn(a, 6.0f);
}

// E4M3 byte -> fp32 (exact): exponent field E (bias 7), mantissa m (3 bits);
// E = 0 is subnormal, m * 2^-9.
__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xF;
  const uint32_t m = code & 0x7;
  const float sig = static_cast<float>(e ? (8u + m) : m);          // integer significand
  const float pw = __uint_as_float(((e ? e : 1u) + 117u) << 23);    // 2^(max(E,1) - 10)
  return sig * pw;
}

// E4M3 scales (NVFP4, and 32-element blocks with E4M3 forced): t =
// min((gs * amax) / 6, 448) with correctly rounded ops, then E4M3 nearest-even
// (CUDA's satfinite fp8 conversion).  inv_s = rn(rn(1/s) * gs) (0 when s = 0,
// which turns every element of the block into code 0).  gs = 1 without a
// global scale.
__device__ __forceinline__ uint32_t e4m3_block_scale(float amax, float gs, float& inv_s) {
  const float t = fminf(div6_rn(__fmul_rn(gs, amax)), 448.0f);
  const uint32_t code = static_cast<uint32_t>(__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
  const float s = e4m3_decode(code);
  inv_s = s > 0.0f ? __fmul_rn(__frcp_rn(s), gs) : 0.0f;
  return code;
}

// UE8M0 scales (MXFP4; the global scale does not apply): t = amax / 6
// (correctly rounded); exponent e = ceil(log2 t) read off
// the fp32 encoding (an exact power of two keeps its exponent, anything above
// it steps up), clamped to [-127, 127]; byte = e + 127.  inv_s = 2^-e exactly,
// so y * inv_s is the correctly rounded y / s.
__device__ __forceinline__ uint32_t ue8m0_block_scale(float amax, float& inv_s) {
  const float t = div6_rn(amax);
  const uint32_t bits = __float_as_uint(t);
  const int E = static_cast<int>(bits >> 23);   // t >= 0: no sign bit
  const uint32_t man = bits & 0x7FFFFFu;
  int e;
  if (E == 0) {
    e = (man <= 0x400000u) ? -127 : -126;      // t <= 2^-127  /  2^-127 < t < 2^-126
  } else {
    e = E - 127 + (man != 0u ? 1 : 0);
  }
  e = min(max(e, -127), 127);
  const int inv_biased = 127 - e;               // biased exponent of 2^-e, in [0, 254]
  inv_s = inv_biased ? __uint_as_float(static_cast<uint32_t>(inv_biased) << 23)
                     : __uint_as_float(0x00400000u);   // 2^-127 is subnormal
  return static_cast<uint32_t>(e + 127);
}

// ---------------------------------------------------------------------------
// E2M1 codes: cvt.rn.satfinite.e2m1x2.f32 rounds two fp32 values to nearest
// even and saturates at +-6; the first source lands in the high nibble.
// pack8 returns 8 codes (4 bytes), element 2j in the low nibble of byte j.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e2m1_pack8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// ---------------------------------------------------------------------------
// 128x4 tiled scale layout (FlashInfer `add_rmsnorm_fp4quant`, parameter
// `is_sf_swizzled_layout`): tile (m/128, k/4) of 512 bytes, row m%32 at 16-byte
// stride, row quarter (m%128)/32 at 4-byte stride, k%4 innermost.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t tiled_sf_offset(int64_t m, int k, int nkt) {
  return (m >> 7) * static_cast<int64_t>(nkt) * 512 + static_cast<int64_t>(k >> 2) * 512 +
         (m & 31) * 16 + ((m & 127) >> 5) * 4 + (k & 3);
}

}  // namespace fp4q
