// debug_checks.h - the checks and fault injection of the debug build of the
// library (compiled with -DFP4Q_DEBUG_CHECKS into libfp4q_debug.so; the
// default build compiles every macro below to nothing).  Internal.
//
// Bounds checks: every global access a kernel computes an address for (row
// loads and stores, packed codes, both scale layouts, the y output, bulk-copy
// sources, GEMM epilogue stores and scale-tile copies) is first compared with
// the extent of its buffer as the C ABI defines it from M, H (or M, N, K) and
// the strides.  An access outside it is counted in a device word the caller
// owns and skipped: nothing traps, nothing is written or read out of bounds.
// A "shrink" knob makes every extent look that many bytes shorter, so a test
// can show that the checks see the accesses near the end of every buffer.
//
// Fault injection: one chosen CTA of the wide-row fused kernel or of the GEMM
// arrives on a stage's barrier expecting the bytes of a copy it then never
// issues, and every bounded wait uses a caller-given limit: the wait on that
// stage runs out with no copy in flight for it, and the kernel's timeout path
// (marked outputs, the device status word) runs as it would on a real fault.
#pragma once

#include <cstddef>
#include <cstdint>

namespace fp4q {

struct DebugKnobs {
  long long wait_limit;       // clock cycles of every bounded wait
  long long shrink;           // bytes taken off every extent the checks use
  int drop_kernel;            // 0 none, 1 wide-row fused kernel, 2 GEMM
  int drop_cta;               // linear CTA index whose copy is dropped
  int drop_iter;              // its ring iteration (fused) or K-block count (GEMM)
  unsigned int* violations;   // device counter of out-of-bounds accesses (skipped)
};

#ifdef FP4Q_DEBUG_CHECKS
// The knobs set with fp4_debug_configure (process-wide), copied into every
// launch's parameters.
DebugKnobs debug_knobs();

#define FP4Q_DEBUG_FIELD DebugKnobs dbg;
#define FP4Q_SET_DEBUG(p) ((p).dbg = debug_knobs())
#define FP4Q_WAIT_LIMIT(p) ((p).dbg.wait_limit)
#define FP4Q_DROP(p, kernel, cta, iter) \
  ((p).dbg.drop_kernel == (kernel) && (p).dbg.drop_cta == (cta) && (p).dbg.drop_iter == (iter))
// true if [ptr, ptr + bytes) lies inside [base, base + size - shrink); else
// the violation is counted and false returned (the caller skips the access)
#define FP4Q_IN_RANGE(p, ptr, bytes, base, size) \
  debug_in_range((p).dbg, (ptr), (bytes), (base), (size))
#ifdef __CUDACC__
__device__ __forceinline__ bool debug_in_range(const DebugKnobs& d, const void* ptr, size_t bytes,
                                               const void* base, long long size) {
  const long long off = static_cast<long long>(reinterpret_cast<uintptr_t>(ptr) -
                                               reinterpret_cast<uintptr_t>(base));
  if (base != nullptr && off >= 0 && off + static_cast<long long>(bytes) <= size - d.shrink)
    return true;
  if (d.violations) atomicAdd(d.violations, 1u);
  return false;
}
#endif
#else
#define FP4Q_DEBUG_FIELD
#define FP4Q_SET_DEBUG(p) ((void)0)
#define FP4Q_WAIT_LIMIT(p) kWaitLimitCycles
#define FP4Q_DROP(p, kernel, cta, iter) false
#define FP4Q_IN_RANGE(p, ptr, bytes, base, size) true
#endif

}  // namespace fp4q
