// fused_launch.cuh - launch helpers instantiated once per storage dtype.
#pragma once

#include <mutex>

#include "fused_direct.cuh"
#include "fused_tma.cuh"

namespace fp4q {

template <typename T, int FMT, int CPT, bool EX>
cudaError_t raise_smem_limit(size_t smem) {
  // The limit is a per-device function attribute, only ever raised: a launch
  // that needs more than any earlier one on this device raises it to its own
  // need.  The check, the attribute call and the record happen under one
  // lock, so two host threads cannot lower the limit below what either has
  // launched with.
  static size_t done[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev] >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(fused_tma_kernel<T, FMT, CPT, EX>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) done[dev] = smem;
  return e;
}

template <typename T, int FMT, int CPT>
int ctas_per_sm_one(int threads, size_t smem) {
  // the last answer per device is kept: calls repeat the same launch shape
  struct Last { int threads; size_t smem; int n; };
  static Last last[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool cacheable = dev >= 0 && dev < 64;
  if (cacheable) {
    std::lock_guard<std::mutex> lock(mu);
    if (last[dev].n > 0 && last[dev].threads == threads && last[dev].smem == smem)
      return last[dev].n;
  }
  if (raise_smem_limit<T, FMT, CPT, false>(smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_tma_kernel<T, FMT, CPT, false>, threads,
                                                    smem) != cudaSuccess)
    return 0;
  if (cacheable) {
    std::lock_guard<std::mutex> lock(mu);
    last[dev] = Last{threads, smem, n};
  }
  return n;
}

template <typename T, int FMT>
int ctas_per_sm_fmt(int cpt, int threads, size_t smem) {
  switch (cpt) {
    case 1: return ctas_per_sm_one<T, FMT, 1>(threads, smem);
    case 2: return ctas_per_sm_one<T, FMT, 2>(threads, smem);
    case 3: return ctas_per_sm_one<T, FMT, 3>(threads, smem);
    case 4: return ctas_per_sm_one<T, FMT, 4>(threads, smem);
    default: return 0;
  }
}

template <typename T>
int ctas_per_sm_dtype(int fmt, int cpt, int threads, size_t smem) {
  switch (fmt) {
    case kFmtNV: return ctas_per_sm_fmt<T, kFmtNV>(cpt, threads, smem);
    case kFmtMX: return ctas_per_sm_fmt<T, kFmtMX>(cpt, threads, smem);
    case kFmtE4B32: return ctas_per_sm_fmt<T, kFmtE4B32>(cpt, threads, smem);
    default: return 0;
  }
}

// EX selects the general instance (strided rows and/or y output); dense calls
// without y run the common instance, which carries none of that code.
template <typename T, int FMT, int CPT, bool EX>
cudaError_t launch_one(const FusedShape& s, const FusedParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(s.threads), 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (s.pdl) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  if (s.path == kPathDirect) {
    if (s.cluster > 1) {
      attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
      attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(s.cluster);
      attr[cfg.numAttrs].val.clusterDim.y = 1;
      attr[cfg.numAttrs].val.clusterDim.z = 1;
      ++cfg.numAttrs;
    }
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, fused_direct_kernel<T, FMT, CPT, EX>, p);
  }
  const cudaError_t e = raise_smem_limit<T, FMT, CPT, EX>(s.smem);
  if (e != cudaSuccess) return e;
  cfg.dynamicSmemBytes = s.smem;
  return cudaLaunchKernelEx(&cfg, fused_tma_kernel<T, FMT, CPT, EX>, p);
}

template <typename T, int FMT>
cudaError_t launch_fmt(const FusedShape& s, const FusedParams& p, cudaStream_t stream) {
  const bool y = p.y != nullptr || p.x_stride != p.H || p.r_stride != p.H;
  switch (s.cpt) {
    case 1: return y ? launch_one<T, FMT, 1, true>(s, p, stream) : launch_one<T, FMT, 1, false>(s, p, stream);
    case 2: return y ? launch_one<T, FMT, 2, true>(s, p, stream) : launch_one<T, FMT, 2, false>(s, p, stream);
    case 3: return y ? launch_one<T, FMT, 3, true>(s, p, stream) : launch_one<T, FMT, 3, false>(s, p, stream);
    case 4: return y ? launch_one<T, FMT, 4, true>(s, p, stream) : launch_one<T, FMT, 4, false>(s, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_dtype(int fmt, const FusedShape& s, const FusedParams& p, cudaStream_t stream) {
  switch (fmt) {
    case kFmtNV: return launch_fmt<T, kFmtNV>(s, p, stream);
    case kFmtMX: return launch_fmt<T, kFmtMX>(s, p, stream);
    case kFmtE4B32: return launch_fmt<T, kFmtE4B32>(s, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp4q
