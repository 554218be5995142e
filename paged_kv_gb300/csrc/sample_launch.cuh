// Cluster launch of the sampler kernel for one logits dtype.  Included by
// exactly one translation unit per dtype so that the instantiations compile in
// parallel.
#pragma once

#include <cuda_runtime.h>

#include "launch_config.h"
#include "sample_kernel.cuh"

namespace pkv {

// Candidate-list capacity: as large as fits next to the slice while keeping
// three CTAs per SM (else two, else one), at most 4096 entries.
inline int list_capacity(size_t slice_bytes) {
  constexpr size_t kSmemPerSm = 228 * 1024;
  constexpr size_t kPerCtaReserved = 1024;
  constexpr size_t kStatic = sizeof(SampleSmem) + 256;
  for (int per_sm = 3; per_sm >= 1; --per_sm) {
    const size_t budget = kSmemPerSm / per_sm;
    const size_t used = kPerCtaReserved + kStatic + slice_bytes;
    if (budget <= used) continue;
    size_t cap = (budget - used) / 8;
    if (cap > 4096) cap = 4096;
    cap = cap / 256 * 256;
    if (cap >= 1024) return static_cast<int>(cap);
  }
  return 1024;
}

template <bool BF16, int NV, bool VEC, bool AG>
cudaError_t launch_one(SampleParams P, int C, cudaStream_t stream) {
  auto kern = sample_kernel<BF16, NV, VEC, AG>;
  constexpr size_t kSliceBytes = static_cast<size_t>(kThreads) * NV * 16;
  static const int cap = list_capacity(kSliceBytes);
  // An all-greedy batch uses neither the slice copy nor the list.
  const size_t dyn = AG ? 0 : kSliceBytes + static_cast<size_t>(cap) * 8;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaSuccess;
    if (dyn > 0) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(dyn));
      if (e != cudaSuccess) return e;
    }
    // Clusters of 9..16 CTAs are a non-portable size; opt in once per kernel.
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  P.list_cap = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C), static_cast<unsigned>(P.B), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <bool BF16, bool AG>
cudaError_t launch_sample_dtype(const SampleParams& P, const SampleConfig& c,
                                cudaStream_t stream) {
  if (!c.vec) return launch_one<BF16, kNvScalar, false, AG>(P, c.cluster, stream);
  switch (c.nv) {
    case 4: return launch_one<BF16, 4, true, AG>(P, c.cluster, stream);
    case 8: return launch_one<BF16, 8, true, AG>(P, c.cluster, stream);
    case 10: return launch_one<BF16, 10, true, AG>(P, c.cluster, stream);
    case 16: return launch_one<BF16, 16, true, AG>(P, c.cluster, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
