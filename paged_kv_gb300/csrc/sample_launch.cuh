// Cluster launch of the sampler kernel for one logits dtype.  Included by
// exactly one translation unit per dtype so that the instantiations compile in
// parallel.
#pragma once

#include <cuda_runtime.h>

#include "launch_config.h"
#include "sample_kernel.cuh"

namespace pkv {

template <bool BF16, int NV, bool VEC, bool AG>
cudaError_t launch_one(SampleParams P, int C, cudaStream_t stream) {
  auto kern = sample_kernel<BF16, NV, VEC, AG>;
  // An all-greedy batch uses neither the candidate list nor the histograms.
  const size_t dyn = AG ? 0 : static_cast<size_t>(sample_dyn_bytes<NV>());
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
  P.list_cap = kListCap;
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
  if (!c.vec) {
    if (c.nv == 10) return launch_one<BF16, 10, false, AG>(P, c.cluster, stream);
    return launch_one<BF16, kNvScalar, false, AG>(P, c.cluster, stream);
  }
  switch (c.nv) {
    case 4: return launch_one<BF16, 4, true, AG>(P, c.cluster, stream);
    case 8: return launch_one<BF16, 8, true, AG>(P, c.cluster, stream);
    case 10: return launch_one<BF16, 10, true, AG>(P, c.cluster, stream);
    case 16: return launch_one<BF16, 16, true, AG>(P, c.cluster, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
