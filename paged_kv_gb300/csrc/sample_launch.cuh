// Launch of the two sampler kernels for one logits dtype: the persistent
// stream kernel, then the finish kernel as its programmatic dependent.
// Included by exactly one translation unit per dtype so that the
// instantiations compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "device_attr.h"
#include "launch_config.h"
#include "sample_finish.cuh"
#include "sample_stream.cuh"

namespace pkv {

template <bool BF16, int NV, bool VEC>
cudaError_t launch_pair(const SampleParams& P, int num_sms, cudaStream_t stream) {
  auto skern = stream_kernel<BF16, NV, VEC>;
  auto fkern = finish_kernel<BF16, NV, VEC>;
  constexpr int kStreamDyn = stream_dyn_bytes<NV>();
  constexpr int kFinishDyn = kFinishDynBytes;
  // The shared-memory limits are per device: set once on each device.
  static std::atomic<unsigned long long> stream_set{0ull}, finish_set{0ull};
  cudaError_t e = set_smem_limit_once(stream_set, skern, kStreamDyn);
  if (e != cudaSuccess) return e;
  e = set_smem_limit_once(finish_set, fkern, kFinishDyn);
  if (e != cudaSuccess) return e;
  const int items = P.B * P.chunks;
  const int ctas = std::min(num_sms, (items + kGroups - 1) / kGroups);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = kStreamDyn;
  cfg.stream = stream;
  e = cudaLaunchKernelEx(&cfg, skern, P);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t fcfg = {};
  fcfg.gridDim = dim3(static_cast<unsigned>(P.B + P.fill_ctas), 1, 1);
  fcfg.blockDim = dim3(kThreads, 1, 1);
  fcfg.dynamicSmemBytes = kFinishDyn;
  fcfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  fcfg.attrs = attr;
  fcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&fcfg, fkern, P);
}

template <bool BF16>
cudaError_t launch_sample_dtype(const SampleParams& P, const SampleConfig& c, int num_sms,
                                cudaStream_t stream) {
  if (!c.vec) {
    if (c.nv == 10) return launch_pair<BF16, 10, false>(P, num_sms, stream);
    return launch_pair<BF16, kNvScalar, false>(P, num_sms, stream);
  }
  switch (c.nv) {
    case 4: return launch_pair<BF16, 4, true>(P, num_sms, stream);
    case 8: return launch_pair<BF16, 8, true>(P, num_sms, stream);
    case 10: return launch_pair<BF16, 10, true>(P, num_sms, stream);
    case 16: return launch_pair<BF16, 16, true>(P, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
