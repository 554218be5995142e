// bf16 instantiations of the sampler kernels.
#include <algorithm>

#include "sample_launch.cuh"

namespace pkv {

cudaError_t launch_sample_bf16(const SampleParams& P, const SampleConfig& c, int num_sms,
                               cudaStream_t stream) {
  return launch_sample_dtype<true>(P, c, num_sms, stream);
}

}  // namespace pkv
