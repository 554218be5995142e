// fp32 instantiations of the sampler kernels.
#include <algorithm>

#include "sample_launch.cuh"

namespace pkv {

cudaError_t launch_sample_fp32(const SampleParams& P, const SampleConfig& c, int num_sms,
                               cudaStream_t stream) {
  return launch_sample_dtype<false>(P, c, num_sms, stream);
}

}  // namespace pkv
