// fp32 instantiations of the sampler kernel.
#include "sample_launch.cuh"

namespace pkv {

cudaError_t launch_sample_fp32(const SampleParams& P, const SampleConfig& c, bool all_greedy,
                               cudaStream_t stream) {
  return all_greedy ? launch_sample_dtype<false, true>(P, c, stream)
                    : launch_sample_dtype<false, false>(P, c, stream);
}

}  // namespace pkv
