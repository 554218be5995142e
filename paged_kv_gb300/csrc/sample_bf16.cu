// bf16 instantiations of the sampler kernel.
#include "sample_launch.cuh"

namespace pkv {

cudaError_t launch_sample_bf16(const SampleParams& P, const SampleConfig& c, bool all_greedy,
                               cudaStream_t stream) {
  return all_greedy ? launch_sample_dtype<true, true>(P, c, stream)
                    : launch_sample_dtype<true, false>(P, c, stream);
}

}  // namespace pkv
