// Counter-based uniforms for the sampler's draw, for sm_103a.  The pages seed
// one generator per engine (torch.manual_seed(42) in Engine) so that every
// tensor-parallel rank draws the same tokens ("The scheduler's IO and
// multi-rank synchronization", section "Sending results"); with a
// counter-based generator each (call, row) pair has its own number, so the
// ranks agree with no generator state to keep in step and the uniforms never
// cross from the host.
//
// Philox-4x64 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): per round, words 0 and 2 are
// multiplied by two odd 64-bit constants; the high halves are XORed with
// words 1 and 3 and the round key, the low halves move into words 1 and 3;
// the key is bumped by two Weyl increments.  Row b of call `offset` uses
// counter (b, offset, 0, 0) and key (seed, 0); its uniform is the top 24
// bits of the first output word times 2^-24, exact in fp32 and in [0, 1).

#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

namespace {

constexpr int kPhiloxThreads = 256;

struct Block4 {
  uint64_t x0, x1, x2, x3;
};

__device__ __forceinline__ Block4 philox4x64_10(Block4 c, uint64_t k0, uint64_t k1) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t hi0 = __umul64hi(kM0, c.x0), lo0 = kM0 * c.x0;
    const uint64_t hi1 = __umul64hi(kM1, c.x2), lo1 = kM1 * c.x2;
    c = Block4{hi1 ^ c.x1 ^ k0, lo1, hi0 ^ c.x3 ^ k1, lo0};
    k0 += kW0;
    k1 += kW1;
  }
  return c;
}

__global__ void __launch_bounds__(kPhiloxThreads) uniforms_kernel(uint64_t seed, uint64_t offset,
                                                                  int B, float* u) {
  const int b = blockIdx.x * kPhiloxThreads + threadIdx.x;
  if (b >= B) return;
  const Block4 out = philox4x64_10(Block4{static_cast<uint64_t>(b), offset, 0ull, 0ull}, seed, 0ull);
  u[b] = static_cast<float>(static_cast<uint32_t>(out.x0 >> 40)) * 0x1p-24f;
}

}  // namespace

cudaError_t launch_uniforms(uint64_t seed, uint64_t offset, int B, float* u, cudaStream_t stream) {
  const int grid = (B + kPhiloxThreads - 1) / kPhiloxThreads;
  uniforms_kernel<<<grid, kPhiloxThreads, 0, stream>>>(seed, offset, B, u);
  return cudaGetLastError();
}

}  // namespace pkv
