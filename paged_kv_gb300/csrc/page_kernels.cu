// Paged-KV bookkeeping and token write-back kernels for sm_103a.
//
// Page fill: the standalone kernel runs page_fill_cta (page_fill.cuh) on a
// grid of one CTA per SM.
//
// Write-back ("The scheduler skeleton and the offline interface", section
// "Preparing a batch": token_pool[write_tuple] = next_tokens) is a plain
// bounds-checked scatter.

#include <cstdint>
#include <cuda_runtime.h>

#include <atomic>

#include "device_attr.h"
#include "page_fill.cuh"
#include "page_kernels.h"

namespace pkv {

namespace {

constexpr int kFillThreads = 512;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;

__global__ void __launch_bounds__(kFillThreads) fill_page_table_kernel(const FillParams F) {
  extern __shared__ int32_t smem[];
  fill::page_fill_cta<kFillThreads>(F, smem, blockIdx.x, gridDim.x, threadIdx.x,
                                    []() { __syncthreads(); });
}

__global__ void writeback_kernel(const int32_t* __restrict__ tokens,
                                 const int32_t* __restrict__ rows,
                                 const int64_t* __restrict__ cols, int B, int32_t* pool,
                                 int64_t pool_rows, int64_t pool_cols, int32_t* status) {
  int st = 0;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    const int64_t c = cols[b];
    const int32_t tok = tokens[b];
    if (c < 0 || tok < 0) continue;
    const int64_t r = rows[b];
    if (r < 0 || r >= pool_rows) {
      st |= kStRowOOB;
    } else if (c >= pool_cols) {
      st |= kStColOOB;
    } else {
      pool[r * pool_cols + c] = tok;
    }
  }
  if (st != 0 && status != nullptr) atomicOr(status, st);
}

}  // namespace

size_t fill_smem_bytes(int B) { return fill::smem_bytes(B); }

cudaError_t launch_fill_page_table(const FillParams& F, int num_sms, cudaStream_t stream) {
  const size_t smem = fill_smem_bytes(F.B);
  static std::atomic<unsigned long long> smem_set{0ull};
  const cudaError_t e = set_smem_limit_once(smem_set, fill_page_table_kernel,
                                            static_cast<int>(fill_smem_bytes(kMaxFillBatch)));
  if (e != cudaSuccess) return e;
  // Enough CTAs to cover the device; each recomputes the (cheap) scan.
  const int grid = num_sms > 0 ? num_sms : 1;
  fill_page_table_kernel<<<grid, kFillThreads, smem, stream>>>(F);
  return cudaGetLastError();
}

cudaError_t launch_writeback(const int32_t* tokens, const int32_t* rows, const int64_t* cols,
                             int B, int32_t* pool, int64_t pool_rows, int64_t pool_cols,
                             int32_t* status, cudaStream_t stream) {
  const int threads = 256;
  const int grid = (B + threads - 1) / threads;
  writeback_kernel<<<grid, threads, 0, stream>>>(tokens, rows, cols, B, pool, pool_rows,
                                                  pool_cols, status);
  return cudaGetLastError();
}

}  // namespace pkv
