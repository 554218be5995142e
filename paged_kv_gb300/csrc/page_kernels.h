// Host-side declarations of the page-fill and write-back launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kMaxFillBatch = 4096;

struct FillParams {
  const int32_t* cached_len;   // [B]
  const int32_t* device_len;   // [B]
  const int32_t* table_idx;    // [B]
  int B;
  int page_size;
  const int32_t* free_slots;   // [free_count] page-start token locations
  int64_t free_count;
  int32_t* page_table;         // [pt_rows, pt_cols]
  int64_t pt_rows;
  int64_t pt_cols;
  int64_t* total_out;          // device, or nullptr
  int32_t* status;             // device, or nullptr
  bool vec4;                   // 16-byte stores are aligned (ps % 4 == 0, pt_cols % 4 == 0)
};

// Batched lazy free (free_kernels.cu).
struct FreeParams {
  const int32_t* table_idx;    // [B]
  const int32_t* begin;        // [B] first freed column of the row
  const int32_t* end;          // [B] one past the last freed column
  int B;
  int page_size;
  const int32_t* page_table;   // [pt_rows, pt_cols]
  int64_t pt_rows;
  int64_t pt_cols;
  int32_t* free_slots;         // [capacity], entries [0, free_count) live
  int64_t free_count;
  int64_t capacity;
  int64_t* total_out;          // device, or nullptr
  int32_t* status;             // device, or nullptr
};

size_t free_smem_bytes(int B);
cudaError_t launch_free_pages(const FreeParams& F, int num_sms, cudaStream_t stream);
cudaError_t launch_check_free_list(const int32_t* free_slots, int64_t free_count, int page_size,
                                   int64_t num_pages, int64_t cache_pages, uint32_t* bitmap,
                                   int32_t* result, int num_sms, cudaStream_t stream);

// The step before the model (prepare_kernels.cu): the page fill of `fill`
// plus the packed positions and the two gathers.
struct PrepareParams {
  FillParams fill;             // total_out receives the pages allocated
  const int32_t* token_pool;   // [pool_rows, pool_cols]
  int64_t pool_rows;
  int64_t pool_cols;
  int32_t* positions;          // [max_tokens]
  int32_t* input_ids;          // [max_tokens]
  int32_t* out_loc;            // [max_tokens]
  int64_t max_tokens;
  int64_t* tokens_out;         // device, or nullptr: the step's token count
};

size_t prepare_smem_bytes(int B);
cudaError_t launch_prepare_step(const PrepareParams& Q, int num_sms, cudaStream_t stream);

// Counter-based uniforms of one sampler call (philox_kernels.cu).
cudaError_t launch_uniforms(uint64_t seed, uint64_t offset, int B, float* u, cudaStream_t stream);

size_t fill_smem_bytes(int B);
cudaError_t launch_fill_page_table(const FillParams& F, int num_sms, cudaStream_t stream);
cudaError_t launch_writeback(const int32_t* tokens, const int32_t* rows, const int64_t* cols,
                             int B, int32_t* pool, int64_t pool_rows, int64_t pool_cols,
                             int32_t* status, cudaStream_t stream);

}  // namespace pkv
