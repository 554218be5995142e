// Launch parameters of the sampler kernel (host and device side).
#pragma once

#include <cstdint>

namespace pkv {

struct SampleParams {
  const void* logits;        // [B, row_stride] fp32 or bf16
  int64_t row_stride;        // elements
  int B;
  int V;
  const float* temperature;  // [B] or nullptr (all greedy)
  const int32_t* top_k;      // [B] or nullptr
  const float* top_p;        // [B] or nullptr
  const float* uniform;      // [B] (sampled rows)
  int32_t* out_tokens;       // [B]
  int32_t* token_pool;       // [pool_rows, pool_cols] or nullptr
  int64_t pool_rows;
  int64_t pool_cols;
  const int32_t* wb_rows;    // [B]
  const int64_t* wb_cols;    // [B]
  float* probs_out;          // [B, V] or nullptr
  int32_t* status;           // device status word or nullptr
  int cta_chunk;             // elements owned by one CTA of a row's cluster
  int list_cap;              // candidate-list entries in the leader's shared memory
};

}  // namespace pkv
