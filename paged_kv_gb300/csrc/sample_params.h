// Launch parameters of the sampler kernel (host and device side).
#pragma once

#include <cstddef>
#include <cstdint>

#include "page_kernels.h"

namespace pkv {

// Bytes of one workspace record (ChunkSlot in sample_common.cuh): a 16-byte
// summary, 4 words per warp, a float per thread and a 2 KB histogram.
constexpr size_t kChunkSlotBytes = 16 + 128 + 256 * 4 + 2048;

// The workspace starts with this header; the records follow it.  It must be
// zero before the first call; every call leaves it ready for the next one.
struct WorkspaceHeader {
  uint32_t ticket;        // next ticket of the stream kernel's main queue
  uint32_t done;          // stream CTAs finished in this call
  uint32_t calls;         // calls completed; records of call n carry n + 1
  uint32_t ticket_heavy;  // next ticket of the queue of count-histogram items
  uint32_t pad[60];
};
constexpr size_t kWorkspaceHeaderBytes = 256;
static_assert(sizeof(WorkspaceHeader) == kWorkspaceHeaderBytes, "header size");

// After the header: the records, then one block of slice histograms per
// (row, chunk): for each of the stream kernel's 8 consumer warps, the 16-bit
// counts of the 1024 keys below the chunk maximum over that warp's slice of
// the chunk (written for count-histogram rows only, which are bf16 rows:
// fp32 workspaces have no slice histograms).  Batches of up to kOrderRows
// rows are streamed in cost order (the order lives in the stream kernel's
// shared memory).
constexpr int kOrderRows = 4096;
constexpr size_t kRecordsOffset = kWorkspaceHeaderBytes;
constexpr size_t kSliceHistBytes = 8 * 1024 * 2;

// Workspace bytes for B rows of `chunks` chunks of bf16 or fp32 logits.
inline size_t sample_workspace_need(int B, int chunks, bool bf16) {
  return kRecordsOffset +
         static_cast<size_t>(B) * chunks * (kChunkSlotBytes + (bf16 ? kSliceHistBytes : 0));
}

struct SampleParams {
  const void* logits;        // [B, row_stride] fp32 or bf16
  int64_t row_stride;        // elements
  int B;
  int V;
  const float* temperature;  // [B] or nullptr (all greedy)
  const int32_t* top_k;      // [B] or nullptr
  const float* top_p;        // [B] or nullptr
  const float* min_p;        // [B] or nullptr (off)
  const float* uniform;      // [B] (sampled rows)
  int32_t* out_tokens;       // [B]
  int32_t* token_pool;       // [pool_rows, pool_cols] or nullptr
  int64_t pool_rows;
  int64_t pool_cols;
  const int32_t* wb_rows;    // [B]
  const int64_t* wb_cols;    // [B]
  float* probs_out;          // [B, V] or nullptr
  int32_t* status;           // device status word or nullptr
  int cta_chunk;             // elements of one chunk (one item of the stream kernel)
  int chunks;                // chunks per row
  void* workspace;           // WorkspaceHeader, then [B * chunks] ChunkSlot records
  FillParams fill;           // page allocation + table fill run by extra finish CTAs
  int fill_ctas;             // 0: no fused page fill
};

}  // namespace pkv
