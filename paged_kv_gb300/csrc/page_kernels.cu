// Paged-KV bookkeeping and token write-back kernels for sm_103a.
//
// Page fill ("mini-sglang from Scratch", page "CacheManager: allocation,
// release and admission control", sections "The free-page list" and
// "Allocating pages for this step's tokens": allocate_paged, _allocate,
// _write_page_table with the page-to-token expansion):
//   n_i = max(0, ceil(device_len_i / ps) - ceil(cached_len_i / ps)) pages for
//   request i, taken from the front of free_slots in batch order, and
//   page_table[table_idx_i, (first_i + j) * ps + o] = free_slots[off_i + j] + o.
//
// Design: every CTA recomputes the per-request counts and their exclusive
// scan from the (small, L2-resident) length arrays in shared memory, so the
// scan needs no second launch, no grid-wide barrier and no global scratch.
// The fill is then a grid-stride loop over (page, 4-entry chunk) items with a
// binary search of the page in the scanned offsets and 16-byte stores when the
// table layout allows them.
//
// Write-back ("The scheduler skeleton and the offline interface", section
// "Preparing a batch": token_pool[write_tuple] = next_tokens) is a plain
// bounds-checked scatter.

#include <cstdint>
#include <cuda_runtime.h>

#include "page_kernels.h"

namespace pkv {

namespace {

constexpr int kFillThreads = 512;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStNoSpc = 32;

__device__ __forceinline__ int64_t div_ceil64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shared-memory layout (dynamic): off[B + 1], first[B], row[B] as int32.
__global__ void __launch_bounds__(kFillThreads) fill_page_table_kernel(const FillParams F) {
  extern __shared__ int32_t smem[];
  const int B = F.B;
  int32_t* s_off = smem;             // B + 1 exclusive offsets
  int32_t* s_first = s_off + B + 1;  // first page per request
  int32_t* s_row = s_first + B;      // table row, or -1 for "skip"
  __shared__ int32_t s_part[kFillThreads];
  __shared__ int s_bad;

  const int tid = threadIdx.x;
  const int ps = F.page_size;
  // Per-thread contiguous run of requests, so the scan keeps batch order.
  const int per = (B + kFillThreads - 1) / kFillThreads;
  const int i0 = min(B, tid * per);
  const int i1 = min(B, i0 + per);
  if (tid == 0) s_bad = 0;
  int32_t run = 0;
  int bad = 0;
  for (int i = i0; i < i1; ++i) {
    const int64_t first = div_ceil64(F.cached_len[i], ps);
    const int64_t last = div_ceil64(F.device_len[i], ps);
    const int32_t n = last > first ? static_cast<int32_t>(last - first) : 0;
    s_first[i] = static_cast<int32_t>(first);
    s_off[i] = n;  // count for now, exclusive offset after the scan
    int32_t r = -1;
    if (n > 0) {
      const int64_t t = F.table_idx[i];
      if (t < 0 || t >= F.pt_rows) {
        bad |= kStRowOOB;
      } else if (last * static_cast<int64_t>(ps) > F.pt_cols) {
        bad |= kStColOOB;
      } else {
        r = static_cast<int32_t>(t);
      }
    }
    s_row[i] = r;
    run += n;
  }
  s_part[tid] = run;
  __syncthreads();
  // Inclusive scan of the per-thread totals (Hillis-Steele over shared memory).
  for (int o = 1; o < kFillThreads; o <<= 1) {
    const int32_t v = tid >= o ? s_part[tid - o] : 0;
    __syncthreads();
    s_part[tid] += v;
    __syncthreads();
  }
  int32_t acc = tid > 0 ? s_part[tid - 1] : 0;
  for (int i = i0; i < i1; ++i) {
    const int32_t n = s_off[i];
    s_off[i] = acc;
    acc += n;
  }
  if (bad) atomicOr(&s_bad, bad);
  const int64_t total = s_part[kFillThreads - 1];
  if (tid == kFillThreads - 1) s_off[B] = static_cast<int32_t>(total);
  __syncthreads();

  const bool nospc = total > F.free_count;
  if (blockIdx.x == 0 && tid == 0) {
    if (F.total_out != nullptr) *F.total_out = nospc ? 0 : total;
    const int st = (nospc ? kStNoSpc : 0) | s_bad;
    if (st != 0 && F.status != nullptr) atomicOr(F.status, st);
  }
  if (nospc || total == 0) return;

  // Items: (page, chunk of 4 entries).  cpp = chunks per page.
  const int cpp = (ps + 3) >> 2;
  const int64_t items = total * cpp;
  const bool vec4 = F.vec4;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kFillThreads + tid; it < items;
       it += static_cast<int64_t>(gridDim.x) * kFillThreads) {
    const int32_t p = static_cast<int32_t>(it / cpp);
    const int q = static_cast<int>(it - static_cast<int64_t>(p) * cpp);
    // Request whose page range holds p: the last i with off[i] <= p.
    int lo = 0, hi = B;  // invariant: off[lo] <= p < off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= p) lo = mid; else hi = mid;
    }
    const int32_t r = s_row[lo];
    if (r < 0) continue;
    const int64_t col0 = (static_cast<int64_t>(s_first[lo]) + (p - s_off[lo])) * ps + 4 * q;
    const int32_t start = F.free_slots[p] + 4 * q;
    int32_t* dst = F.page_table + static_cast<int64_t>(r) * F.pt_cols + col0;
    if (vec4) {
      *reinterpret_cast<int4*>(dst) = make_int4(start, start + 1, start + 2, start + 3);
    } else {
      const int cnt = min(4, ps - 4 * q);
      for (int o = 0; o < cnt; ++o) dst[o] = start + o;
    }
  }
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

size_t fill_smem_bytes(int B) { return static_cast<size_t>(3 * B + 1) * sizeof(int32_t); }

cudaError_t launch_fill_page_table(const FillParams& F, int num_sms, cudaStream_t stream) {
  const size_t smem = fill_smem_bytes(F.B);
  static bool attr_done = false;
  if (!attr_done) {
    const cudaError_t e = cudaFuncSetAttribute(
        fill_page_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(fill_smem_bytes(kMaxFillBatch)));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
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
