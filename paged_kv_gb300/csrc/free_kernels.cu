// Free-path kernels for sm_103a ("mini-sglang from Scratch", page "CacheManager:
// allocation, release and admission control"):
//
// * free_pages_kernel -- section "Freeing, and freeing lazily": the batch's
//   freed slices page_table[t_i, b_i : e_i] each contribute every ps-th entry
//   from their first, appended in batch order after the live free list.  Like
//   the page fill, every CTA recomputes the per-request counts and their
//   exclusive scan in shared memory (B <= kMaxFillBatch), then the grid copies
//   one entry per thread and step: consecutive threads write consecutive free
//   list entries (coalesced) and gather from the table with a stride of ps.
// * check_free_list_kernel -- section "The integrity check": alignment and
//   range of every entry, duplicates through a bitmap of the pool's pages, and
//   the count equation; one OR into the result per CTA.

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "device_attr.h"
#include "page_kernels.h"

namespace pkv {

namespace {

constexpr int kFreeThreads = 512;
constexpr int kCheckThreads = 256;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStNoSpc = 32;

__global__ void __launch_bounds__(kFreeThreads) free_pages_kernel(const FreeParams F) {
  constexpr int kW = kFreeThreads / 32;
  extern __shared__ int32_t smem[];
  __shared__ long long s_warp[kW];
  __shared__ int s_bad;
  const int B = F.B;
  int32_t* s_off = smem;             // B + 1 exclusive offsets (valid when the batch fits)
  int32_t* s_begin = s_off + B + 1;  // first freed column per request
  int32_t* s_row = s_begin + B;      // table row, or -1 for "frees nothing"
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ps = F.page_size;
  // Per-thread contiguous run of requests, so the scan keeps batch order.
  const int per = (B + kFreeThreads - 1) / kFreeThreads;
  const int i0 = min(B, tid * per);
  const int i1 = min(B, i0 + per);
  if (tid == 0) s_bad = 0;
  long long run = 0;
  int bad = 0;
  for (int i = i0; i < i1; ++i) {
    const int32_t b = F.begin[i], e = F.end[i];
    int32_t n = 0, r = -1;
    if (e > b) {
      const int64_t t = F.table_idx[i];
      if (t < 0 || t >= F.pt_rows) {
        bad |= kStRowOOB;
      } else if (b < 0 || e > F.pt_cols) {
        bad |= kStColOOB;
      } else {
        // e - b > 0 fits in 32 bits; ceil by unsigned division.
        const uint32_t len = static_cast<uint32_t>(e) - static_cast<uint32_t>(b);
        n = static_cast<int32_t>((len + static_cast<uint32_t>(ps) - 1u) / static_cast<uint32_t>(ps));
        r = static_cast<int32_t>(t);
      }
    }
    s_begin[i] = b;
    s_row[i] = r;
    s_off[i] = n;  // count for now, exclusive offset after the scan
    run += n;
  }
  long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  long long wbase = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const long long v = s_warp[w];
    if (w < warp) wbase += v;
    total += v;
  }
  const bool nospc = F.free_count + total > F.capacity;
  if (!nospc) {
    long long acc = wbase + incl - run;
    for (int i = i0; i < i1; ++i) {
      const int32_t n = s_off[i];
      s_off[i] = static_cast<int32_t>(acc);
      acc += n;
    }
    if (tid == 0) s_off[B] = static_cast<int32_t>(total);
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0) {
    if (F.total_out != nullptr) *F.total_out = nospc ? 0 : total;
    const int st = (nospc ? kStNoSpc : 0) | s_bad;
    if (st != 0 && F.status != nullptr) atomicOr(F.status, st);
  }
  if (nospc || total == 0) return;

  int32_t* dst = F.free_slots + F.free_count;
  for (int64_t g64 = static_cast<int64_t>(blockIdx.x) * kFreeThreads + tid; g64 < total;
       g64 += static_cast<int64_t>(gridDim.x) * kFreeThreads) {
    const int32_t g = static_cast<int32_t>(g64);  // total <= capacity < 2^31
    // Request whose entries hold g: the last i with off[i] <= g.
    int lo = 0, hi = B;  // invariant: off[lo] <= g < off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= g) lo = mid; else hi = mid;
    }
    const int64_t col = static_cast<int64_t>(s_begin[lo]) + static_cast<int64_t>(g - s_off[lo]) * ps;
    dst[g] = F.page_table[static_cast<int64_t>(s_row[lo]) * F.pt_cols + col];
  }
}

__global__ void __launch_bounds__(kCheckThreads) check_free_list_kernel(
    const int32_t* __restrict__ free_slots, int64_t free_count, int page_size, int64_t num_pages,
    int64_t cache_pages, uint32_t* bitmap, int32_t* result) {
  int bits = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0 && free_count + cache_pages != num_pages) bits |= 1;
  const int64_t limit = num_pages * page_size;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * kCheckThreads + threadIdx.x; g < free_count;
       g += static_cast<int64_t>(gridDim.x) * kCheckThreads) {
    const int32_t slot = free_slots[g];
    if (page_size > 1 && slot % page_size != 0) {
      bits |= 2;
      continue;
    }
    if (slot < 0 || slot >= limit) {
      bits |= 4;
      continue;
    }
    const uint32_t page = static_cast<uint32_t>(slot / page_size);
    const uint32_t bit = 1u << (page & 31u);
    if (atomicOr(&bitmap[page >> 5], bit) & bit) bits |= 8;
  }
  bits = __reduce_or_sync(0xffffffffu, bits);
  __shared__ int s_bits;
  if (threadIdx.x == 0) s_bits = 0;
  __syncthreads();
  if ((threadIdx.x & 31) == 0 && bits != 0) atomicOr(&s_bits, bits);
  __syncthreads();
  if (threadIdx.x == 0 && s_bits != 0) atomicOr(result, s_bits);
}

}  // namespace

size_t free_smem_bytes(int B) { return static_cast<size_t>(3 * B + 1) * sizeof(int32_t); }

cudaError_t launch_free_pages(const FreeParams& F, int num_sms, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0ull};
  const cudaError_t e = set_smem_limit_once(smem_set, free_pages_kernel,
                                            static_cast<int>(free_smem_bytes(kMaxFillBatch)));
  if (e != cudaSuccess) return e;
  // One CTA per SM; each recomputes the (cheap) scan.
  const int grid = num_sms > 0 ? num_sms : 1;
  free_pages_kernel<<<grid, kFreeThreads, free_smem_bytes(F.B), stream>>>(F);
  return cudaGetLastError();
}

cudaError_t launch_check_free_list(const int32_t* free_slots, int64_t free_count, int page_size,
                                   int64_t num_pages, int64_t cache_pages, uint32_t* bitmap,
                                   int32_t* result, int num_sms, cudaStream_t stream) {
  const int64_t want = (free_count + kCheckThreads - 1) / kCheckThreads;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
  check_free_list_kernel<<<grid, kCheckThreads, 0, stream>>>(free_slots, free_count, page_size,
                                                               num_pages, cache_pages, bitmap, result);
  return cudaGetLastError();
}

}  // namespace pkv
