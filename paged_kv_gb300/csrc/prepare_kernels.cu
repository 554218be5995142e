// The step before the model for sm_103a ("mini-sglang from Scratch", page
// "The scheduler skeleton and the offline interface", section "Preparing a
// batch": Scheduler._prepare_batch and Scheduler._forward), in one launch:
//   * allocate_paged: the new pages [ceil(c_i / ps), ceil(d_i / ps)) of every
//     request, from the front of the free list in batch order, written into
//     the page table (as page_fill.cuh);
//   * _make_positions: positions [c_i, d_i) of every request, packed in
//     batch order;
//   * the input tuple (table_idx_i, position): input_ids =
//     token_pool[input tuple] and out_loc = page_table[input tuple], the
//     latter as it stands after this step's allocation.
//
// Every CTA recomputes the per-request page and token counts and their
// exclusive scans (64-bit) in shared memory from the small length arrays, so
// the kernel needs no second launch, grid barrier or scratch.  Then two
// grid-stride loops: (page, 4-entry chunk) items of the fill, and tokens.  A
// token of a new page takes its out_loc from the free list (the value the
// fill writes), one of an earlier page reads the table, which this launch
// does not write there; consecutive threads write consecutive packed
// entries and read consecutive pool and table columns of one request.

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "device_attr.h"
#include "page_fill.cuh"
#include "page_kernels.h"

namespace pkv {

namespace {

constexpr int kPrepThreads = 512;
constexpr int kPrepWarps = kPrepThreads / 32;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStNoSpc = 32;
constexpr int kStTokenCap = 128;
constexpr int kHeadWords = 128;  // warp totals (2 x 16 int64) and the flag word

// Shared memory: head, then poff[B + 1], toff[B + 1] (int64), then first[B],
// frow[B], grow[B], c[B] (int32).
__host__ __device__ constexpr size_t prep_smem_bytes(int B) {
  return static_cast<size_t>(kHeadWords) * 4 + static_cast<size_t>(B + 1) * 16 +
         static_cast<size_t>(B) * 16;
}

__device__ __forceinline__ long long warp_incl_scan64(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Index i of the request holding item x: the last i with off[i] <= x, given
// off[0] = 0 <= x < off[B].
__device__ __forceinline__ int find_request(const long long* off, int B, long long x) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kPrepThreads) prepare_step_kernel(const PrepareParams Q) {
  extern __shared__ __align__(16) int32_t smem[];
  const FillParams& F = Q.fill;
  const int B = F.B;
  const int ps = F.page_size;
  long long* s_wp = reinterpret_cast<long long*>(smem);  // warp page totals
  long long* s_wt = s_wp + kPrepWarps;                    // warp token totals
  int* s_bad = smem + 4 * kPrepWarps;
  long long* s_poff = reinterpret_cast<long long*>(smem + kHeadWords);  // B + 1
  long long* s_toff = s_poff + B + 1;                                    // B + 1
  int32_t* s_first = reinterpret_cast<int32_t*>(s_toff + B + 1);         // B
  int32_t* s_frow = s_first + B;  // table row of the fill, or -1
  int32_t* s_grow = s_frow + B;   // table and pool row of the gathers, or -1
  int32_t* s_c = s_grow + B;      // cached_len
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Per-thread contiguous run of requests, so the scans keep batch order.
  const int per = (B + kPrepThreads - 1) / kPrepThreads;
  const int i0 = min(B, tid * per);
  const int i1 = min(B, i0 + per);
  if (tid == 0) *s_bad = 0;
  long long prun = 0, trun = 0;
  int bad = 0;
  for (int i = i0; i < i1; ++i) {
    const int32_t c = F.cached_len[i], d = F.device_len[i];
    const int64_t first = fill::div_ceil_len(c, ps);
    const int64_t last = fill::div_ceil_len(d, ps);
    const long long n = last > first ? last - first : 0;
    const long long len = d > c ? static_cast<long long>(d) - c : 0;
    const int64_t t = F.table_idx[i];
    int32_t fr = -1, gr = -1;
    if (n > 0) {
      if (t < 0 || t >= F.pt_rows) {
        bad |= kStRowOOB;
      } else if (last * static_cast<int64_t>(ps) > F.pt_cols) {
        bad |= kStColOOB;
      } else {
        fr = static_cast<int32_t>(t);
      }
    }
    if (len > 0) {
      if (t < 0 || t >= F.pt_rows || t >= Q.pool_rows) {
        bad |= kStRowOOB;
      } else if (c < 0 || d > F.pt_cols || d > Q.pool_cols || (n > 0 && fr < 0)) {
        bad |= kStColOOB;
      } else {
        gr = static_cast<int32_t>(t);
      }
    }
    s_first[i] = static_cast<int32_t>(first);
    s_frow[i] = fr;
    s_grow[i] = gr;
    s_c[i] = c;
    s_poff[i] = n;    // counts for now, exclusive offsets after the scans
    s_toff[i] = len;
    prun += n;
    trun += len;
  }
  const long long pincl = warp_incl_scan64(prun, lane);
  const long long tincl = warp_incl_scan64(trun, lane);
  __syncthreads();  // s_bad is zero before any thread ORs into it
  if (bad) atomicOr(s_bad, bad);
  if (lane == 31) {
    s_wp[warp] = pincl;
    s_wt[warp] = tincl;
  }
  __syncthreads();
  long long pbase = 0, tbase = 0, P = 0, N = 0;
#pragma unroll
  for (int w = 0; w < kPrepWarps; ++w) {
    const long long vp = s_wp[w], vt = s_wt[w];
    if (w < warp) {
      pbase += vp;
      tbase += vt;
    }
    P += vp;
    N += vt;
  }
  long long pacc = pbase + pincl - prun, tacc = tbase + tincl - trun;
  for (int i = i0; i < i1; ++i) {
    const long long n = s_poff[i], len = s_toff[i];
    s_poff[i] = pacc;
    s_toff[i] = tacc;
    pacc += n;
    tacc += len;
  }
  if (tid == 0) {
    s_poff[B] = P;
    s_toff[B] = N;
  }
  __syncthreads();

  // Checks before any write: the token capacity, then the free pages.
  const bool over = N > Q.max_tokens;
  const bool nospc = !over && P > F.free_count;
  if (blockIdx.x == 0 && tid == 0) {
    if (Q.tokens_out != nullptr) *Q.tokens_out = N;
    if (F.total_out != nullptr) *F.total_out = (over || nospc) ? 0 : P;
    const int st = over ? kStTokenCap : (nospc ? kStNoSpc : *s_bad);
    if (st != 0 && F.status != nullptr) atomicOr(F.status, st);
  }
  if (over || nospc) return;

  const long long stride = static_cast<long long>(gridDim.x) * kPrepThreads;
  const long long start = static_cast<long long>(blockIdx.x) * kPrepThreads + tid;
  // ---- page fill: items (page, chunk of 4 entries); cpp chunks per page.
  const int cpp = (ps + 3) >> 2;
  const long long items = P * cpp;
  for (long long it = start; it < items; it += stride) {
    const long long p = it / cpp;
    const int q = static_cast<int>(it - p * cpp);
    const int i = find_request(s_poff, B, p);
    const int32_t r = s_frow[i];
    if (r < 0) continue;
    const int64_t col0 = (static_cast<int64_t>(s_first[i]) + (p - s_poff[i])) * ps + 4 * q;
    const int32_t slot = F.free_slots[p] + 4 * q;
    int32_t* dst = F.page_table + static_cast<int64_t>(r) * F.pt_cols + col0;
    if (F.vec4) {
      *reinterpret_cast<int4*>(dst) = make_int4(slot, slot + 1, slot + 2, slot + 3);
    } else {
      const int cnt = min(4, ps - 4 * q);
      for (int o = 0; o < cnt; ++o) dst[o] = slot + o;
    }
  }
  // ---- tokens: position, input id and out_loc of packed entry j.
  for (long long j = start; j < N; j += stride) {
    const int i = find_request(s_toff, B, j);
    const int64_t pos = static_cast<int64_t>(s_c[i]) + (j - s_toff[i]);
    Q.positions[j] = static_cast<int32_t>(pos);
    const int32_t r = s_grow[i];
    int32_t id = -1, loc = -1;
    if (r >= 0) {
      id = Q.token_pool[static_cast<int64_t>(r) * Q.pool_cols + pos];
      const int64_t page = pos / ps;
      const int64_t first = s_first[i];
      if (page >= first) {
        loc = F.free_slots[s_poff[i] + (page - first)] + static_cast<int32_t>(pos - page * ps);
      } else {
        loc = F.page_table[static_cast<int64_t>(r) * F.pt_cols + pos];
      }
    }
    Q.input_ids[j] = id;
    Q.out_loc[j] = loc;
  }
}

}  // namespace

size_t prepare_smem_bytes(int B) { return prep_smem_bytes(B); }

cudaError_t launch_prepare_step(const PrepareParams& Q, int num_sms, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0ull};
  const cudaError_t e = set_smem_limit_once(smem_set, prepare_step_kernel,
                                            static_cast<int>(prep_smem_bytes(kMaxFillBatch)));
  if (e != cudaSuccess) return e;
  const int grid = num_sms > 0 ? num_sms : 1;
  prepare_step_kernel<<<grid, kPrepThreads, prep_smem_bytes(Q.fill.B), stream>>>(Q);
  return cudaGetLastError();
}

}  // namespace pkv
