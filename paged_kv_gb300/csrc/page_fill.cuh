// Page allocation and page-table fill for one CTA of a grid ("mini-sglang
// from Scratch", page "CacheManager: allocation, release and admission
// control", sections "The free-page list" and "Allocating pages for this
// step's tokens": allocate_paged, _allocate, _write_page_table with the
// page-to-token expansion):
//   n_i = max(0, ceil(device_len_i / ps) - ceil(cached_len_i / ps)) pages for
//   request i, taken from the front of free_slots in batch order, and
//   page_table[table_idx_i, (first_i + j) * ps + o] = free_slots[off_i + j] + o.
//
// Every CTA recomputes the per-request counts and their exclusive scan in
// shared memory from the small length arrays, so the scan needs no second
// launch, no grid-wide barrier and no scratch; the fill is then a grid-stride
// loop over (page, 4-entry chunk) items with a binary search of the page in
// the scanned offsets and 16-byte stores when the table layout allows.  Used
// by the standalone fill kernel and by the finish kernel's extra CTAs.
#pragma once

#include <cstdint>

#include "page_kernels.h"

namespace pkv {
namespace fill {

constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStNoSpc = 32;

// ceil(a / b) for b >= 1: 32-bit unsigned division for the valid range
// (a >= 0); negative lengths (invalid input) keep the 64-bit arithmetic.
__device__ __forceinline__ int64_t div_ceil_len(int32_t a, int32_t b) {
  if (a >= 0) return static_cast<int64_t>((static_cast<uint32_t>(a) + static_cast<uint32_t>(b) - 1u) /
                                          static_cast<uint32_t>(b));
  return (static_cast<int64_t>(a) + b - 1) / b;
}

// Shared memory of page_fill_cta: 64 words of warp totals and flags, then
// off[B + 1], first[B], row[B].
constexpr int kFillHeadWords = 64;
__host__ __device__ constexpr size_t smem_bytes(int B) {
  return static_cast<size_t>(kFillHeadWords + 3 * B + 1) * sizeof(int32_t);
}

// Run by the kT threads (index tid) of CTA `cta` of `ncta` fill CTAs.
// sync() is the barrier of those kT threads; smem holds smem_bytes(F.B).
template <int kT, class Sync>
__device__ __forceinline__ void page_fill_cta(const FillParams& F, int32_t* smem, int cta,
                                              int ncta, int tid, Sync sync) {
  constexpr int kW = kT / 32;
  static_assert(kW < kFillHeadWords, "warp totals fit the head");
  int32_t* s_warp = smem;
  int* s_bad = smem + kW;
  const int B = F.B;
  int32_t* s_off = smem + kFillHeadWords;  // B + 1 exclusive offsets
  int32_t* s_first = s_off + B + 1;        // first page per request
  int32_t* s_row = s_first + B;            // table row, or -1 for "skip"
  const int lane = tid & 31, warp = tid >> 5;
  const int ps = F.page_size;
  // Per-thread contiguous run of requests, so the scan keeps batch order.
  const int per = (B + kT - 1) / kT;
  const int i0 = min(B, tid * per);
  const int i1 = min(B, i0 + per);
  if (tid == 0) *s_bad = 0;
  int32_t run = 0;
  int bad = 0;
  for (int i = i0; i < i1; ++i) {
    const int64_t first = div_ceil_len(F.cached_len[i], ps);
    const int64_t last = div_ceil_len(F.device_len[i], ps);
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
  // Exclusive scan of the per-thread runs: warp shuffles, then the warp totals.
  int32_t incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  sync();  // s_bad is zero before any thread ORs into it
  if (bad) atomicOr(s_bad, bad);
  if (lane == 31) s_warp[warp] = incl;
  sync();
  int32_t wbase = 0, total32 = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const int32_t v = s_warp[w];
    if (w < warp) wbase += v;
    total32 += v;
  }
  int32_t acc = wbase + incl - run;
  for (int i = i0; i < i1; ++i) {
    const int32_t n = s_off[i];
    s_off[i] = acc;
    acc += n;
  }
  const int64_t total = total32;
  if (tid == 0) s_off[B] = total32;
  sync();

  const bool nospc = total > F.free_count;
  if (cta == 0 && tid == 0) {
    if (F.total_out != nullptr) *F.total_out = nospc ? 0 : total;
    const int st = (nospc ? kStNoSpc : 0) | *s_bad;
    if (st != 0 && F.status != nullptr) atomicOr(F.status, st);
  }
  if (nospc || total == 0) return;

  // Items: (page, chunk of 4 entries).  cpp = chunks per page.
  const int cpp = (ps + 3) >> 2;
  const int64_t items = total * cpp;
  const bool vec4 = F.vec4;
  for (int64_t it = static_cast<int64_t>(cta) * kT + tid; it < items;
       it += static_cast<int64_t>(ncta) * kT) {
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

}  // namespace fill
}  // namespace pkv
