// Launch-shape choice for the sampler: how many chunks a row is split into
// and how many 16-byte vectors each thread holds per chunk.
#pragma once

#include <cstdint>
#include <initializer_list>

namespace pkv {

constexpr int kSampleThreads = 256;
constexpr int kNvScalar = 16;     // largest vectors-per-thread on the unaligned (element-load) path
constexpr int kMaxRowChunks = 16;  // chunks per row (the finish kernel's capacity)

struct SampleConfig {
  int chunks;  // chunks per row
  int nv;      // 16-byte vectors per thread
  bool vec;    // 16-byte vector loads and bulk copies (aligned rows)
  int chunk;   // elements per chunk = kSampleThreads * nv * elements-per-vector
};

// Chooses (chunks, nv) so that chunks * chunk >= V with the least padded
// capacity (nv 16 only when nothing else fits: it spills and runs one ring
// stage).  Small batches are split into more, smaller chunks while the
// stream kernel would have fewer than two items per SM.  Returns false if V
// does not fit.
inline bool choose_sample_config(int B, int V, bool bf16, bool vec, int num_sms,
                                 SampleConfig* out) {
  const int per_nv = kSampleThreads * (bf16 ? 8 : 4);  // elements per unit of nv
  static const int kNvs[] = {4, 8, 10, 16};
  if (!vec) {
    // Element loads: 10 vectors per thread while that covers V, else 16.
    for (int nv : {10, kNvScalar}) {
      const int64_t cap = static_cast<int64_t>(per_nv) * nv;
      const int64_t c = (V + cap - 1) / cap;
      if (c > kMaxRowChunks) continue;
      out->chunks = static_cast<int>(c);
      out->nv = nv;
      out->vec = false;
      out->chunk = static_cast<int>(cap);
      return true;
    }
    return false;
  }
  int best_c = 0, best_nv = 0;
  int64_t best_cost = INT64_MAX;
  for (int c = 1; c <= kMaxRowChunks; ++c) {
    for (int nv : kNvs) {
      const int64_t cap = static_cast<int64_t>(per_nv) * nv * c;
      if (cap < V) continue;
      int64_t cost = static_cast<int64_t>(c) * nv * 4;
      if (nv > 10) cost += 1000;
      if (cost < best_cost) {
        best_cost = cost;
        best_c = c;
        best_nv = nv;
      }
    }
  }
  if (best_c == 0) return false;
  // Spread small batches over more chunks while each thread keeps >= 4
  // vectors.  Every chunk holds at least one element: chunks = ceil(V / chunk).
  while (static_cast<int64_t>(B) * best_c < 2LL * num_sms && best_c * 2 <= kMaxRowChunks) {
    const int c2 = best_c * 2;
    int nv2 = 0;
    for (int nv : kNvs) {
      if (static_cast<int64_t>(per_nv) * nv * c2 >= V) {
        nv2 = nv;
        break;
      }
    }
    if (nv2 == 0 || nv2 >= best_nv) break;
    const int64_t cap2 = static_cast<int64_t>(per_nv) * nv2;
    const int c_used = static_cast<int>((V + cap2 - 1) / cap2);
    if (c_used <= best_c) break;
    best_c = c_used;
    best_nv = nv2;
  }
  out->chunks = best_c;
  out->nv = best_nv;
  out->vec = true;
  out->chunk = per_nv * best_nv;
  return true;
}

}  // namespace pkv
