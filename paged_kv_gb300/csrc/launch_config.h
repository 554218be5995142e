// Launch-shape choice for the sampler: how many CTAs form one row's cluster
// and how many 16-byte vectors each thread keeps in registers.
#pragma once

#include <cstdint>

namespace pkv {

constexpr int kSampleThreads = 256;
constexpr int kNvScalar = 16;     // largest vectors-per-thread on the unaligned (element-load) path
constexpr int kMaxCluster = 16;   // 9..16 are non-portable cluster sizes

struct SampleConfig {
  int cluster;  // CTAs per row
  int nv;       // 16-byte vectors per thread
  bool vec;     // 16-byte vector loads (aligned rows)
  int chunk;    // elements per CTA = kSampleThreads * nv * elements-per-vector
};

// Chooses (cluster, nv) so that cluster * chunk >= V with the least padded
// capacity, preferring portable clusters (<= 8) and nv <= 10 (register
// budget for two CTAs per SM).  Small batches are spread over more CTAs so
// that B * cluster covers the SMs.  Returns false if V does not fit.
inline bool choose_sample_config(int B, int V, bool bf16, bool vec, int num_sms,
                                 SampleConfig* out) {
  const int per_nv = kSampleThreads * (bf16 ? 8 : 4);  // elements per unit of nv
  static const int kNvs[] = {4, 8, 10, 16};
  if (!vec) {
    // Element loads: 10 vectors per thread while that covers V, else 16.
    for (int nv : {10, kNvScalar}) {
      const int64_t cap = static_cast<int64_t>(per_nv) * nv;
      const int64_t c = (V + cap - 1) / cap;
      if (c > kMaxCluster) continue;
      out->cluster = static_cast<int>(c);
      out->nv = nv;
      out->vec = false;
      out->chunk = static_cast<int>(cap);
      return true;
    }
    return false;
  }
  int best_c = 0, best_nv = 0;
  int64_t best_cost = INT64_MAX;
  for (int c = 1; c <= kMaxCluster; ++c) {
    for (int nv : kNvs) {
      const int64_t cap = static_cast<int64_t>(per_nv) * nv * c;
      if (cap < V) continue;
      int64_t cost = static_cast<int64_t>(c) * nv * 4;
      if (c > 8) cost += 6;     // non-portable cluster
      if (nv > 10) cost += 24;  // register pressure
      if (cost < best_cost) {
        best_cost = cost;
        best_c = c;
        best_nv = nv;
      }
    }
  }
  if (best_c == 0) return false;
  // Spread small batches over more CTAs while each thread keeps >= 4 vectors.
  while (static_cast<int64_t>(B) * best_c < num_sms && best_c * 2 <= 8) {
    const int c2 = best_c * 2;
    int nv2 = 0;
    for (int nv : kNvs) {
      if (static_cast<int64_t>(per_nv) * nv * c2 >= V) {
        nv2 = nv;
        break;
      }
    }
    if (nv2 == 0 || nv2 >= best_nv) break;
    best_c = c2;
    best_nv = nv2;
  }
  out->cluster = best_c;
  out->nv = best_nv;
  out->vec = true;
  out->chunk = per_nv * best_nv;
  return true;
}

}  // namespace pkv
