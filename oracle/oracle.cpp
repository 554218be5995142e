// CPU oracle for the decode-step tail: batched per-request sampling, token
// write-back and paged-KV page allocation / page-table fill.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
// definition that the CUDA path is checked against.  Only the tests, the smoke
// check and the benchmark's CPU-baseline leg load it.  It shares no code,
// header, table or helper with the CUDA library, and the CUDA library never
// calls it.
//
// Source of every rule: "mini-sglang from Scratch", pages
//   * "The engine and the sampler" -- sections "The sampler" (Sampler.prepare,
//     Sampler.sample, sample_torch) and "Tests" (test_sampler_greedy_and_filters);
//   * "The scheduler skeleton and the offline interface" -- section "Preparing a
//     batch" (_prepare_batch, _make_write_tuple, Scheduler._forward);
//   * "CacheManager: allocation, release and admission control" -- sections
//     "The free-page list", "Allocating pages for this step's tokens"
//     (allocate_paged, _write_page_table), the self-test answer 4, "Freeing,
//     and freeing lazily" (lazy_free_region) and "The integrity check"
//     (check_integrity).
//
// Arithmetic is fp64 throughout.  Sorting uses std::sort with a total order,
// which is a library primitive used as one step.  Readings of points the pages
// leave open are marked READING below.
//
// Parity pins for every function live in tests/test_oracle_pins.py.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// Row status bits (same meaning as the library's status word; the values are
// restated here on purpose so that the two sides share no header).
constexpr int kNonFinite = 1;   // NaN anywhere in the row, or +inf in a sampled row
constexpr int kAllNegInf = 2;   // sampled row whose logits are all -inf
constexpr int kRowOOB = 4;      // write-back row outside the token pool
constexpr int kColOOB = 8;      // write-back column outside the token pool
constexpr int kBadUniform = 16; // uniform outside [0, 1)

double load_logit(const void* logits, int dtype, int64_t off) {
  if (dtype == 0) {  // fp32
    return static_cast<double>(static_cast<const float*>(logits)[off]);
  }
  // bf16: the upper 16 bits of an IEEE fp32; widening is exact.
  uint16_t h = static_cast<const uint16_t*>(logits)[off];
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return static_cast<double>(f);
}

struct RowResult {
  int32_t token = -1;
  int32_t kept = 0;          // |S|, the size of the kept set
  int32_t status = 0;
  double topp_margin = INFINITY;  // min over K of |before_i / Z_k - p|
  double cdf_margin = INFINITY;   // min over S of |u - c_i|
  double minp_margin = INFINITY;  // min over S (before min_p) of |w_i / min_p - 1|
};

// Greedy decoding: the page's all-greedy path is torch.argmax.  READING: ties
// go to the lowest index; values compare as numbers, so -0 == +0.
RowResult greedy_row(const std::vector<double>& l, double* q_row) {
  RowResult r;
  const int V = static_cast<int>(l.size());
  for (int i = 0; i < V; ++i) {
    if (std::isnan(l[i])) {
      r.status |= kNonFinite;
      return r;
    }
  }
  int best = 0;
  for (int i = 1; i < V; ++i) {
    if (l[i] > l[best]) best = i;  // strict: an equal later value never wins
  }
  r.token = best;
  r.kept = 1;
  if (q_row) q_row[best] = 1.0;
  return r;
}

// One sampled row: sample_torch with torch.multinomial replaced by an inverse
// CDF against the supplied uniform u.
//   1. probabilities ~ exp(l / T)                          (softmax of logits / T)
//   2. order tokens by probability, descending               (probs.sort)
//   3. top-k: drop ranks >= k                                 (masked_fill rank >= top_k)
//   4. top-p on the renormalised top-k distribution: drop a token when the
//      probability mass before it is >= p                    (before = cumsum - p)
//   5. renormalise what is left and draw by inverse CDF in vocab order
//      (the probabilities are scattered back to vocab order before drawing).
// With min_p > 0 (exercise 2 of the same page and its answer), step 4b drops
// from S every token whose probability is below min_p times the largest
// probability: a mask on the full tempered distribution, intersected with
// the top-k / top-p set.
RowResult sampled_row(const std::vector<double>& l, double T, int k, double p,
                      double min_p, double u, double* q_row) {
  RowResult r;
  const int V = static_cast<int>(l.size());
  bool any_finite = false;
  for (int i = 0; i < V; ++i) {
    if (std::isnan(l[i]) || l[i] == INFINITY) {
      r.status |= kNonFinite;  // READING: the pages assume finite logits
      return r;
    }
    if (l[i] != -INFINITY) any_finite = true;
  }
  if (!any_finite) {
    r.status |= kAllNegInf;
    return r;
  }
  if (!(u >= 0.0 && u < 1.0)) {  // READING: flag and clamp to [0, 1 - 2^-24]
    r.status |= kBadUniform;
    u = std::isnan(u) ? 0.0 : std::min(std::max(u, 0.0), 1.0 - std::ldexp(1.0, -24));
  }

  // Step 2.  READING: ties in the sort are broken by ascending index, i.e. the
  // order is (logit descending, index ascending).  Ranking by logit equals
  // ranking by probability because T > 0.
  std::vector<int> order(V);
  for (int i = 0; i < V; ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (l[a] != l[b]) return l[a] > l[b];
    return a < b;
  });

  // Step 1 restricted to the top-k set K (softmax's normaliser cancels once
  // the kept set is renormalised, so unnormalised weights are used).
  const double m = l[order[0]];
  std::vector<double> w(V, 0.0);
  std::vector<char> in_k(V, 0);
  double zk = 0.0;
  for (int j = 0; j < k; ++j) {
    const int i = order[j];
    in_k[i] = 1;
    w[i] = std::exp((l[i] - m) / T);
    zk += w[i];
  }

  // Step 4: walk K in sorted order; keep i iff (mass before i) / Z_k < p.
  std::vector<char> in_s(V, 0);
  if (p < 1.0) {
    double before = 0.0;
    for (int j = 0; j < k; ++j) {
      const int i = order[j];
      const double frac = before / zk;
      r.topp_margin = std::min(r.topp_margin, std::fabs(frac - p));
      if (frac < p) in_s[i] = 1;
      before += w[i];
    }
  } else {
    // READING: p == 1 keeps all of K (exact arithmetic never reaches
    // before >= 1 while tokens remain).
    for (int i = 0; i < V; ++i) in_s[i] = in_k[i];
  }

  // Step 4b: p_i / p_max = exp((l_i - m) / T) = w_i, since m is the row
  // maximum.  READING: the mask is intersected with S as computed above (top-p
  // is not recomputed on the masked distribution).
  if (min_p > 0.0) {
    for (int i = 0; i < V; ++i) {
      if (!in_s[i]) continue;
      r.minp_margin = std::min(r.minp_margin, std::fabs(w[i] / min_p - 1.0));
      if (w[i] < min_p) in_s[i] = 0;
    }
  }

  // Step 5: renormalise over S and scan S in ascending vocab index.
  double zs = 0.0;
  int kept = 0;
  for (int i = 0; i < V; ++i) {
    if (in_s[i]) {
      zs += w[i];
      ++kept;
    }
  }
  r.kept = kept;
  double c = 0.0;
  int chosen = -1;
  int last_positive = -1;
  for (int i = 0; i < V; ++i) {
    if (!in_s[i]) continue;
    const double q = w[i] / zs;
    if (q_row) q_row[i] = q;
    if (q > 0.0) last_positive = i;
    c += q;
    r.cdf_margin = std::min(r.cdf_margin, std::fabs(u - c));
    // READING: right-open intervals, token i is drawn when u < c_i.
    if (chosen < 0 && u < c) chosen = i;
  }
  // READING: when rounding leaves u >= the final sum, the draw falls to the
  // largest index of S that carries probability.
  r.token = chosen >= 0 ? chosen : last_positive;
  return r;
}

void sample_rows(const void* logits, int dtype, int V, int64_t row_stride,
                 const float* temperature, const int32_t* top_k,
                 const float* top_p, const float* min_p, const float* uniform,
                 int row_begin, int row_end, int32_t* tokens, double* probs,
                 double* topp_margin, double* cdf_margin, double* minp_margin,
                 int32_t* kept, int32_t* row_status) {
  std::vector<double> l(V);
  for (int b = row_begin; b < row_end; ++b) {
    for (int i = 0; i < V; ++i) l[i] = load_logit(logits, dtype, b * row_stride + i);
    double* q_row = probs ? probs + static_cast<int64_t>(b) * V : nullptr;
    if (q_row) std::fill(q_row, q_row + V, 0.0);

    // Parameter normalisation, Sampler.prepare.  READING: a row is greedy
    // when no temperature tensor is given (the all-greedy batch) or its
    // temperature is <= 0; a greedy row in a mixed batch returns the exact
    // argmax rather than sampling at T = 1e-6.
    RowResult r;
    const bool greedy = (temperature == nullptr) || !(temperature[b] > 0.0f);
    if (greedy) {
      r = greedy_row(l, q_row);
    } else {
      const double T = std::max(static_cast<double>(temperature[b]), 1e-6);
      int k = V;  // top_k < 1 means "no limit"; k >= V is the same thing
      if (top_k != nullptr && top_k[b] >= 1 && top_k[b] < V) k = top_k[b];
      double p = 1.0;  // top_p clamped into [1e-6, 1]
      if (top_p != nullptr) {
        p = std::min(std::max(static_cast<double>(top_p[b]), 1e-6), 1.0);
      }
      // READING: min_p NULL, <= 0 or NaN is off; above 1 it is 1.
      double mp = 0.0;
      if (min_p != nullptr && min_p[b] > 0.0f) mp = std::min(static_cast<double>(min_p[b]), 1.0);
      const double u = static_cast<double>(uniform[b]);
      r = sampled_row(l, T, k, p, mp, u, q_row);
    }
    tokens[b] = r.token;
    if (topp_margin) topp_margin[b] = r.topp_margin;
    if (cdf_margin) cdf_margin[b] = r.cdf_margin;
    if (minp_margin) minp_margin[b] = r.minp_margin;
    if (kept) kept[b] = r.kept;
    if (row_status) row_status[b] = r.status;
  }
}

int64_t div_ceil(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

// Sample one token per row.  logits: [B, V] with the given row stride (in
// elements); dtype 0 = fp32, 1 = bf16 (raw bits).  temperature == NULL means
// an all-greedy batch; top_k / top_p == NULL mean "off" for every row;
// uniform is required unless all rows are greedy.  Outputs per row: token,
// optional dense probabilities q [B, V] (fp64), the top-p and CDF margins,
// |S| and the row status bits.  n_threads > 1 splits rows over std::threads.
// Returns the OR of all row status bits.
int oracle_sample_ex(const void* logits, int dtype, int B, int V, int64_t row_stride,
                     const float* temperature, const int32_t* top_k,
                     const float* top_p, const float* min_p, const float* uniform,
                     int32_t* tokens, double* probs, double* topp_margin, double* cdf_margin,
                     double* minp_margin, int32_t* kept, int32_t* row_status, int n_threads) {
  std::vector<int32_t> local_status;
  if (row_status == nullptr) {
    local_status.assign(B, 0);
    row_status = local_status.data();
  }
  if (n_threads <= 1 || B <= 1) {
    sample_rows(logits, dtype, V, row_stride, temperature, top_k, top_p, min_p, uniform,
                0, B, tokens, probs, topp_margin, cdf_margin, minp_margin, kept, row_status);
  } else {
    const int nt = std::min(n_threads, B);
    std::vector<std::thread> pool;
    for (int t = 0; t < nt; ++t) {
      const int b0 = static_cast<int>(static_cast<int64_t>(B) * t / nt);
      const int b1 = static_cast<int>(static_cast<int64_t>(B) * (t + 1) / nt);
      pool.emplace_back(sample_rows, logits, dtype, V, row_stride, temperature,
                        top_k, top_p, min_p, uniform, b0, b1, tokens, probs,
                        topp_margin, cdf_margin, minp_margin, kept, row_status);
    }
    for (auto& th : pool) th.join();
  }
  int all = 0;
  for (int b = 0; b < B; ++b) all |= row_status[b];
  return all;
}

// oracle_sample_ex with min_p off for every row.
int oracle_sample(const void* logits, int dtype, int B, int V, int64_t row_stride,
                  const float* temperature, const int32_t* top_k,
                  const float* top_p, const float* uniform, int32_t* tokens,
                  double* probs, double* topp_margin, double* cdf_margin,
                  int32_t* kept, int32_t* row_status, int n_threads) {
  return oracle_sample_ex(logits, dtype, B, V, row_stride, temperature, top_k, top_p, nullptr,
                          uniform, tokens, probs, topp_margin, cdf_margin, nullptr, kept,
                          row_status, n_threads);
}

// Token write-back, Scheduler._forward: token_pool[rows[b], cols[b]] = tok[b].
// READING: a column < 0 means "do not write" (the write tuple's -1), and a
// negative token (a row that produced no token) is not written either.
// Out-of-range rows / columns are flagged and skipped.  Returns status bits.
int oracle_writeback(const int32_t* tokens, const int32_t* rows,
                     const int64_t* cols, int B, int32_t* pool,
                     int64_t pool_rows, int64_t pool_cols) {
  int status = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t col = cols[b];
    if (col < 0 || tokens[b] < 0) continue;
    const int64_t row = rows[b];
    if (row < 0 || row >= pool_rows) {
      status |= kRowOOB;
      continue;
    }
    if (col >= pool_cols) {
      status |= kColOOB;
      continue;
    }
    pool[row * pool_cols + col] = tokens[b];
  }
  return status;
}

// Page counts and offsets, allocate_paged: for request i the pages
// [ceil(cached/ps), ceil(device/ps)) are new; they are taken from the front
// of the free list in batch order.  Returns 0, or -2 (no space) when the total
// exceeds free_count (the pages' eviction fallback is out of scope).
int oracle_alloc_pages(const int32_t* cached_len, const int32_t* device_len,
                       int B, int page_size, int64_t free_count,
                       int32_t* first_page, int32_t* num_pages, int64_t* offset,
                       int64_t* total) {
  int64_t needed = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t first = div_ceil(cached_len[i], page_size);
    const int64_t last = div_ceil(device_len[i], page_size);
    const int64_t n = last > first ? last - first : 0;
    first_page[i] = static_cast<int32_t>(first);
    num_pages[i] = static_cast<int32_t>(n);
    offset[i] = needed;
    needed += n;
  }
  *total = needed;
  return needed > free_count ? -2 : 0;
}

// Page-table fill, _write_page_table with the page-to-token expansion: every
// newly allocated page of request i covers the whole page, so for j < n_i and
// o < ps, page_table[table_idx[i], (first_i + j) * ps + o] =
// free_slots[offset_i + j] + o.  Nothing is written when the allocation does
// not fit (-2) or when any target lies outside the table (-1, status bits).
int oracle_fill_page_table(const int32_t* cached_len, const int32_t* device_len,
                           const int32_t* table_idx, int B, int page_size,
                           const int32_t* free_slots, int64_t free_count,
                           int32_t* page_table, int64_t pt_rows,
                           int64_t pt_cols, int64_t* total, int32_t* status) {
  std::vector<int32_t> first(B), num(B);
  std::vector<int64_t> off(B);
  int rc = oracle_alloc_pages(cached_len, device_len, B, page_size, free_count,
                              first.data(), num.data(), off.data(), total);
  *status = 0;
  if (rc != 0) {
    *status = 32;
    return rc;
  }
  for (int i = 0; i < B; ++i) {
    if (num[i] == 0) continue;
    const int64_t t = table_idx[i];
    if (t < 0 || t >= pt_rows) {
      *status |= kRowOOB;
      continue;
    }
    if ((static_cast<int64_t>(first[i]) + num[i]) * page_size > pt_cols) {
      *status |= kColOOB;
      continue;
    }
    for (int64_t j = 0; j < num[i]; ++j) {
      const int32_t start = free_slots[off[i] + j];
      for (int o = 0; o < page_size; ++o) {
        page_table[t * pt_cols + (first[i] + j) * page_size + o] = start + o;
      }
    }
  }
  return 0;
}

// Batched lazy free, lazy_free_region: inside the region every freed index
// tensor contributes indices[::ps] -- its first element and every ps-th one
// after it -- and on exit the contributions are concatenated onto the end of
// the free list in the order they were freed.  The freed indices of request
// i are the slice page_table[table_idx[i], begin[i] : end[i]] of its table
// row (cache_req frees slices of page_table[table_idx, :cached_len]).
// READING: requests are freed in batch order; an empty or reversed range
// (end <= begin) frees nothing; a range whose row lies outside the table or
// whose bounds lie outside [0, pt_cols] is flagged (status 4 or 8) and frees
// nothing; when the free list's capacity cannot take the whole batch, nothing
// is appended (status 32, return -2).  *total = the number of entries
// appended.  free_slots holds free_count entries and room for capacity.
int oracle_free_pages(const int32_t* table_idx, const int32_t* begin, const int32_t* end,
                      int B, int page_size, const int32_t* page_table, int64_t pt_rows,
                      int64_t pt_cols, int32_t* free_slots, int64_t free_count,
                      int64_t capacity, int64_t* total, int32_t* status) {
  *status = 0;
  *total = 0;
  std::vector<int32_t> appended;
  for (int i = 0; i < B; ++i) {
    const int64_t b = begin[i], e = end[i];
    if (e <= b) continue;
    const int64_t t = table_idx[i];
    if (t < 0 || t >= pt_rows) {
      *status |= kRowOOB;
      continue;
    }
    if (b < 0 || e > pt_cols) {
      *status |= kColOOB;
      continue;
    }
    for (int64_t col = b; col < e; col += page_size) {
      appended.push_back(page_table[t * pt_cols + col]);
    }
  }
  if (free_count + static_cast<int64_t>(appended.size()) > capacity) {
    *status |= 32;
    return -2;
  }
  for (size_t g = 0; g < appended.size(); ++g) free_slots[free_count + g] = appended[g];
  *total = static_cast<int64_t>(appended.size());
  return 0;
}

// The integrity check, check_integrity: the free pages and the pages the
// prefix cache holds add up to the pool (bit 1 when they do not), and with
// ps > 1 every free entry is a page start, a multiple of ps (bit 2).
// READING, two more bits for what the pages say the check is for ("anything
// forgotten, or freed twice"): an entry that is not the start of a pool page
// [0, num_pages * ps) (bit 4), and a page listed more than once (bit 8).
int oracle_check_free_list(const int32_t* free_slots, int64_t free_count, int page_size,
                           int64_t num_pages, int64_t cache_pages) {
  int bits = 0;
  if (free_count + cache_pages != num_pages) bits |= 1;
  std::vector<char> seen(static_cast<size_t>(num_pages > 0 ? num_pages : 0), 0);
  for (int64_t g = 0; g < free_count; ++g) {
    const int64_t slot = free_slots[g];
    if (page_size > 1 && slot % page_size != 0) {
      bits |= 2;
      continue;
    }
    if (slot < 0 || slot >= num_pages * page_size) {
      bits |= 4;
      continue;
    }
    const int64_t page = slot / page_size;
    if (seen[page]) bits |= 8;
    seen[page] = 1;
  }
  return bits;
}

// Counter-based uniforms for the draw.  The pages seed one generator per
// engine (torch.manual_seed(42) in Engine) and rely on every rank making the
// same random calls in the same order ("The scheduler's IO and multi-rank
// synchronization", section "Sending results"); a counter-based generator
// gives each (call, row) its own number with no state to keep in step.
// Philox-4x64 with 10 rounds, from its published definition (Salmon, Moraes,
// Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
// each round multiplies words 0 and 2 by two odd constants, takes the high
// and low halves, and mixes them with words 1 and 3 and the round key; the
// key is bumped by two Weyl increments (the golden ratio and sqrt(3) - 1,
// scaled to 64 bits) between rounds.
void oracle_philox4x64(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  const uint64_t m0 = 0xD2E7470EE14C6C93ull, m1 = 0xCA5A826395121157ull;
  const uint64_t w0 = 0x9E3779B97F4A7C15ull, w1 = 0xBB67AE8584CAA73Bull;
  uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    const unsigned __int128 p0 = static_cast<unsigned __int128>(m0) * x0;
    const unsigned __int128 p1 = static_cast<unsigned __int128>(m1) * x2;
    const uint64_t hi0 = static_cast<uint64_t>(p0 >> 64), lo0 = static_cast<uint64_t>(p0);
    const uint64_t hi1 = static_cast<uint64_t>(p1 >> 64), lo1 = static_cast<uint64_t>(p1);
    const uint64_t y0 = hi1 ^ x1 ^ k0, y1 = lo1, y2 = hi0 ^ x3 ^ k1, y3 = lo0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
    k0 += w0;
    k1 += w1;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

// The uniform of row b in call `offset` under `seed`: the first word of the
// Philox block at counter (b, offset, 0, 0) with key (seed, 0), its top 24
// bits scaled by 2^-24 (exact in fp32, in [0, 1)).  READING: the pages fix
// only the seed; the counter layout and the 24-bit conversion are this
// library's choices.
void oracle_uniforms(uint64_t seed, uint64_t offset, int B, float* u) {
  const uint64_t key[2] = {seed, 0};
  for (int b = 0; b < B; ++b) {
    const uint64_t ctr[4] = {static_cast<uint64_t>(b), offset, 0, 0};
    uint64_t out[4];
    oracle_philox4x64(ctr, key, out);
    u[b] = static_cast<float>(static_cast<double>(out[0] >> 40) * (1.0 / 16777216.0));
  }
}

// The step before the model, Scheduler._prepare_batch and Scheduler._forward
// ("The scheduler skeleton and the offline interface", section "Preparing a
// batch"), in their order:
//   1. allocate_paged: the new pages of every request are taken from the
//      free list and written into the page table (oracle_fill_page_table);
//   2. _make_positions: the positions [cached_len, device_len) of every
//      request, packed into one array in batch order;
//   3. the input tuple (table_idx, position) of each packed token gathers
//      input_ids = token_pool[input tuple] and out_loc = page_table[input
//      tuple], the latter after step 1.
// READINGS: a request with device_len <= cached_len has no tokens.  The token
// count is checked before anything is written: above max_tokens, status bit
// 128, return -3, nothing written.  When the pages do not fit (status 32,
// return -2) nothing is written either and *total_pages is 0.  A request
// whose gathers would leave the token pool or the page table (a table row
// outside either, cached_len < 0, device_len past either's columns, or new
// pages that the fill skipped) still gets its positions, its input_ids and
// out_loc entries are -1, and status bit 4 (row) or 8 (column) is set.
// *total_tokens is always the step's token count.
int oracle_prepare_step(const int32_t* cached_len, const int32_t* device_len,
                        const int32_t* table_idx, int B, int page_size,
                        const int32_t* free_slots, int64_t free_count, int32_t* page_table,
                        int64_t pt_rows, int64_t pt_cols, const int32_t* token_pool,
                        int64_t pool_rows, int64_t pool_cols, int32_t* positions,
                        int32_t* input_ids, int32_t* out_loc, int64_t max_tokens,
                        int64_t* total_pages, int64_t* total_tokens, int32_t* status) {
  *status = 0;
  *total_pages = 0;
  int64_t ntok = 0;
  for (int i = 0; i < B; ++i) {
    if (device_len[i] > cached_len[i]) ntok += static_cast<int64_t>(device_len[i]) - cached_len[i];
  }
  *total_tokens = ntok;
  if (ntok > max_tokens) {
    *status = 128;
    return -3;
  }
  // 1. pages.
  int32_t fill_status = 0;
  int64_t pages = 0;
  const int rc = oracle_fill_page_table(cached_len, device_len, table_idx, B, page_size,
                                        free_slots, free_count, page_table, pt_rows, pt_cols,
                                        &pages, &fill_status);
  *status |= fill_status;
  if (rc != 0) return rc;
  *total_pages = pages;
  // 2. and 3. positions and the two gathers, request by request.
  int64_t j = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t c = cached_len[i], d = device_len[i];
    if (d <= c) continue;
    const int64_t first = div_ceil(c, page_size), last = div_ceil(d, page_size);
    const int64_t t = table_idx[i];
    bool ok = true;
    if (t < 0 || t >= pt_rows || t >= pool_rows) {
      *status |= kRowOOB;
      ok = false;
    } else if (c < 0 || d > pt_cols || d > pool_cols ||
               (last > first && last * page_size > pt_cols)) {
      *status |= kColOOB;
      ok = false;
    }
    for (int64_t pos = c; pos < d; ++pos, ++j) {
      positions[j] = static_cast<int32_t>(pos);
      input_ids[j] = ok ? token_pool[t * pool_cols + pos] : -1;
      out_loc[j] = ok ? page_table[t * pt_cols + pos] : -1;
    }
  }
  return 0;
}

}  // extern "C"
