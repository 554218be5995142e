// Batched per-request sampler for sm_103a.
//
// Operation ("mini-sglang from Scratch", page "The engine and the sampler",
// section "The sampler": Sampler.sample / sample_torch): greedy rows return
// the argmax (lowest index on ties); other rows are scaled by 1/T, filtered
// top-k first and then top-p on the renormalised top-k distribution (keep a
// token while the mass ranked before it is < p), renormalised, and a token is
// drawn by inverse CDF in ascending vocab index against the supplied uniform.
// Order between equal logits is by ascending index everywhere.
//
// GB300 design:
//   * One thread-block cluster of C CTAs per row (grid = C x B, not
//     persistent, so rows never wait for each other).  CTA r owns the
//     contiguous slice [r*chunk, (r+1)*chunk) of the row.  Its first thread
//     issues one TMA bulk copy (cp.async.bulk + mbarrier) of the slice into
//     shared memory, so a CTA holds no registers while its bytes are in flight
//     and several CTAs per SM keep HBM busy.  Every logit is read from HBM
//     exactly once; all later passes read shared memory.
//   * Cross-CTA steps are cluster barriers.  Scalars are PUSHED into every
//     CTA's shared memory before a barrier (DSMEM stores), so each CTA reads
//     only its own shared memory afterwards and can exit right after its last
//     barrier.
//   * Fast selection (no per-element atomics): a guaranteed lower bound theta of
//     the final threshold comes from the warps' per-thread maxima -- by count
//     for top-k (each warp has >= k_w elements >= its k_w-th largest thread
//     maximum), by probability mass for top-p (the warp's thread maxima that
//     carry >= p of the warp's mass).  The few elements >= theta are compacted,
//     in index order, into a list in the leader CTA's shared memory; the
//     leader finishes top-k, top-p and the inverse CDF exactly on that list
//     (radix selects with 256-bucket histograms over the list only).
//   * Fallback (lists that would overflow, dense top-p rows): the same
//     selections as radix selects over the whole row held on chip, with
//     cluster-wide histogram exchanges.  Masses are 2^-40 fixed-point
//     integers accumulated with pairs of 32-bit atomics, so every sum is exact
//     and independent of atomic order (deterministic).
//   * The draw: per-warp partial sums -> per-CTA sums exchanged across the
//     cluster -> the CTA, warp, 256-element slab, lane and element where the
//     cumulative mass first exceeds u * Z_S (or a block scan over the list).
//   * No tensor cores (nothing here is a contraction); exp is MUFU.EX2.
#pragma once

#include <climits>
#include <cstdint>

#include "device_common.cuh"
#include "sample_params.h"

namespace pkv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 256;
constexpr int kMaxClusterCtas = 16;
constexpr float kMassScale = 1099511627776.0f;  // 2^40: fixed-point unit of probability mass

constexpr int kStNonFinite = 1;
constexpr int kStAllNegInf = 2;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStBadUniform = 16;

// One CTA's values for one exchange phase, pushed into every CTA.
struct Slot {
  float f0;
  float f1;
  int32_t i0;
  uint32_t u0;
  unsigned long long l0;
  uint32_t pad0;
  uint32_t pad1;
};
static_assert(sizeof(Slot) == 32, "Slot is pushed as two 16-byte stores");

// Histogram a CTA publishes for the others to read (fallback radix select).
struct PullBuf {
  uint32_t lo[kBuckets];  // counts, or low words of fixed-point masses
  uint32_t hi[kBuckets];  // high words of fixed-point masses
};

struct SampleSmem {
  Slot push[2][kMaxClusterCtas];
  Slot gather[kMaxClusterCtas];  // collected by the leader only
  uint32_t cnt[kMaxClusterCtas];
  PullBuf pull[2];
  unsigned long long scan[kBuckets];
  uint32_t hlo[kBuckets];  // CTA-local histogram (list selects)
  uint32_t hhi[kBuckets];
  unsigned long long wl[kWarps];
  float wf[kWarps];
  uint32_t wu[kWarps];
  int32_t wi[kWarps];
  float wt[kWarps];
  float wz[kWarps];
  float bf[4];
  int32_t bi[4];
  uint32_t bu[4];
  unsigned long long bl[4];
};

// ----------------------------------------------------------------- element access
//
// The slice is an array of 16-byte vectors.  Thread (warp w, lane l) owns the
// vectors (w*NV + j)*32 + l, j < NV, so every warp owns a contiguous
// sub-slice.  Element c of the thread's vector j has row index
// lane_base + j*32*VW + c.

template <bool BF16>
struct Layout {
  static constexpr int VW = BF16 ? 8 : 4;   // elements per 16-byte vector
  static constexpr int EPW = BF16 ? 2 : 1;  // elements per 32-bit word
  static constexpr int ELT = BF16 ? 2 : 4;  // bytes per element
};

template <bool BF16>
__device__ __forceinline__ float elem(uint32_t word, int h) {
  if constexpr (BF16) {
    return __uint_as_float(h == 0 ? (word << 16) : (word & 0xffff0000u));
  } else {
    return __uint_as_float(word);
  }
}

// f(x, e) for the elements of one 16-byte vector whose first index is e0.
template <bool BF16, typename F>
__device__ __forceinline__ void for_vector(const uint4& v, int e0, F&& f) {
  using L = Layout<BF16>;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int h = 0; h < L::EPW; ++h) f(elem<BF16>(w[c], h), e0 + c * L::EPW + h);
  }
}

// NaN-propagating maximum of one 16-byte vector.
template <bool BF16>
__device__ __forceinline__ float vector_max(const uint4& v) {
  if constexpr (BF16) {
    const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
    return fmax_nan(elem<true>(m2, 0), elem<true>(m2, 1));
  } else {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

struct Ctx {
  int tid, lane, warp;
  uint32_t crank, csize;
  int row, V;
  int lane_base;  // row index of the thread's first element
  const uint4* sv;
};

// f(x, e) for every element the thread owns, in ascending index order.
template <bool BF16, int NV, typename F>
__device__ __forceinline__ void for_each(const Ctx& c, F&& f) {
  using L = Layout<BF16>;
#pragma unroll 2
  for (int j = 0; j < NV; ++j) {
    const uint4 v = c.sv[(c.warp * NV + j) * 32 + c.lane];
    for_vector<BF16>(v, c.lane_base + j * 32 * L::VW, f);
  }
}

// ----------------------------------------------------------------- block helpers

template <typename T>
__device__ __forceinline__ T block_suffix_scan(T v, T* s_w, int lane, int warp) {
  v = warp_suffix_scan(v, lane);
  if (lane == 0) s_w[warp] = v;
  __syncthreads();
  T add = 0;
  for (int w = warp + 1; w < kWarps; ++w) add += s_w[w];
  __syncthreads();
  return v + add;
}

// Exclusive prefix over threads in tid order; *total receives the block sum.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* s_w, int lane, int warp, T* total) {
  const T incl = warp_inclusive_scan(v, lane);
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  T before = 0, all = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += s_w[w];
    all += s_w[w];
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

__device__ __forceinline__ int block_max_int(int v, int32_t* s_w, int lane, int warp) {
  v = __reduce_max_sync(kFull, v);
  if (lane == 0) s_w[warp] = v;
  __syncthreads();
  int r = s_w[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = max(r, s_w[w]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ int block_min_int(int v, int32_t* s_w, int lane, int warp) {
  v = __reduce_min_sync(kFull, v);
  if (lane == 0) s_w[warp] = v;
  __syncthreads();
  int r = s_w[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = min(r, s_w[w]);
  __syncthreads();
  return r;
}

// Radix-select step: thread t holds the weight `tot` of bucket t (t < 256).
// Returns the highest bucket b whose suffix weight S(b) = sum_{t >= b} tot_t
// reaches `rem`, and S(b + 1) (the weight strictly above it) in *above.
__device__ __forceinline__ int select_bucket(unsigned long long tot, unsigned long long rem,
                                             SampleSmem& sm, unsigned long long* above,
                                             int tid, int lane, int warp) {
  const unsigned long long S = block_suffix_scan<unsigned long long>(tot, sm.wl, lane, warp);
  sm.scan[tid] = S;
  int b = block_max_int(S >= rem ? tid : -1, sm.wi, lane, warp);
  if (b < 0) b = 0;  // unreachable: callers keep rem <= S(0)
  *above = (b + 1 < kBuckets) ? sm.scan[b + 1] : 0ull;
  __syncthreads();
  return b;
}

// Adds a 64-bit fixed-point value to a (lo, hi) pair of 32-bit counters.
__device__ __forceinline__ void atomic_add_u64_split(uint32_t* lo, uint32_t* hi,
                                                     unsigned long long v) {
  const uint32_t vlo = static_cast<uint32_t>(v);
  const uint32_t vhi = static_cast<uint32_t>(v >> 32);
  const uint32_t old = atomicAdd(lo, vlo);
  const uint32_t carry = (old + vlo < old) ? 1u : 0u;
  if (vhi + carry != 0u) atomicAdd(hi, vhi + carry);
}

__device__ __forceinline__ unsigned long long mass_fx(float w) {
  return static_cast<unsigned long long>(__float2ull_rz(w * kMassScale));
}

// ----------------------------------------------------------------- exchange

// Pushes this CTA's slot into slot[crank] of every CTA, then waits at the
// cluster barrier.  Returns the buffer to read locally.
__device__ __forceinline__ const Slot* push_exchange(SampleSmem& sm, int& ph, const Ctx& c,
                                                     const Slot& mine) {
  Slot* buf = sm.push[ph & 1];
  if (c.tid < static_cast<int>(c.csize)) {
    const uint32_t a = dsmem(&buf[c.crank], static_cast<uint32_t>(c.tid));
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&mine);
    st_dsmem_v4(a, w[0], w[1], w[2], w[3]);
    st_dsmem_v4(a + 16, w[4], w[5], w[6], w[7]);
  }
  cluster_sync();
  ++ph;
  return buf;
}

// ----------------------------------------------------------------- output

__device__ __forceinline__ void emit_token(const SampleParams& P, int row, int tok, int st) {
  P.out_tokens[row] = tok;
  if (P.token_pool != nullptr && tok >= 0) {
    const int64_t col = P.wb_cols[row];
    if (col >= 0) {
      const int64_t r = P.wb_rows[row];
      if (r < 0 || r >= P.pool_rows) {
        st |= kStRowOOB;
      } else if (col >= P.pool_cols) {
        st |= kStColOOB;
      } else {
        P.token_pool[r * P.pool_cols + col] = tok;
      }
    }
  }
  if (st != 0 && P.status != nullptr) atomicOr(P.status, st);
}

// ----------------------------------------------------------------- warp helpers

// 32 floats sorted descending across the warp (bitonic network).
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(kFull, v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_max ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

// ----------------------------------------------------------------- list selects
//
// The leader's list holds n entries (value, row index) in ascending index
// order.  These run in one CTA with __syncthreads only.

// Smallest and largest key of the list entries satisfying `keep`.
template <typename K>
__device__ __forceinline__ void list_key_range(const float* val, int n, K&& keep, SampleSmem& sm,
                                               const Ctx& c, uint32_t* kmin, uint32_t* kmax) {
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = c.tid; i < n; i += kThreads) {
    if (keep(i)) {
      const uint32_t k = float_key(val[i]);
      lo = min(lo, k);
      hi = max(hi, k);
    }
  }
  lo = __reduce_min_sync(kFull, lo);
  hi = __reduce_max_sync(kFull, hi);
  if (c.lane == 0) {
    sm.wu[c.warp] = lo;
    sm.wi[c.warp] = static_cast<int32_t>(hi);
  }
  __syncthreads();
  uint32_t a = 0xffffffffu, b = 0u;
  for (int w = 0; w < kWarps; ++w) {
    a = min(a, sm.wu[w]);
    b = max(b, static_cast<uint32_t>(sm.wi[w]));
  }
  __syncthreads();
  *kmin = a;
  *kmax = b;
}

// Radix select over the list: the key t such that the weight of entries with
// key > t is < target <= the weight with key >= t.  weight(i) is 1 (count) or
// a fixed-point mass; entries with keep(i) false weigh nothing.  Returns t and
// the weight still needed from the entries equal to t in *rem.
template <bool MASS, typename K, typename W>
__device__ __forceinline__ float list_select(const float* val, int n, K&& keep, W&& weight,
                                             unsigned long long target, SampleSmem& sm,
                                             const Ctx& c, unsigned long long* rem_out) {
  uint32_t kmin, kmax;
  list_key_range(val, n, keep, sm, c, &kmin, &kmax);
  unsigned long long rem = target;
  if (kmin == kmax) {
    *rem_out = rem;
    return key_float(kmin);
  }
  const int top = 31 - __clz(kmin ^ kmax);
  uint32_t prefix = static_cast<uint32_t>(
      static_cast<unsigned long long>(kmin) & ~((2ull << top) - 1ull));
  for (int hi = top; hi >= 0; hi -= 8) {
    const int lo = hi >= 7 ? hi - 7 : 0;
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    const uint32_t amask =
        static_cast<uint32_t>(~((2ull << hi) - 1ull));  // bits above the digit
    sm.hlo[c.tid] = 0u;
    sm.hhi[c.tid] = 0u;
    __syncthreads();
    for (int i = c.tid; i < n; i += kThreads) {
      if (!keep(i)) continue;
      const uint32_t key = float_key(val[i]);
      if ((key & amask) != (prefix & amask)) continue;
      const uint32_t d = (key >> lo) & dmask;
      if constexpr (MASS) {
        atomic_add_u64_split(&sm.hlo[d], &sm.hhi[d], weight(i));
      } else {
        atomicAdd(&sm.hlo[d], 1u);
      }
    }
    __syncthreads();
    const unsigned long long tot =
        MASS ? ((static_cast<unsigned long long>(sm.hhi[c.tid]) << 32) | sm.hlo[c.tid])
             : static_cast<unsigned long long>(sm.hlo[c.tid]);
    unsigned long long above;
    const int b = select_bucket(tot, rem, sm, &above, c.tid, c.lane, c.warp);
    rem -= above;
    prefix |= static_cast<uint32_t>(b) << lo;
  }
  *rem_out = rem;
  return key_float(prefix);
}

// Position cut for ties in the list: among entries with member(i), the first
// r (list order = index order) are kept.  Returns the position after the r-th
// member (n if there are fewer than r).
template <typename M>
__device__ __forceinline__ int list_tie_cut(int n, M&& member, unsigned long long r,
                                            SampleSmem& sm, const Ctx& c) {
  const int per = (n + kThreads - 1) / kThreads;
  const int i0 = min(n, c.tid * per);
  const int i1 = min(n, i0 + per);
  uint32_t cnt = 0;
  for (int i = i0; i < i1; ++i) cnt += member(i) ? 1u : 0u;
  uint32_t total;
  const uint32_t before = block_exclusive_scan<uint32_t>(cnt, sm.wu, c.lane, c.warp, &total);
  if (c.tid == 0) sm.bi[3] = n;
  __syncthreads();
  if (r <= total && before < r && r <= before + cnt) {
    uint32_t need = static_cast<uint32_t>(r - before);
    for (int i = i0; i < i1; ++i) {
      if (member(i) && --need == 0) {
        sm.bi[3] = i + 1;
        break;
      }
    }
  }
  __syncthreads();
  const int cut = sm.bi[3];
  __syncthreads();
  return cut;
}

// Inverse CDF over the list entries with in_s(i): the first entry (list
// order) whose cumulative weight exceeds u * Z_S; else the last with weight.
// Writes Z_S to *zs.  Returns the row index of the token (-1 if none).
template <typename S, typename W>
__device__ __forceinline__ int list_draw(const int32_t* idx, int n, S&& in_s, W&& w_of, float u,
                                         SampleSmem& sm, const Ctx& c, float* zs) {
  const int per = (n + kThreads - 1) / kThreads;
  const int i0 = min(n, c.tid * per);
  const int i1 = min(n, i0 + per);
  float seg = 0.0f;
  int last = -1;
  for (int i = i0; i < i1; ++i) {
    if (in_s(i)) {
      const float w = w_of(i);
      seg += w;
      if (w > 0.0f) last = i;
    }
  }
  float total;
  const float before = block_exclusive_scan<float>(seg, sm.wt, c.lane, c.warp, &total);
  const float target = u * total;
  const int cand = block_min_int((target < before + seg && seg > 0.0f) ? c.tid : INT_MAX, sm.wi,
                                 c.lane, c.warp);
  const int lastpos = block_max_int(last, sm.wi, c.lane, c.warp);
  if (c.tid == 0) sm.bi[2] = lastpos;
  __syncthreads();
  if (cand != INT_MAX && c.tid == cand) {
    float run = before;
    int sel = -1;
    for (int i = i0; i < i1; ++i) {
      if (in_s(i)) {
        run += w_of(i);
        if (target < run) {
          sel = i;
          break;
        }
      }
    }
    sm.bi[2] = sel >= 0 ? sel : last;
  }
  __syncthreads();
  const int pos = sm.bi[2];
  *zs = total;
  __syncthreads();
  return pos >= 0 ? idx[pos] : -1;
}

// ----------------------------------------------------------------- the kernel

// ----------------------------------------------------------------- leader finish

// The leader CTA holds every candidate of the row in its list, region r
// (entries r*R .. r*R + cnt[r]) coming from CTA r, each region in index
// order.  Packs the regions, then finishes exactly on the list: top-k (count
// select, ties by index), top-p inside K (mass select on 2^-40 fixed-point
// weights; target_fx is given for rows without top-k), renormalisation and
// the inverse-CDF draw.  Emits the token and, if asked, the probabilities.
__device__ __forceinline__ void leader_finish(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                              float* l_val, int32_t* l_idx, int R, int row,
                                              bool topk_row, int k, bool use_p, float p,
                                              unsigned long long target_fx, float m, float c2,
                                              float u, int st, float* q_row) {
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  int n = 0;
  for (uint32_t r = 0; r < c.csize; ++r) n += static_cast<int>(sm.cnt[r]);
  {
    // Packed index i comes from region r at offset i - (earlier counts),
    // never from a position below i: read, barrier, write.
    constexpr int kMovePer = 16;
    float mv[kMovePer];
    int mi[kMovePer];
    for (int b0 = 0; b0 < n; b0 += kThreads * kMovePer) {
#pragma unroll
      for (int q = 0; q < kMovePer; ++q) {
        const int i = b0 + q * kThreads + tid;
        if (i < n) {
          int r = 0, off = i;
          while (off >= static_cast<int>(sm.cnt[r])) {
            off -= static_cast<int>(sm.cnt[r]);
            ++r;
          }
          mv[q] = l_val[r * R + off];
          mi[q] = l_idx[r * R + off];
        }
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < kMovePer; ++q) {
        const int i = b0 + q * kThreads + tid;
        if (i < n) {
          l_val[i] = mv[q];
          l_idx[i] = mi[q];
        }
      }
      __syncthreads();
    }
  }
  int cut_k = n;
  float tk = -INFINITY;
  if (topk_row) {
    unsigned long long rk;
    tk = list_select<false>(l_val, n, [](int) { return true; }, [](int) { return 1ull; },
                            static_cast<unsigned long long>(k), sm, c, &rk);
    const float tkv = tk;
    cut_k = list_tie_cut(n, [&](int i) { return l_val[i] == tkv; }, rk, sm, c);
  }
  const float tkv = tk;
  const int ckv = cut_k;
  auto in_k = [&](int i) { return l_val[i] > tkv || (l_val[i] == tkv && i < ckv); };
  auto w_of = [&](int i) { return ex2((l_val[i] - m) * c2); };
  float tp = tk;
  int cut_p = cut_k;
  if (use_p) {
    if (topk_row) {
      unsigned long long zfx = 0;
      for (int i = tid; i < n; i += kThreads) {
        if (in_k(i)) zfx += mass_fx(w_of(i));
      }
      zfx = warp_sum(zfx);
      if (lane == 0) sm.wl[warp] = zfx;
      __syncthreads();
      unsigned long long z = 0;
      for (int w = 0; w < kWarps; ++w) z += sm.wl[w];
      __syncthreads();
      const double t = static_cast<double>(z) * static_cast<double>(p);
      target_fx = static_cast<unsigned long long>(ceil(t));
      if (target_fx < 1) target_fx = 1;
      if (target_fx > z) target_fx = z;
    }
    unsigned long long rem;
    tp = list_select<true>(l_val, n, in_k, [&](int i) { return mass_fx(w_of(i)); }, target_fx, sm,
                           c, &rem);
    // Members of the threshold group share one weight wt: member j (index
    // order) is kept iff above + j * wt < target, i.e. j < ceil(rem / wt).
    const unsigned long long wt = mass_fx(ex2((tp - m) * c2));
    const unsigned long long rp = wt == 0 ? ~0ull : (rem + wt - 1) / wt;
    const float tpv = tp;
    cut_p = list_tie_cut(n, [&](int i) { return l_val[i] == tpv && in_k(i); }, rp, sm, c);
  }
  const float tpv = tp;
  const int cpv = cut_p;
  auto in_s = [&](int i) { return in_k(i) && (l_val[i] > tpv || (l_val[i] == tpv && i < cpv)); };
  float zs;
  const int tok = list_draw(l_idx, n, in_s, w_of, u, sm, c, &zs);
  if (tid == 0) emit_token(P, row, tok, tok < 0 ? (st | kStNonFinite) : st);
  if (q_row != nullptr) {
    const float inv = 1.0f / zs;
    for (int i = tid; i < n; i += kThreads) {
      if (in_s(i)) q_row[l_idx[i]] = w_of(i) * inv;
    }
  }
}

// ----------------------------------------------------------------- CTA-local selects

// Among this CTA's elements with member(x, e), the first r in index order:
// returns the element-index cutoff (members with e < cutoff), INT_MAX if there
// are no more than r members.  CTA barriers only.
template <bool BF16, int NV, typename M>
__device__ __forceinline__ int cta_tie_cut(const Ctx& c, SampleSmem& sm, M&& member,
                                           unsigned long long r) {
  using L = Layout<BF16>;
  const int lane = c.lane, warp = c.warp;
  uint32_t cnt = 0;
  for_each<BF16, NV>(c, [&](float x, int e) { cnt += member(x, e) ? 1u : 0u; });
  const uint32_t wc = __reduce_add_sync(kFull, cnt);
  if (lane == 0) sm.wu[warp] = wc;
  __syncthreads();
  unsigned long long cum = 0;
  int wstar = -1;
  uint32_t rw = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (wstar < 0 && cum + sm.wu[w] >= r) {
      wstar = w;
      rw = static_cast<uint32_t>(r - cum);
    }
    cum += sm.wu[w];
  }
  if (r == 0) wstar = -2;
  if (c.tid == 0) sm.bi[1] = wstar == -2 ? INT_MIN : INT_MAX;
  __syncthreads();
  if (warp == wstar) {
    uint32_t acc = 0;
    int found = INT_MAX;
    for (int j = 0; j < NV; ++j) {
      const uint4 v = c.sv[(warp * NV + j) * 32 + lane];
      const int e0 = c.lane_base + j * 32 * L::VW;
      uint32_t cj = 0;
      for_vector<BF16>(v, e0, [&](float x, int e) { cj += member(x, e) ? 1u : 0u; });
      const uint32_t incl = warp_inclusive_scan(cj, lane);
      const uint32_t stot = __shfl_sync(kFull, incl, 31);
      if (acc + stot >= rw) {
        const unsigned bal = __ballot_sync(kFull, acc + incl >= rw);
        const int lx = __ffs(bal) - 1;
        int sel = INT_MAX;
        if (lane == lx) {
          uint32_t need = rw - (acc + incl - cj);
          for_vector<BF16>(v, e0, [&](float x, int e) {
            if (member(x, e)) {
              if (need == 1 && sel == INT_MAX) sel = e;
              --need;
            }
          });
        }
        found = __shfl_sync(kFull, sel, lx);
        break;
      }
      acc += stot;
    }
    if (lane == 0) sm.bi[1] = found == INT_MAX ? INT_MAX : found + 1;
  }
  __syncthreads();
  const int cut = sm.bi[1];
  __syncthreads();
  return cut;
}

// Exact top-k of this CTA's elements with keep(x, e), by (value desc, index
// asc): returns t and *cut such that the top-k are {keep, x > t} and
// {keep, x == t, e < cut}.  Radix select over keys with 32-bit shared atomics.
template <bool BF16, int NV, typename K>
__device__ __forceinline__ float cta_select_topk(const Ctx& c, SampleSmem& sm, K&& keep,
                                                 unsigned long long k, int* cut) {
  uint32_t lo = 0xffffffffu, hi = 0u;
  for_each<BF16, NV>(c, [&](float x, int e) {
    if (keep(x, e)) {
      const uint32_t key = float_key(x);
      lo = min(lo, key);
      hi = max(hi, key);
    }
  });
  lo = __reduce_min_sync(kFull, lo);
  hi = __reduce_max_sync(kFull, hi);
  if (c.lane == 0) {
    sm.wu[c.warp] = lo;
    sm.wi[c.warp] = static_cast<int32_t>(hi);
  }
  __syncthreads();
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int w = 0; w < kWarps; ++w) {
    kmin = min(kmin, sm.wu[w]);
    kmax = max(kmax, static_cast<uint32_t>(sm.wi[w]));
  }
  __syncthreads();
  unsigned long long rem = k;
  uint32_t prefix = kmin;
  if (kmin != kmax) {
    const int top = 31 - __clz(kmin ^ kmax);
    prefix = static_cast<uint32_t>(static_cast<unsigned long long>(kmin) & ~((2ull << top) - 1ull));
    for (int hb = top; hb >= 0; hb -= 8) {
      const int lb = hb >= 7 ? hb - 7 : 0;
      const uint32_t dmask = (1u << (hb - lb + 1)) - 1u;
      const uint32_t amask = static_cast<uint32_t>(~((2ull << hb) - 1ull));
      sm.hlo[c.tid] = 0u;
      __syncthreads();
      for_each<BF16, NV>(c, [&](float x, int e) {
        if (!keep(x, e)) return;
        const uint32_t key = float_key(x);
        if ((key & amask) == (prefix & amask)) atomicAdd(&sm.hlo[(key >> lb) & dmask], 1u);
      });
      __syncthreads();
      unsigned long long above;
      const int b = select_bucket(sm.hlo[c.tid], rem, sm, &above, c.tid, c.lane, c.warp);
      rem -= above;
      prefix |= static_cast<uint32_t>(b) << lb;
    }
  }
  const float t = key_float(prefix);
  *cut = cta_tie_cut<BF16, NV>(c, sm, [&](float x, int e) { return keep(x, e) && x == t; }, rem);
  return t;
}

// ----------------------------------------------------------------- the kernel

template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void load_slice(const SampleParams& P, int row, int lane_base,
                                           uint32_t (&d)[NV][4]) {
  using L = Layout<BF16>;
  const char* rp = static_cast<const char*>(P.logits) +
                   static_cast<size_t>(row) * static_cast<size_t>(P.row_stride) * L::ELT;
  const int V = P.V;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e0 = lane_base + j * 32 * L::VW;
    if (VEC && e0 + L::VW <= V) {
      const uint4 v = ld_stream_v4(rp + static_cast<size_t>(e0) * L::ELT);
      d[j][0] = v.x;
      d[j][1] = v.y;
      d[j][2] = v.z;
      d[j][3] = v.w;
    } else {
      // Row tail or unaligned row: element loads, -inf past the end.
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (BF16) {
          const int e = e0 + 2 * q;
          const uint32_t lo = e < V ? reinterpret_cast<const uint16_t*>(rp)[e] : 0xff80u;
          const uint32_t hi = e + 1 < V ? reinterpret_cast<const uint16_t*>(rp)[e + 1] : 0xff80u;
          d[j][q] = lo | (hi << 16);
        } else {
          const int e = e0 + q;
          d[j][q] = e < V ? reinterpret_cast<const uint32_t*>(rp)[e] : 0xff800000u;
        }
      }
    }
  }
}

// One cluster of C CTAs per row (grid C x B).  CTA r holds elements
// [r*chunk, (r+1)*chunk) of its row: 16-byte loads into registers, copied
// to shared memory when later passes need them.  Cross-CTA traffic is pushed
// into the receiving CTA's shared memory.  The leader (rank 0) is the only
// CTA that waits when it merely collects: the others arrive at the cluster
// barrier and exit.
template <bool BF16, int NV, bool VEC, bool ALL_GREEDY>
__global__ void __launch_bounds__(kThreads, 3) sample_kernel(const SampleParams P) {
  using L = Layout<BF16>;
  constexpr int CHUNK = kThreads * NV * L::VW;  // elements per CTA
  constexpr int NLEV = BF16 ? 2 : 4;            // 8-bit radix levels (fallback)
  constexpr int kWarpSpan = 32 * NV * L::VW;    // elements per warp
  __shared__ SampleSmem sm;
  extern __shared__ __align__(128) unsigned char dyn[];
  uint4* s_vec = reinterpret_cast<uint4*>(dyn);
  float* l_val = reinterpret_cast<float*>(dyn + CHUNK * L::ELT);
  int32_t* l_idx = reinterpret_cast<int32_t*>(l_val + P.list_cap);

  // Every CTA of the cluster must have started before anyone stores into its
  // shared memory: arrive now, wait just before the first remote store.
  cluster_arrive();

  Ctx c;
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  c.crank = cluster_rank();
  c.csize = cluster_size();
  c.row = blockIdx.y;
  c.V = P.V;
  c.sv = s_vec;
  const int V = P.V;
  const int row = c.row;
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int cta_begin = static_cast<int>(c.crank) * CHUNK;
  c.lane_base = cta_begin + ((warp * NV) * 32 + lane) * L::VW;
  const bool has_pad = cta_begin + CHUNK > V;  // this slice reaches past the row end
  constexpr uint32_t leader = 0;
  const int R = P.list_cap / static_cast<int>(c.csize);  // list entries per CTA region

  // Row parameters (Sampler.prepare's normalisation).
  const bool greedy = ALL_GREEDY || !(P.temperature[row] > 0.0f);
  float T = 1.0f, p = 1.0f, u = 0.0f;
  int k = V;
  int st = 0;
  if (!greedy) {
    T = fmaxf(P.temperature[row], 1e-6f);
    k = P.top_k != nullptr ? P.top_k[row] : -1;
    if (k < 1 || k >= V) k = V;
    p = P.top_p != nullptr ? fminf(fmaxf(P.top_p[row], 1e-6f), 1.0f) : 1.0f;
    u = P.uniform[row];
    if (!(u >= 0.0f && u < 1.0f)) {
      st |= kStBadUniform;
      u = (u != u) ? 0.0f : fminf(fmaxf(u, 0.0f), 0x1.fffffep-1f);
    }
  }
  const float c2 = 1.4426950408889634f / T;  // log2(e) / T
  float* q_row = P.probs_out != nullptr ? P.probs_out + static_cast<size_t>(row) * V : nullptr;

  // ---- load the slice and take thread maxima (NaN-propagating).
  uint32_t d[NV][4];
  load_slice<BF16, NV, VEC>(P, row, c.lane_base, d);
  float tmax = -INFINITY;
  int tidx = INT_MAX;
  bool nan = false;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const uint4 v = make_uint4(d[j][0], d[j][1], d[j][2], d[j][3]);
    const float vm = vector_max<BF16>(v);
    if (vm != vm) {
      nan = true;
    } else if (vm > tmax || tidx == INT_MAX) {
      tmax = vm;
      if (greedy) {
        int first = INT_MAX;
        for_vector<BF16>(v, c.lane_base + j * 32 * L::VW, [&](float x, int e) {
          if (x == vm && e < first) first = e;
        });
        tidx = first;
      } else {
        tidx = 0;
      }
    }
  }
  if (q_row != nullptr) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const uint4 v = make_uint4(d[j][0], d[j][1], d[j][2], d[j][3]);
      for_vector<BF16>(v, c.lane_base + j * 32 * L::VW, [&](float, int e) {
        if (e < V) q_row[e] = 0.0f;
      });
    }
  }

  if (greedy) {
    // ---- greedy rows: (max, first index) to the leader, which alone waits.
    const int nan_any = __any_sync(kFull, nan);
    float v = tmax;
    int i = tidx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, v, o);
      const int oi = __shfl_xor_sync(kFull, i, o);
      if (ov > v || (ov == v && oi < i)) {
        v = ov;
        i = oi;
      }
    }
    if (lane == 0) {
      sm.wf[warp] = v;
      sm.wi[warp] = i;
      sm.wu[warp] = static_cast<uint32_t>(nan_any);
    }
    __syncthreads();
    cluster_wait();
    if (tid == 0) {
      float bv = sm.wf[0];
      int bi = sm.wi[0];
      uint32_t bn = sm.wu[0];
      for (int w = 1; w < kWarps; ++w) {
        if (sm.wf[w] > bv || (sm.wf[w] == bv && sm.wi[w] < bi)) {
          bv = sm.wf[w];
          bi = sm.wi[w];
        }
        bn |= sm.wu[w];
      }
      const uint32_t a = dsmem(&sm.gather[c.crank], leader);
      st_dsmem_v4(a, __float_as_uint(bv), 0u, static_cast<uint32_t>(bi), bn);
    }
    __syncthreads();
    cluster_arrive();
    if (c.crank != leader) return;
    cluster_wait();
    if (tid == 0) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      uint32_t bn = 0;
      for (uint32_t r = 0; r < c.csize; ++r) {
        const float gv = sm.gather[r].f0;
        const int gi = sm.gather[r].i0;
        if (gv > bv || (gv == bv && gi < bi)) {
          bv = gv;
          bi = gi;
        }
        bn |= sm.gather[r].u0;
      }
      const int tok = bn ? -1 : bi;
      emit_token(P, row, tok, (bn ? kStNonFinite : 0) | st);
      if (q_row != nullptr && tok >= 0) q_row[tok] = 1.0f;
    }
    return;
  }

  if constexpr (!ALL_GREEDY) {
    // ---- sampled rows: later passes read the slice from shared memory.
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      s_vec[(warp * NV + j) * 32 + lane] = make_uint4(d[j][0], d[j][1], d[j][2], d[j][3]);
    }
    const bool use_p = p < 1.0f;
    const int nan_any = __any_sync(kFull, nan);

    // Chunk-local top-k: if this chunk has >= k elements >= theta_c, every
    // element of the row's top-k that lies in this chunk is >= theta_c (k
    // elements > the row's k-th value cannot exist), so each CTA can pick its
    // candidates with no information from the others.  theta_c is the min over
    // the chunk's full warps of their kw-th largest thread maximum,
    // kw = ceil(k / full warps).  Uniform eligibility: k <= 256, k <= R, and
    // the last CTA (fewest full warps) still has kw <= 32.
    const int nfull_cta = max(0, min(kWarps, (V - cta_begin) / kWarpSpan));
    const int nfull_min =
        max(0, min(kWarps, (V - static_cast<int>(c.csize - 1) * CHUNK) / kWarpSpan));
    const bool local_topk = k < V && k <= 256 && k <= R && nfull_min >= 1 &&
                            (k + nfull_min - 1) / nfull_min <= 32;
    if (local_topk) {
      const int kw = (k + nfull_cta - 1) / nfull_cta;
      const bool full = cta_begin + (warp + 1) * kWarpSpan <= V;
      const float sorted = warp_sort_desc(tmax, lane);
      const float tw = full ? __shfl_sync(kFull, sorted, kw - 1) : INFINITY;
      float wmax = tmax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wmax = fmax_nan(wmax, __shfl_xor_sync(kFull, wmax, o));
      if (lane == 0) {
        sm.wt[warp] = tw;
        sm.wf[warp] = wmax;
        sm.wu[warp] = static_cast<uint32_t>(nan_any);
      }
      __syncthreads();
      float theta = INFINITY, cmax = -INFINITY;
      uint32_t cnan = 0;
      for (int w = 0; w < kWarps; ++w) {
        theta = fminf(theta, sm.wt[w]);
        cmax = fmax_nan(cmax, sm.wf[w]);
        cnan |= sm.wu[w];
      }
      __syncthreads();
      auto cand = [&](float x, int e) { return x >= theta && (!has_pad || e < V); };
      uint32_t cnt = 0;
      for_each<BF16, NV>(c, [&](float x, int e) { cnt += cand(x, e) ? 1u : 0u; });
      const uint32_t wc = __reduce_add_sync(kFull, cnt);
      if (lane == 0) sm.wu[warp] = wc;
      __syncthreads();
      uint32_t ncta = 0;
      for (int w = 0; w < kWarps; ++w) ncta += sm.wu[w];
      __syncthreads();
      // Ties can push the count past the region: keep exactly the chunk's top-k.
      float tloc = -INFINITY;
      int cloc = INT_MAX;
      if (static_cast<int>(ncta) > R) {
        tloc = cta_select_topk<BF16, NV>(c, sm, cand, static_cast<unsigned long long>(k), &cloc);
      }
      const float tlv = tloc;
      const int clv = cloc;
      auto keep = [&](float x, int e) {
        return cand(x, e) && (x > tlv || (x == tlv && e < clv));
      };
      cnt = 0;
      for_each<BF16, NV>(c, [&](float x, int e) { cnt += keep(x, e) ? 1u : 0u; });
      const uint32_t wk = __reduce_add_sync(kFull, cnt);
      if (lane == 0) sm.wu[warp] = wk;
      __syncthreads();
      uint32_t woff = 0, nkeep = 0;
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) woff += sm.wu[w];
        nkeep += sm.wu[w];
      }
      cluster_wait();
      {
        const uint32_t base = static_cast<uint32_t>(c.crank) * R + woff;
        const uint32_t a_val = dsmem(l_val, leader);
        const uint32_t a_idx = dsmem(l_idx, leader);
        uint32_t acc = 0;
        for (int j = 0; j < NV; ++j) {
          const uint4 v = s_vec[(warp * NV + j) * 32 + lane];
          const int e0 = c.lane_base + j * 32 * L::VW;
          uint32_t cj = 0;
          for_vector<BF16>(v, e0, [&](float x, int e) { cj += keep(x, e) ? 1u : 0u; });
          if (__ballot_sync(kFull, cj != 0) == 0) continue;
          const uint32_t incl = warp_inclusive_scan(cj, lane);
          uint32_t pos = base + acc + incl - cj;
          for_vector<BF16>(v, e0, [&](float x, int e) {
            if (keep(x, e)) {
              st_dsmem_f32(a_val + 4u * pos, x);
              st_dsmem_u32(a_idx + 4u * pos, static_cast<uint32_t>(e));
              ++pos;
            }
          });
          acc += __shfl_sync(kFull, incl, 31);
        }
      }
      if (tid == 0) {
        const uint32_t a = dsmem(&sm.gather[c.crank], leader);
        st_dsmem_v4(a, __float_as_uint(cmax), 0u, 0u, cnan);
        st_dsmem_u32(dsmem(&sm.cnt[c.crank], leader), nkeep);
      }
      __syncthreads();
      cluster_arrive();
      if (c.crank != leader) return;
      cluster_wait();
      float m = -INFINITY;
      uint32_t rn = 0;
      for (uint32_t r = 0; r < c.csize; ++r) {
        m = fmax_nan(m, sm.gather[r].f0);
        rn |= sm.gather[r].u0;
      }
      if (rn != 0 || m != m || m == INFINITY || m == -INFINITY) {
        const int est = (m == -INFINITY && rn == 0) ? kStAllNegInf : kStNonFinite;
        if (tid == 0) emit_token(P, row, -1, est | st);
        return;
      }
      leader_finish(P, sm, c, l_val, l_idx, R, row, true, k, use_p, p, 0ull, m, c2, u, st,
                    q_row);
      return;
    }

    // ---- other sampled rows: one all-to-all exchange of the chunk maximum,
    // the chunk mass (relative to the chunk maximum) and a bound theta_c.
    const bool topk_row = k < V;
    const bool need_z = !topk_row;
    float zt = 0.0f;
    if (need_z && tmax > -INFINITY) {
      for_each<BF16, NV>(c, [&](float x, int) { zt += ex2((x - tmax) * c2); });
    }
    float wmax = tmax;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wmax = fmax_nan(wmax, __shfl_xor_sync(kFull, wmax, o));
    const float zw = warp_sum(tmax > -INFINITY ? zt * ex2((tmax - wmax) * c2) : 0.0f);
    float tw = -INFINITY;
    if (topk_row) {
      // kw-th largest thread maximum of every warp fully inside the row.
      const int w_full = V / kWarpSpan;
      const int kw = w_full > 0 ? (k + w_full - 1) / w_full : INT_MAX;
      const bool full = cta_begin + (warp + 1) * kWarpSpan <= V;
      if (kw <= 32) {
        const float sorted = warp_sort_desc(tmax, lane);
        tw = full ? __shfl_sync(kFull, sorted, kw - 1) : INFINITY;
      }
    } else if (use_p) {
      // Largest theta_w whose thread maxima above it carry >= p' of the
      // warp's mass (p' = p raised by 1e-3, so that rounding rarely forces
      // the fallback; the decision below is exact).  A warp without mass
      // does not constrain theta.
      const float sorted = warp_sort_desc(tmax, lane);
      const float ws = sorted > -INFINITY ? ex2((sorted - wmax) * c2) : 0.0f;
      const float cum = warp_inclusive_scan(ws, lane);
      const float need = fminf(1.0f, p * 1.001f) * zw;
      const unsigned hit = __ballot_sync(kFull, cum >= need);
      tw = zw > 0.0f ? (hit ? __shfl_sync(kFull, sorted, __ffs(hit) - 1) : -INFINITY) : INFINITY;
    }
    if (lane == 0) {
      sm.wt[warp] = tw;
      sm.wf[warp] = wmax;
      sm.wz[warp] = zw;
      sm.wu[warp] = static_cast<uint32_t>(nan_any);
    }
    __syncthreads();
    Slot mine = {};
    {
      float cm = -INFINITY, th = INFINITY, cz = 0.0f;
      uint32_t cn = 0;
      for (int w = 0; w < kWarps; ++w) {
        cm = fmax_nan(cm, sm.wf[w]);
        th = fminf(th, sm.wt[w]);
        cn |= sm.wu[w];
      }
      if (cm > -INFINITY) {
        for (int w = 0; w < kWarps; ++w) {
          if (sm.wf[w] > -INFINITY) cz += sm.wz[w] * ex2((sm.wf[w] - cm) * c2);
        }
      }
      mine.f0 = cm;
      mine.f1 = th;
      mine.u0 = cn;
      mine.pad0 = __float_as_uint(cz);
    }
    __syncthreads();
    cluster_wait();
    int ph = 0;
    float m, theta, zrow, before_cta;
    bool nan_row;
    {
      const Slot* s = push_exchange(sm, ph, c, mine);
      float mm = -INFINITY, th = INFINITY;
      uint32_t nn = 0;
      for (uint32_t r = 0; r < c.csize; ++r) {
        mm = fmax_nan(mm, s[r].f0);
        th = fminf(th, s[r].f1);
        nn |= s[r].u0;
      }
      float zz = 0.0f;
      if (mm > -INFINITY && mm == mm) {
        for (uint32_t r = 0; r < c.csize; ++r) {
          if (s[r].f0 > -INFINITY) zz += __uint_as_float(s[r].pad0) * ex2((s[r].f0 - mm) * c2);
        }
      }
      m = mm;
      theta = th;
      zrow = zz;
      nan_row = nn != 0;
      // CTA prefix of the masses, for the plain rows' draw (same summation
      // order as zrow, so the CTA intervals tile [0, zrow) exactly).
      float before = 0.0f;
      for (uint32_t r = 0; r < c.crank; ++r) {
        if (s[r].f0 > -INFINITY) before += __uint_as_float(s[r].pad0) * ex2((s[r].f0 - mm) * c2);
      }
      before_cta = before;
    }
    if (nan_row || m != m || m == INFINITY || m == -INFINITY) {
      const int est = (m == -INFINITY && !nan_row) ? kStAllNegInf : kStNonFinite;
      if (c.crank == leader && tid == 0) emit_token(P, row, -1, est | st);
      return;
    }

    if (!topk_row && !use_p) {
      // ---- plain rows: draw over the whole row; the CTA holding the
      // crossing finds the token.
      // Keep the target strictly below zrow so that it falls in the interval
      // of a CTA that holds mass.
      float target = u * zrow;
      if (!(target < zrow)) target = nextafterf(zrow, 0.0f);
      const float before = before_cta;
      const float mine_z =
          mine.f0 > -INFINITY ? __uint_as_float(mine.pad0) * ex2((mine.f0 - m) * c2) : 0.0f;
      if (target >= before && target < before + mine_z) {
        // Warp holding the crossing (sequential over warps).
        const float tloc = target - before;
        int wstar = -1;
        float tw2 = INFINITY, cw = 0.0f;
        int wlast = -1;
        for (int w = 0; w < kWarps; ++w) {
          const float ww = sm.wf[w] > -INFINITY ? sm.wz[w] * ex2((sm.wf[w] - m) * c2) : 0.0f;
          if (wstar < 0 && tloc < cw + ww) {
            wstar = w;
            tw2 = tloc - cw;
          }
          if (ww > 0.0f) wlast = w;
          cw += ww;
        }
        if (wstar < 0) {
          wstar = wlast < 0 ? 0 : wlast;
          tw2 = INFINITY;
        }
        if (warp == wstar) {
          float acc = 0.0f;
          int found = -1, lastpos = -1;
          for (int j = 0; j < NV; ++j) {
            const uint4 v = s_vec[(warp * NV + j) * 32 + lane];
            const int e0 = c.lane_base + j * 32 * L::VW;
            float lj = 0.0f;
            int llast = -1;
            for_vector<BF16>(v, e0, [&](float x, int e) {
              const float w = ex2((x - m) * c2);
              lj += w;
              if (w > 0.0f) llast = e;
            });
            const unsigned has = __ballot_sync(kFull, llast >= 0);
            if (has != 0) lastpos = __shfl_sync(kFull, llast, 31 - __clz(has));
            const float incl = warp_inclusive_scan(lj, lane);
            const float stot = __shfl_sync(kFull, incl, 31);
            if (tw2 < acc + stot) {
              const unsigned bal = __ballot_sync(kFull, tw2 < acc + incl);
              const int lx = bal ? __ffs(bal) - 1 : 31;
              int sel = -1;
              if (lane == lx) {
                float run = acc + (incl - lj);
                for_vector<BF16>(v, e0, [&](float x, int e) {
                  run += ex2((x - m) * c2);
                  if (sel < 0 && tw2 < run) sel = e;
                });
                if (sel < 0) sel = llast;
              }
              found = __shfl_sync(kFull, sel, lx);
              if (found < 0) found = lastpos;
              break;
            }
            acc += stot;
          }
          if (found < 0) found = lastpos;
          if (lane == 0 && found >= 0) emit_token(P, row, found, st);
        }
      }
      if (q_row != nullptr) {
        const float inv = 1.0f / zrow;
        for_each<BF16, NV>(c, [&](float x, int e) {
          if (e < V) q_row[e] = ex2((x - m) * c2) * inv;
        });
      }
      return;
    }

    // ---- global theta: candidates >= theta into the leader's list.
    const bool fast = theta > -INFINITY;
    if (fast) {
      auto cand = [&](float x, int e) { return x >= theta && (!has_pad || e < V); };
      uint32_t cnt = 0;
      unsigned long long mfx = 0;
      for_each<BF16, NV>(c, [&](float x, int e) {
        if (cand(x, e)) {
          ++cnt;
          if (!topk_row) mfx += mass_fx(ex2((x - m) * c2));
        }
      });
      const uint32_t wc = __reduce_add_sync(kFull, cnt);
      mfx = warp_sum(mfx);
      if (lane == 0) {
        sm.wu[warp] = wc;
        sm.wl[warp] = mfx;
      }
      __syncthreads();
      uint32_t woff = 0, ncta = 0;
      unsigned long long mcta = 0;
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) woff += sm.wu[w];
        ncta += sm.wu[w];
        mcta += sm.wl[w];
      }
      if (static_cast<int>(ncta) <= R) {
        const uint32_t base = static_cast<uint32_t>(c.crank) * R + woff;
        const uint32_t a_val = dsmem(l_val, leader);
        const uint32_t a_idx = dsmem(l_idx, leader);
        uint32_t acc = 0;
        for (int j = 0; j < NV; ++j) {
          const uint4 v = s_vec[(warp * NV + j) * 32 + lane];
          const int e0 = c.lane_base + j * 32 * L::VW;
          uint32_t cj = 0;
          for_vector<BF16>(v, e0, [&](float x, int e) { cj += cand(x, e) ? 1u : 0u; });
          if (__ballot_sync(kFull, cj != 0) == 0) continue;
          const uint32_t incl = warp_inclusive_scan(cj, lane);
          uint32_t pos = base + acc + incl - cj;
          for_vector<BF16>(v, e0, [&](float x, int e) {
            if (cand(x, e)) {
              st_dsmem_f32(a_val + 4u * pos, x);
              st_dsmem_u32(a_idx + 4u * pos, static_cast<uint32_t>(e));
              ++pos;
            }
          });
          acc += __shfl_sync(kFull, incl, 31);
        }
      }
      Slot cs = {};
      cs.u0 = ncta;
      cs.l0 = mcta;
      __syncthreads();
      const Slot* s = push_exchange(sm, ph, c, cs);
      // Uniform decision: every region fits, and (top-p rows) the list holds
      // enough mass that no element below theta can be kept.
      uint32_t over = 0;
      unsigned long long lmass = 0;
      for (uint32_t r = 0; r < c.csize; ++r) {
        if (static_cast<int>(s[r].u0) > R) over = 1;
        lmass += s[r].l0;
      }
      unsigned long long target_fx = 0;
      if (!topk_row) {
        const double t = static_cast<double>(p) * static_cast<double>(zrow) * 1099511627776.0;
        target_fx = static_cast<unsigned long long>(ceil(t));
        if (target_fx < 1) target_fx = 1;
        if (lmass < target_fx) over = 1;
      }
      if (over == 0) {
        if (c.crank != leader) return;
        if (tid < static_cast<int>(c.csize)) sm.cnt[tid] = s[tid].u0;
        __syncthreads();
        leader_finish(P, sm, c, l_val, l_idx, R, row, topk_row, k, use_p, p, target_fx, m, c2, u,
                      st, q_row);
        return;
      }
      // Over capacity: every CTA falls through to the on-chip fallback.
    }

    // ---- fallback / plain rows: whole-row passes over the on-chip slices.
    float tk = -INFINITY;
    int ck = INT_MAX;
    bool pulled = false;  // other CTAs read this CTA's histograms: final barrier due
    auto tie_cutoff = [&](auto member, unsigned long long r) -> int {
      // First r members (index order) across the cluster; returns this
      // CTA's index cutoff.
      uint32_t cnt = 0;
      for_each<BF16, NV>(c, [&](float x, int e) { cnt += member(x, e) ? 1u : 0u; });
      const uint32_t wc = __reduce_add_sync(kFull, cnt);
      if (lane == 0) sm.wu[warp] = wc;
      __syncthreads();
      Slot cs = {};
      for (int w = 0; w < kWarps; ++w) cs.u0 += sm.wu[w];
      const Slot* s = push_exchange(sm, ph, c, cs);
      unsigned long long before = 0;
      for (uint32_t r2 = 0; r2 < c.crank; ++r2) before += s[r2].u0;
      const uint32_t mine_cnt = s[c.crank].u0;
      unsigned long long rl = r > before ? r - before : 0ull;
      if (rl > mine_cnt) rl = mine_cnt;
      int cut;
      if (rl == 0) {
        cut = INT_MIN;
      } else if (rl >= mine_cnt) {
        cut = INT_MAX;
      } else {
        uint32_t cum = 0, rw = 0;
        int wstar = kWarps - 1;
        for (int w = 0; w < kWarps; ++w) {
          if (cum + sm.wu[w] >= rl) {
            wstar = w;
            rw = static_cast<uint32_t>(rl) - cum;
            break;
          }
          cum += sm.wu[w];
        }
        if (warp == wstar) {
          uint32_t acc = 0;
          int found = INT_MAX;
          for (int j = 0; j < NV; ++j) {
            const uint4 v = s_vec[(warp * NV + j) * 32 + lane];
            const int e0 = c.lane_base + j * 32 * L::VW;
            uint32_t cj = 0;
            for_vector<BF16>(v, e0, [&](float x, int e) { cj += member(x, e) ? 1u : 0u; });
            const uint32_t incl = warp_inclusive_scan(cj, lane);
            const uint32_t stot = __shfl_sync(kFull, incl, 31);
            if (acc + stot >= rw) {
              const unsigned bal = __ballot_sync(kFull, acc + incl >= rw);
              const int lx = __ffs(bal) - 1;
              int sel = INT_MAX;
              if (lane == lx) {
                uint32_t need = rw - (acc + incl - cj);
                for_vector<BF16>(v, e0, [&](float x, int e) {
                  if (member(x, e)) {
                    if (need == 1 && sel == INT_MAX) sel = e;
                    --need;
                  }
                });
              }
              found = __shfl_sync(kFull, sel, lx);
              break;
            }
            acc += stot;
          }
          if (lane == 0) sm.bi[1] = found == INT_MAX ? INT_MAX : found + 1;
        }
        __syncthreads();
        cut = sm.bi[1];
      }
      __syncthreads();
      return cut;
    };

    if (topk_row) {
      // Count radix select of the k-th key over the whole row.
      uint32_t prefix = 0, pmask = 0;
      unsigned long long rem = static_cast<unsigned long long>(k);
      for (int lvl = 0; lvl < NLEV; ++lvl) {
        const int shift = 24 - 8 * lvl;
        PullBuf& pb = sm.pull[ph & 1];
        pb.lo[tid] = 0u;
        __syncthreads();
        for_each<BF16, NV>(c, [&](float x, int) {
          const uint32_t key = float_key(x);
          if ((key & pmask) == prefix) atomicAdd(&pb.lo[(key >> shift) & 0xffu], 1u);
        });
        cluster_sync();
        ++ph;
        pulled = true;
        unsigned long long tot = 0;
        for (uint32_t r = 0; r < c.csize; ++r) tot += ld_dsmem_u32(dsmem(&pb.lo[tid], r));
        unsigned long long above;
        const int b = select_bucket(tot, rem, sm, &above, tid, lane, warp);
        rem -= above;
        prefix |= static_cast<uint32_t>(b) << shift;
        pmask |= 0xffu << shift;
      }
      if (BF16 && !(prefix & 0x80000000u)) prefix |= 0xffffu;  // bf16 negatives: low bits ones
      tk = key_float(prefix);
      const float tkv = tk;
      ck = tie_cutoff([&](float x, int) { return x == tkv; }, rem);
    }
    const float tkf = tk;
    const int ckf = ck;
    auto in_k = [&](float x, int e) { return x > tkf || (x == tkf && e < ckf); };

    float tp = tk;
    int cp = ck;
    if (use_p) {
      uint32_t prefix = 0, pmask = 0;
      unsigned long long rem = 0;
      for (int lvl = 0; lvl < NLEV; ++lvl) {
        const int shift = 24 - 8 * lvl;
        PullBuf& pb = sm.pull[ph & 1];
        pb.lo[tid] = 0u;
        pb.hi[tid] = 0u;
        __syncthreads();
        for_each<BF16, NV>(c, [&](float x, int e) {
          const uint32_t key = float_key(x);
          if ((key & pmask) == prefix && in_k(x, e)) {
            const uint32_t d = (key >> shift) & 0xffu;
            atomic_add_u64_split(&pb.lo[d], &pb.hi[d], mass_fx(ex2((x - m) * c2)));
          }
        });
        cluster_sync();
        ++ph;
        pulled = true;
        unsigned long long tot = 0;
        for (uint32_t r = 0; r < c.csize; ++r) {
          tot += (static_cast<unsigned long long>(ld_dsmem_u32(dsmem(&pb.hi[tid], r))) << 32) +
                 ld_dsmem_u32(dsmem(&pb.lo[tid], r));
        }
        if (lvl == 0) {
          // Target: keep while (mass before) < p * Z_k, Z_k the exact total.
          const unsigned long long z_fx =
              block_suffix_scan<unsigned long long>(tot, sm.wl, lane, warp);
          if (tid == 0) sm.bl[0] = z_fx;
          __syncthreads();
          const unsigned long long zt = sm.bl[0];
          rem = static_cast<unsigned long long>(
              ceil(static_cast<double>(zt) * static_cast<double>(p)));
          if (rem < 1) rem = 1;
          if (rem > zt) rem = zt;
          __syncthreads();
        }
        unsigned long long above;
        const int b = select_bucket(tot, rem, sm, &above, tid, lane, warp);
        rem -= above;
        prefix |= static_cast<uint32_t>(b) << shift;
        pmask |= 0xffu << shift;
      }
      if (BF16 && !(prefix & 0x80000000u)) prefix |= 0xffffu;
      tp = key_float(prefix);
      const unsigned long long wt = mass_fx(ex2((tp - m) * c2));
      const unsigned long long rp = wt == 0 ? ~0ull : (rem + wt - 1) / wt;
      const float tpv = tp;
      cp = tie_cutoff([&](float x, int e) { return x == tpv && in_k(x, e); }, rp);
      if (tp == tk && ck < cp) cp = ck;  // the cut counted only K members
    }
    const float tpf = tp;
    const int cpf = cp;
    auto in_s = [&](float x, int e) {
      return in_k(x, e) && (x > tpf || (x == tpf && e < cpf));
    };

    // ---- inverse CDF over S in vocab order.
    float ts = 0.0f;
    for_each<BF16, NV>(c, [&](float x, int e) {
      if (in_s(x, e)) ts += ex2((x - m) * c2);
    });
    const float wsum = warp_sum(ts);
    if (lane == 0) sm.wf[warp] = wsum;
    __syncthreads();
    Slot cs = {};
    for (int w = 0; w < kWarps; ++w) cs.f0 += sm.wf[w];
    const Slot* s = push_exchange(sm, ph, c, cs);
    if (warp == 0) {
      const float t = lane < static_cast<int>(c.csize) ? s[lane].f0 : 0.0f;
      const float cum = warp_inclusive_scan(t, lane);
      const float Z = __shfl_sync(kFull, cum, 31);
      const float target = u * Z;
      const unsigned hit = __ballot_sync(kFull, lane < static_cast<int>(c.csize) && target < cum);
      int rstar;
      float tloc;
      if (hit != 0) {
        rstar = __ffs(hit) - 1;
        tloc = target - __shfl_sync(kFull, cum - t, rstar);
      } else {
        const unsigned pos = __ballot_sync(kFull, lane < static_cast<int>(c.csize) && t > 0.0f);
        rstar = pos ? 31 - __clz(pos) : 0;
        tloc = INFINITY;  // take the last kept token with mass
      }
      if (lane == 0) {
        sm.bi[0] = rstar;
        sm.bf[0] = tloc;
        sm.bf[1] = Z;
      }
    }
    __syncthreads();
    const int rstar = sm.bi[0];
    const float tloc = sm.bf[0];
    const float zs_all = sm.bf[1];
    if (c.crank == static_cast<uint32_t>(rstar)) {
      int wstar = -1;
      float tw = INFINITY;
      float cw = 0.0f;
      int wlast = -1;
      for (int w = 0; w < kWarps; ++w) {
        const float nc = cw + sm.wf[w];
        if (wstar < 0 && tloc < nc) {
          wstar = w;
          tw = tloc - cw;
        }
        if (sm.wf[w] > 0.0f) wlast = w;
        cw = nc;
      }
      if (wstar < 0) {
        wstar = wlast < 0 ? 0 : wlast;
        tw = INFINITY;
      }
      if (warp == wstar) {
        float acc = 0.0f;
        int found = -1;
        int lastpos = -1;
        for (int j = 0; j < NV; ++j) {
          const uint4 v = s_vec[(warp * NV + j) * 32 + lane];
          const int e0 = c.lane_base + j * 32 * L::VW;
          float lj = 0.0f;
          int llast = -1;
          for_vector<BF16>(v, e0, [&](float x, int e) {
            if (in_s(x, e)) {
              const float w = ex2((x - m) * c2);
              lj += w;
              if (w > 0.0f) llast = e;
            }
          });
          const unsigned has = __ballot_sync(kFull, llast >= 0);
          if (has != 0) lastpos = __shfl_sync(kFull, llast, 31 - __clz(has));
          const float incl = warp_inclusive_scan(lj, lane);
          const float stot = __shfl_sync(kFull, incl, 31);
          if (tw < acc + stot) {
            const unsigned bal = __ballot_sync(kFull, tw < acc + incl);
            const int lx = bal ? __ffs(bal) - 1 : 31;
            int sel = -1;
            if (lane == lx) {
              float run = acc + (incl - lj);
              for_vector<BF16>(v, e0, [&](float x, int e) {
                if (in_s(x, e)) {
                  run += ex2((x - m) * c2);
                  if (sel < 0 && tw < run) sel = e;
                }
              });
              if (sel < 0) sel = llast;
            }
            found = __shfl_sync(kFull, sel, lx);
            if (found < 0) found = lastpos;
            break;
          }
          acc += stot;
        }
        if (found < 0) found = lastpos;
        if (lane == 0) emit_token(P, row, found, found < 0 ? (st | kStNonFinite) : st);
      }
    }
    if (q_row != nullptr) {
      const float inv = 1.0f / zs_all;
      for_each<BF16, NV>(c, [&](float x, int e) {
        if (e < V) q_row[e] = in_s(x, e) ? ex2((x - m) * c2) * inv : 0.0f;
      });
    }
    // Other CTAs read this CTA's histograms after the barriers above; stay
    // until every CTA is past them.
    if (pulled) cluster_sync();

  }
}

}  // namespace pkv
