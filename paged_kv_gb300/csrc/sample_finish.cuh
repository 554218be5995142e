// Finish kernel of the batched sampler: one CTA per row reads the stream
// kernel's records of the row from the workspace and settles the token (see
// sample_common.cuh for the row kinds).
//
// Every phase here runs once per row, so the kernel is built for latency:
// the record parts a row reads arrive in bulk copies issued together,
// per-record work is spread over the threads and combined by warp
// reductions (no thread walks the C * 8 warp records alone), and the
// write-back coordinates are loaded at the start.
#pragma once

#include "page_fill.cuh"
#include "sample_common.cuh"

namespace pkv {

// The row's head: its maximum m over the warp maxima (NaN if any is NaN),
// the first record entry (chunk * kWarps + warp, index order) holding m, and
// whether any warp record is stale (not from this call).
struct RowHead {
  float m;
  int first;
  bool nan;
  bool stale;
};

__device__ __forceinline__ RowHead row_head(const ChunkSlot* recs, int C, uint32_t seq,
                                            SampleSmem& sm, const Ctx& c) {
  const int i = c.tid;
  const bool in = i < C * kWarps;
  const float x = in ? recs[i / kWarps].wm[i % kWarps] : -INFINITY;
  const bool nan = x != x;
  const bool stale = in && recs[i / kWarps].wseq[i % kWarps] != seq;
  const uint32_t key = nan ? 0u : float_key(x);
  const uint32_t wk = __reduce_max_sync(kFull, key);
  const int wfirst = static_cast<int>(
      __reduce_min_sync(kFull, (in && !nan && key == wk) ? static_cast<uint32_t>(i) : 0x7fffffffu));
  const unsigned flags = (__any_sync(kFull, nan) ? 1u : 0u) | (__any_sync(kFull, stale) ? 2u : 0u);
  if (c.lane == 0) {
    sm.wu[c.warp] = wk;
    sm.wi[c.warp] = wfirst;
    sm.bi[c.warp] = static_cast<int32_t>(flags);
  }
  group_sync();
  uint32_t k = 0;
  unsigned f = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    k = max(k, sm.wu[w]);
    f |= static_cast<unsigned>(sm.bi[w]);
  }
  int first = INT_MAX;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (sm.wu[w] == k) first = min(first, sm.wi[w]);
  }
  group_sync();
  RowHead h;
  h.m = (f & 1u) ? __uint_as_float(0x7fc00000u) : key_float(k);
  h.first = first;
  h.nan = (f & 1u) != 0;
  h.stale = (f & 2u) != 0;
  return h;
}

// The write-back coordinates of a row, loaded early so that emitting the
// token costs no dependent global loads.
struct WriteBack {
  int64_t col;
  int64_t prow;
};

__device__ __forceinline__ WriteBack load_write_back(const SampleParams& P, int row) {
  WriteBack wb;
  wb.col = -1;
  wb.prow = 0;
  if (P.token_pool != nullptr) {
    wb.col = P.wb_cols[row];
    wb.prow = P.wb_rows[row];
  }
  return wb;
}

// out_tokens[row] = tok and the fused write-back (column < 0: no write; a
// token of -1 is not written); status bits are OR-ed in.
__device__ __forceinline__ void emit(const SampleParams& P, int row, int tok, int st,
                                     const WriteBack& wb) {
  P.out_tokens[row] = tok;
  if (P.token_pool != nullptr && tok >= 0 && wb.col >= 0) {
    if (wb.prow < 0 || wb.prow >= P.pool_rows) {
      st |= kStRowOOB;
    } else if (wb.col >= P.pool_cols) {
      st |= kStColOOB;
    } else {
      P.token_pool[wb.prow * P.pool_cols + wb.col] = tok;
    }
  }
  if (st != 0 && P.status != nullptr) atomicOr(P.status, st);
}

// ----------------------------------------------------------------- plain finish (P)

// Inclusive prefix over the CTA's threads in tid order, with each thread's
// exclusive prefix taken as its predecessor's inclusive one (not incl - v):
// the intervals [before, incl) of threads with mass then tile [0, total)
// without gaps or overlaps, so at most one thread owns a point of it.
__device__ __forceinline__ float block_incl_scan_f(float v, float* s_w, int lane, int warp,
                                                   float* before, float* total) {
  const float wincl = warp_inclusive_scan(v, lane);
  if (lane == 31) s_w[warp] = wincl;
  group_sync();
  float off = 0.0f, all = 0.0f;
#pragma unroll 1
  for (int w = 0; w < kWarps; ++w) {
    if (w == warp) off = all;
    all += s_w[w];
  }
  group_sync();
  const float incl = off + wincl;
  const float prev = __shfl_up_sync(kFull, incl, 1);
  *before = lane == 0 ? off : prev;
  *total = all;
  return incl;
}

// No filter: the draw is over the whole row.  Warp 0 scans the record masses
// (warp w of chunk r: wz relative to its maximum wm) in index order to find
// the (chunk, warp) holding u * Z; the CTA re-reads that warp's slice (an L2
// hit; two consecutive vectors per thread), one prefix over the CTA finds the
// thread holding the rest of the draw, and that thread the token.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void finish_plain(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                             const ChunkSlot* recs, int row, const RowParams& rp,
                                             float m, const WriteBack& wb, float* q_row) {
  using L = Layout<BF16>;
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  if (warp == 0) {
    // Lane l holds entries 4l .. 4l + 3 (entry chunk * kWarps + warp; C * kWarps <= 128).
    float mw[4];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * lane + j;
      mw[j] = 0.0f;
      if (e < C * kWarps) {
        const float wmax = recs[e / kWarps].wm[e % kWarps];
        if (wmax > -INFINITY) mw[j] = recs[e / kWarps].wz[e % kWarps] * ex2((wmax - m) * rp.c2);
      }
      s += mw[j];
    }
    const float incl = warp_inclusive_scan(s, lane);
    const float zrow = __shfl_sync(kFull, incl, 31);
    float target = rp.u * zrow;
    if (!(target < zrow)) target = nextafterf(zrow, 0.0f);
    // The lane whose interval holds target; rounding can leave none: then
    // the last lane with mass, at the end of its last entry with mass.
    const unsigned hit = __ballot_sync(kFull, s > 0.0f && target < incl);
    const unsigned pos = __ballot_sync(kFull, s > 0.0f);
    const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    if (lane == l) {
      float run = incl - s;
      int estar = -1, elast = -1;
      float tau = INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (mw[j] > 0.0f) {
          elast = 4 * lane + j;
          if (estar < 0 && hit != 0u && target < run + mw[j]) {
            estar = elast;
            tau = fmaxf(target - run, 0.0f);
          }
          run += mw[j];
        }
      }
      if (estar < 0) {
        estar = elast;
        tau = INFINITY;
      }
      sm.bi[0] = pos ? estar : -1;
      sm.bf4[0] = tau;
      sm.bf4[1] = zrow;
    }
  }
  group_sync();
  const int estar = sm.bi[0];
  const float tau = sm.bf4[0];
  const float zrow = sm.bf4[1];
  if (estar < 0) {
    if (tid == 0) emit(P, row, -1, rp.st | kStNonFinite, wb);
  } else {
    // Vectors 2t and 2t + 1 of the slice (vector j * 32 + l of the stream
    // layout): 2 * VW consecutive elements from e0.
    const int r = estar / kWarps, w = estar % kWarps;
    const bool active = tid < NV * 16;
    const int e0 = vec_base<BF16, NV>(r, w, (2 * tid) % 32, (2 * tid) / 32);
    uint4 v[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    if (active) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t q[4];
        load_vec<BF16, NV, VEC>(P, row, e0 + k * L::VW, q);
        v[k] = make_uint4(q[0], q[1], q[2], q[3]);
      }
    }
    float s = 0.0f;
    int last = -1;
    if (active) {
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        for_vec_c<BF16>(k == 0 ? v[0] : v[1], e0 + k * L::VW, [&](float x, int e) {
          const float wt = e < V ? weight(x, m, rp.c2) : 0.0f;
          s += wt;
          if (wt > 0.0f) last = e;
        });
      }
    }
    float before, total;
    const float incl = block_incl_scan_f(s, sm.wt, lane, warp, &before, &total);
    const bool mine = s > 0.0f && tau >= before && tau < incl;
    if (mine) {
      float run = before;
      int sel = -1;
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        for_vec_c<BF16>(k == 0 ? v[0] : v[1], e0 + k * L::VW, [&](float x, int e) {
          const float wt = e < V ? weight(x, m, rp.c2) : 0.0f;
          if (sel < 0 && wt > 0.0f && tau < run + wt) sel = e;
          run += wt;
        });
      }
      emit(P, row, sel >= 0 ? sel : last, rp.st, wb);
    }
    if (!(tau < total)) {
      // The rest of the draw lies past the slice's own mass (rounding): its
      // last element with mass.
      const int lastall = block_max_int(last, sm.wi, lane, warp);
      if (tid == 0) emit(P, row, lastall, lastall < 0 ? (rp.st | kStNonFinite) : rp.st, wb);
    }
  }
  if (q_row != nullptr) {
    const float inv = 1.0f / zrow;
    for (int r = 0; r < C; ++r) {
      uint32_t d[NV][4];
      load_chunk<BF16, NV, VEC>(P, row, r, warp, lane, d);
      for_regs<BF16, NV>(d, r, warp, lane, [&](float x, int e) {
        if (e < V) q_row[e] = weight(x, m, rp.c2) * inv;
      });
    }
  }
}

// ----------------------------------------------------------------- top-k finish (K)

// theta = the k-th largest thread maximum of the row (or a lower bound on
// it): at least k elements are >= theta, so the top-k lies in the threads
// whose maximum is >= theta.  Their vectors are re-read (an L2 hit) and the
// elements >= theta appended to a list (any order).  The list is ranked by
// (value desc, index asc) with all-pairs comparisons (it holds about k
// entries), which gives the top-k in order; top-p is a prefix scan over it,
// and the draw a scan over the kept entries in index order.  Returns false,
// having emitted nothing, when the list overflows (pathological ties); the
// caller then runs the exact fallback.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ bool finish_topk(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                            const ChunkSlot* recs, float* l_val, int32_t* l_idx,
                                            int row, const RowParams& rp, float m,
                                            const WriteBack& wb, float* q_row) {
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  const int k = rp.k;
  const int nT = C * kThreads;
  auto tmax_at = [&](int i) { return recs[i / kThreads].tmax[i % kThreads]; };
  // ---- theta: thread maxima counted per 16-bit key below the row maximum
  // (bucket i = key(m) - key; keys beyond 255 share the last bucket); the
  // key where the count from the top reaches k.  For bf16 rows it is the
  // exact k-th largest thread maximum when within 256 values of m;
  // otherwise a lower bound, or (last bucket) the exact select.
  const uint32_t km = key16(m);
  sm.hlo[tid] = 0u;
  group_sync();
  for (int i = tid; i < nT; i += kThreads) {
    const float t = tmax_at(i);
    if (t == t) {
      const uint32_t kt = key16(t);
      atomicAdd(&sm.hlo[kt >= km ? 0u : min(km - kt, 255u)], 1u);
    }
  }
  group_sync();
  {
    const uint32_t h = sm.hlo[tid];
    uint32_t tot;
    const uint32_t before = block_exclusive_scan<uint32_t>(h, sm.wu, lane, warp, &tot);
    if (before < static_cast<uint32_t>(k) && before + h >= static_cast<uint32_t>(k)) sm.bi[1] = tid;
    if (tid == 0 && tot < static_cast<uint32_t>(k)) sm.bi[1] = -1;
  }
  group_sync();
  const int bk = sm.bi[1];
  group_sync();
  if (bk < 0) return false;
  float theta;
  if (bk < 255) {
    theta = key16_float(km - static_cast<uint32_t>(bk));
  } else {
    for (int i = tid; i < nT; i += kThreads) l_val[i] = tmax_at(i);
    group_sync();
    unsigned long long rk;
    theta = list_select<false>(l_val, nT, [](int) { return true; }, [](int) { return 1ull; },
                               static_cast<unsigned long long>(k), sm, c, &rk);
  }
  if (!(theta > -INFINITY)) return false;
  // ---- candidate threads, then their vectors: elements >= theta appended.
  uint16_t* cand = reinterpret_cast<uint16_t*>(sm.scan);  // up to 4 * kBuckets thread ids
  constexpr int kCandCap = 4 * kBuckets;
  if (tid == 0) {
    sm.bi[4] = 0;
    sm.bi[5] = 0;
  }
  group_sync();
  for (int i = tid; i < nT; i += kThreads) {
    if (tmax_at(i) >= theta) {
      const int at = atomicAdd(&sm.bi[4], 1);
      if (at < kCandCap) cand[at] = static_cast<uint16_t>(i);
    }
  }
  group_sync();
  const int ncand = sm.bi[4];
  if (ncand > kCandCap) return false;
  // Entries are packed sort keys: order key of the value above, the
  // complement of the index below, so that a larger key comes first in
  // (value desc, index asc).
  unsigned long long* list = reinterpret_cast<unsigned long long*>(l_val);
  auto append = [&](const uint32_t (&w4)[4], int e0) {
    for_vec<BF16>(w4, e0, [&](float x, int e) {
      if (e < V && x >= theta) {
        const int at = atomicAdd(&sm.bi[5], 1);
        if (at < kFinListCap) {
          list[at] = (static_cast<unsigned long long>(float_key(x)) << 32) |
                     static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(e));
        }
      }
    });
  };
  auto cand_vec = [&](int v) {
    const int i = cand[v / NV];
    const int ct = i % kThreads;
    return vec_base<BF16, NV>(i / kThreads, ct / 32, ct % 32, v % NV);
  };
  for (int v = tid; v < ncand * NV; v += kThreads) {
    const int e = cand_vec(v);
    uint32_t w[4];
    load_vec<BF16, NV, VEC>(P, row, e, w);
    append(w, e);
  }
  group_sync();
  const int n = sm.bi[5];
  if (n > kFinListCap || n < k) return false;
  // ---- ranks: the number of entries with a larger key; sorted[rank] for rank < k.
  uint32_t* sorted = sm.hlo;
  for (int i = tid; i < n; i += kThreads) {
    const unsigned long long ki = list[i];
    int rank = 0;
#pragma unroll 4
    for (int j = 0; j < n; ++j) rank += list[j] > ki ? 1 : 0;
    if (rank < k) sorted[rank] = static_cast<uint32_t>(i);
  }
  group_sync();
  // ---- top-p inside K: thread t < k holds the t-th of the order.
  const bool in_k = tid < k;
  const unsigned long long kme = in_k ? list[sorted[tid]] : 0ull;
  const float xv = in_k ? key_float(static_cast<uint32_t>(kme >> 32)) : -INFINITY;
  const int xi = in_k ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(kme)) : INT_MAX;
  const float wf = in_k ? weight(xv, m, rp.c2) : 0.0f;
  const unsigned long long w = in_k ? mass_fx(wf) : 0ull;
  unsigned long long zk;
  const unsigned long long before =
      block_exclusive_scan<unsigned long long>(w, sm.wl, lane, warp, &zk);
  unsigned long long target = zk + 1ull;  // p == 1: keep all of K
  if (rp.use_p) {
    target = mul_fx(zk, rp.p, true);
    if (target < 1ull) target = 1ull;
    if (target > zk) target = zk;
  }
  // min_p: weights fall with the rank, so the cut keeps S a prefix.
  const bool kept = in_k && before < target && (rp.minp <= 0.0f || wf >= rp.minp);
  // ---- draw in index order over S = the first s of the order: entry t
  // owns [c_t, c_t + w_t) with c_t the mass of the kept entries of smaller
  // index; the intervals tile [0, Z_S) exactly (fixed point).
  int32_t* kidx = reinterpret_cast<int32_t*>(sm.hhi);
  unsigned long long* kw = sm.scan;  // the candidate ids are consumed
  kidx[tid] = kept ? xi : INT_MAX;
  kw[tid] = kept ? w : 0ull;
  const int s = block_max_int(kept ? tid + 1 : 0, sm.wi, lane, warp);  // its barriers publish kidx, kw
  unsigned long long cum = 0, zs = 0;
#pragma unroll 4
  for (int t = 0; t < s; ++t) {
    const unsigned long long wt = kw[t];
    zs += wt;
    cum += kidx[t] < xi ? wt : 0ull;
  }
  const unsigned long long tdraw = mul_fx(zs, rp.u, false);
  const bool owner = kept && w > 0ull && tdraw >= cum && tdraw < cum + w;
  if (owner) emit(P, row, xi, rp.st, wb);
  if (__syncthreads_or(owner) == 0 && tid == 0) emit(P, row, -1, rp.st | kStNonFinite, wb);
  if (q_row != nullptr) {
    const float zf = block_sum<float>(kept ? wf : 0.0f, sm.wt, lane, warp);
    if (kept) q_row[xi] = wf / zf;
  }
  return true;
}

// ----------------------------------------------------------------- histogram finish (H)

// Chunk r counted its elements per 16-bit key over the kHistKeys keys below
// a_r = its summary's i0, the key of its maximum: 16-bit count d of its
// histogram is the count of key a_r - d.  Merged key i (0 = the row maximum,
// key A - i) has count sum_r h_r[i - (A - a_r)]; every element within
// kHistKeys keys of the row maximum is counted in its chunk (a_r <= A).
//
// The finisher settles top-k (by count) and top-p (by fixed-point mass)
// exactly on the merged keys: keys i < is are wholly in the kept set S, the
// first rs members (in index order) of key is are in it too.  It then picks
// the chunk holding the draw from per-chunk masses of S, the slice of that
// chunk from the stream kernel's per-warp histograms, and the token from one
// prefix over the slice's elements.  Returns false,
// having emitted nothing, when a cut lies below the merged window; the
// caller then runs the exact fallback.
template <int NV, bool VEC>
__device__ __forceinline__ bool finish_hist(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                            const ChunkSlot* recs, unsigned long long* table,
                                            uint4* stage, int row, const RowParams& rp, float m,
                                            const WriteBack& wb, float* q_row) {
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  const int k = rp.k;
  const bool topk = k < V;
  const uint32_t A = key16(m);
  // The row's total mass (for top-p without top-k), from the warp records:
  // warp 0 alone (lane l: entries 4l .. 4l + 3), published by the barriers
  // of the scans below.
  if (!topk && warp == 0) {
    float z = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * lane + j;
      if (e < C * kWarps) {
        const float wmax = recs[e / kWarps].wm[e % kWarps];
        if (wmax > -INFINITY) z += recs[e / kWarps].wz[e % kWarps] * ex2((wmax - m) * rp.c2);
      }
    }
    z = warp_sum(z);
    if (lane == 0) sm.bf4[2] = z;
  }
  // ---- merged counts and fixed-point weights; thread t holds keys 4t .. 4t + 3.
  uint32_t cnt[4] = {0u, 0u, 0u, 0u};
#pragma unroll 1
  for (int r = 0; r < C; ++r) {
    const uint32_t delta = A - static_cast<uint32_t>(recs[r].s.i0);
    const uint16_t* h16 = reinterpret_cast<const uint16_t*>(recs[r].hist);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t i = static_cast<uint32_t>(4 * tid + jj);
      if (i >= delta) cnt[jj] += h16[i - delta];
    }
  }
  // Every key's weight, empty keys included (they only ever meet a zero
  // count); one rolled loop, read back from the table below.
#pragma unroll 1
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t i = static_cast<uint32_t>(4 * tid + jj);
    table[i] = A >= i ? mass_fx(weight(key16_float(A - i), m, rp.c2)) : 0ull;
  }
  const unsigned long long* wfx = table + 4 * tid;  // this thread's four keys
  // No owner below leaves a cut at kHistKeys (the barriers of the scans
  // order these before the owners' writes).
  if (tid == 0) {
    sm.bi[6] = kHistKeys;
    sm.bi[7] = kHistKeys;
  }
  // ---- top-k by count: keys i < ik are wholly in K, key ik keeps rk members.
  int ik = kHistKeys;
  unsigned long long rk = 0;
  if (topk) {
    const uint32_t local = cnt[0] + cnt[1] + cnt[2] + cnt[3];
    uint32_t total;
    const uint32_t before = block_exclusive_scan<uint32_t>(local, sm.wu, lane, warp, &total);
    if (total < static_cast<uint32_t>(k)) return false;  // the k-th value lies below the window
    // Exactly one key brings the count from below k to k or more.
    uint32_t run = before;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (run < static_cast<uint32_t>(k) && run + cnt[jj] >= static_cast<uint32_t>(k)) {
        sm.bi[6] = 4 * tid + jj;
        sm.bl[0] = static_cast<unsigned long long>(k) - run;
      }
      run += cnt[jj];
    }
    group_sync();
    ik = sm.bi[6];
    rk = sm.bl[0];
  }
  // ---- top-p inside K by mass: keys i < is wholly in S, key is keeps rs.
  int is = ik;
  unsigned long long rs = rk;
  if (rp.use_p) {
    unsigned long long mk[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int i = 4 * tid + jj;
      mk[jj] = i < ik ? cnt[jj] * wfx[jj] : (i == ik ? rk * wfx[jj] : 0ull);
    }
    const unsigned long long local = mk[0] + mk[1] + mk[2] + mk[3];
    unsigned long long zk;
    const unsigned long long before =
        block_exclusive_scan<unsigned long long>(local, sm.wl, lane, warp, &zk);
    unsigned long long target;
    if (topk) {
      target = mul_fx(zk, rp.p, true);
      if (target > zk) target = zk;
    } else {
      target = mul_fx(fx40(sm.bf4[2]), rp.p, true);
      if (zk < target) return false;  // the top-p cut lies below the window
    }
    if (target < 1) target = 1;
    // Exactly one key brings the mass from below target to target or more
    // (1 <= target <= zk).
    int cand = INT_MAX;
    unsigned long long run = before, rem = 0, wc = 0, nc = 0;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (run < target && run + mk[jj] >= target) {
        cand = 4 * tid + jj;
        rem = target - run;
        wc = wfx[jj];
        nc = cnt[jj];
      }
      run += mk[jj];
    }
    if (cand != INT_MAX) {
      // Members j of the cut key are kept iff run + j * w < target; at most
      // the key's count of them.
      unsigned long long need = wc == 0 ? ~0ull : ceil_div_small(rem, wc, nc);
      if (cand == ik && need > rk) need = rk;
      sm.bl[1] = need;
      sm.bi[7] = cand;
    }
    group_sync();
    is = sm.bi[7];
    rs = sm.bl[1];
  }
  if (rp.minp > 0.0f) {
    // min_p: the first key whose weight is below minp ends the kept set (key
    // 0, the row maximum, weighs 1).
    int cut = INT_MAX;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int i = 4 * tid + jj;
      if (weight(key16_float(A - static_cast<uint32_t>(i)), m, rp.c2) < rp.minp) cut = min(cut, i);
    }
    cut = block_min_int(cut, sm.wi, lane, warp);
    if (cut <= is) {
      is = cut;
      rs = 0;
    }
  }
  if (is >= kHistKeys) return false;  // a cut below the window: the exact path
  const unsigned long long wcut = table[is];
  // ---- per-chunk mass of S above the cut key and the cut key's members.
  for (int r = warp; r < C; r += kWarps) {
    const uint32_t delta = A - static_cast<uint32_t>(recs[r].s.i0);
    const uint16_t* h16 = reinterpret_cast<const uint16_t*>(recs[r].hist);
    unsigned long long part = 0;
#pragma unroll 1
    for (int i = lane; i < is; i += 32) {
      if (static_cast<uint32_t>(i) >= delta) part += h16[i - delta] * table[i];
    }
    part = warp_sum_u64(part);
    if (lane == 0) {
      sm.cmass[r][0] = part;
      sm.ties[r] = static_cast<uint32_t>(is) >= delta ? h16[is - delta] : 0u;
    }
  }
  group_sync();
  // ---- the chunk holding the draw (warp 0, lane r = chunk r; C <= 32):
  // chunk r keeps the first kept_r = clamp(rs - ties before r, 0, ties_r)
  // members of the cut key, since they follow one another in index order.
  if (warp == 0) {
    const bool v = lane < C;
    const uint32_t ties = v ? sm.ties[lane] : 0u;
    const uint32_t tb = warp_inclusive_scan(ties, lane) - ties;
    const unsigned long long kept =
        v ? min(static_cast<unsigned long long>(ties), rs > tb ? rs - tb : 0ull) : 0ull;
    const unsigned long long mr = v ? sm.cmass[lane][0] + kept * wcut : 0ull;
    const unsigned long long incl = warp_inclusive_scan(mr, lane);
    const unsigned long long zs = __shfl_sync(kFull, incl, 31);
    unsigned long long tdraw = mul_fx(zs, rp.u, false);
    if (tdraw >= zs) tdraw = zs - 1;  // zs >= the row maximum's own weight > 0
    const unsigned bal = __ballot_sync(kFull, v && tdraw < incl);
    const int cstar = bal ? __ffs(bal) - 1 : C - 1;
    if (v) sm.cnt[lane] = static_cast<uint32_t>(kept);
    if (lane == cstar) {
      sm.bi[0] = cstar;
      sm.bi[4] = static_cast<int>(A - static_cast<uint32_t>(recs[cstar].s.i0));
      sm.bl[3] = tdraw - (incl - mr);
      sm.bl[5] = zs;
    }
  }
  group_sync();
  const int cstar = sm.bi[0];
  const unsigned long long tau = sm.bl[3];
  const unsigned long long zs = sm.bl[5];
  const uint32_t kept_c = sm.cnt[cstar];
  // In a chunk, the mass of S before a position is the mass above the cut
  // key plus wcut * min(cut-key members so far, kept): the first kept
  // members count, later ones do not.
  auto above_and_ties = [&](const uint4 v4, int e0, unsigned long long* a, uint32_t* t) {
    unsigned long long s = 0;
    uint32_t n = 0;
    for_vec_c<true>(v4, e0, [&](float x, int e) {
      if (e < V) {
        const uint32_t i = A - key16(x);
        if (i < static_cast<uint32_t>(is)) s += table[i];
        n += i == static_cast<uint32_t>(is) ? 1u : 0u;
      }
    });
    *a = s;
    *t = n;
  };
  // ---- the slice of the chunk holding the draw, from the stream kernel's
  // per-warp histograms of the chunk (copied over the consumed records):
  // slice w (NV vectors of 32 lanes, contiguous in index order) has mass
  // a_w above the cut key and t_w cut-key members.
  const uint32_t dc = static_cast<uint32_t>(sm.bi[4]);  // merged key i = slice key i - dc
  {
    const uint4* src = ws_slice_hist(P, row, cstar);
#pragma unroll 1
    for (int k = tid; k < static_cast<int>(kSliceHistBytes / 16); k += kThreads) {
      cp_async16(stage + k, src + k);
    }
    cp_async_wait_all();
  }
  group_sync();
  {
    const uint16_t* hw = reinterpret_cast<const uint16_t*>(stage) + warp * kHistKeys;
    unsigned long long a = 0;
    uint32_t t = 0;
#pragma unroll 1
    for (int i = static_cast<int>(dc) + lane; i <= is; i += 32) {
      const uint32_t n = hw[i - static_cast<int>(dc)];
      if (i < is) {
        a += n * table[i];
      } else {
        t = n;
      }
    }
    a = warp_sum_u64(a);
    t = __reduce_add_sync(kFull, t);
    if (lane == 0) {
      sm.scan[warp] = a;
      sm.hlo[warp] = t;
    }
  }
  group_sync();
  // Every warp finds the draw's slice (lanes 0 .. kWarps - 1 hold the slices).
  int wstar;
  unsigned long long a_w;  // mass of S in the chunk before that slice without
  uint32_t t_w;            // the cut key, and the cut-key members before it
  {
    const unsigned long long a = lane < kWarps ? sm.scan[lane] : 0ull;
    const uint32_t t = lane < kWarps ? sm.hlo[lane] : 0u;
    const unsigned long long ai = warp_inclusive_scan(a, lane);
    const uint32_t ti = warp_inclusive_scan(t, lane);
    const unsigned long long pi =
        ai + wcut * min(static_cast<unsigned long long>(ti), static_cast<unsigned long long>(kept_c));
    const unsigned bal = __ballot_sync(kFull, lane < kWarps && tau < pi);
    wstar = bal ? __ffs(bal) - 1 : -1;
    const int from = wstar < 0 ? 0 : wstar;
    a_w = __shfl_sync(kFull, ai - a, from);
    t_w = __shfl_sync(kFull, ti - t, from);
  }
  // ---- the slice's NV * 32 vectors, two consecutive ones per thread (L2
  // reads), one prefix over the CTA, and the element in the thread whose
  // range holds tau.
  const bool active = wstar >= 0 && tid < NV * 16;
  uint32_t v[2][4] = {{0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};
  int e0[2] = {0, 0};
  unsigned long long a = 0;
  uint32_t t = 0;
  if (active) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      e0[k] = cstar * (kThreads * NV * 8) + (wstar * NV * 32 + 2 * tid + k) * 8;
      load_vec<true, NV, VEC>(P, row, e0[k], v[k]);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      unsigned long long ak;
      uint32_t tk;
      above_and_ties(make_uint4(v[k][0], v[k][1], v[k][2], v[k][3]), e0[k], &ak, &tk);
      a += ak;
      t += tk;
    }
  }
  const unsigned long long ai = warp_inclusive_scan(a, lane);
  const uint32_t ti = warp_inclusive_scan(t, lane);
  if (lane == 31) {
    sm.wl[warp] = ai;
    sm.wu[warp] = ti;
  }
  group_sync();
  unsigned long long ab = a_w;
  uint32_t tb = t_w;
#pragma unroll 1
  for (int w = 0; w < warp; ++w) {
    ab += sm.wl[w];
    tb += sm.wu[w];
  }
  const unsigned long long a_in = ab + ai, a_ex = a_in - a;
  const uint32_t t_in = tb + ti, t_ex = t_in - t;
  const unsigned long long p_in =
      a_in + wcut * min(static_cast<unsigned long long>(t_in), static_cast<unsigned long long>(kept_c));
  const unsigned long long p_ex =
      a_ex + wcut * min(static_cast<unsigned long long>(t_ex), static_cast<unsigned long long>(kept_c));
  const bool mine = active && tau >= p_ex && tau < p_in;
  // The owner of tau (at most one thread) hands its 16 elements to lanes
  // 0..15 of its warp, in index order; two warp scans give each element the
  // mass of S before it, and the first element whose interval holds tau is
  // the token (else the last one that carries mass).
  const unsigned own = __ballot_sync(kFull, mine);
  if (own != 0u) {
    const int ol = __ffs(own) - 1;
    const int j = lane & 15;
    const int want = (j >> 3) * 4 + ((j & 7) >> 1);  // word of element j
    uint32_t word = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t x = __shfl_sync(kFull, q < 4 ? v[0][q] : v[1][q - 4], ol);
      if (q == want) word = x;
    }
    const int e = __shfl_sync(kFull, e0[0], ol) + j;  // e0[1] = e0[0] + 8
    const unsigned long long aex = __shfl_sync(kFull, a_ex, ol);
    const uint32_t tex = __shfl_sync(kFull, t_ex, ol);
    const float x = elem<true>(word, j & 1);
    const bool valid = lane < 16 && e < V;
    const uint32_t i = A - key16(x);
    const bool above = valid && i < static_cast<uint32_t>(is);
    const bool tie = valid && i == static_cast<uint32_t>(is);
    const unsigned long long wa = above ? table[i] : 0ull;
    const uint32_t ti1 = tie ? 1u : 0u;
    const unsigned long long abefore = aex + warp_inclusive_scan(wa, lane) - wa;
    const uint32_t tc = tex + warp_inclusive_scan(ti1, lane) - ti1;
    const unsigned long long pb =
        abefore + wcut * min(static_cast<unsigned long long>(tc),
                             static_cast<unsigned long long>(kept_c));
    const unsigned long long w = above ? wa : ((tie && tc < kept_c) ? wcut : 0ull);
    const unsigned hit = __ballot_sync(kFull, w > 0 && tau < pb + w);
    const unsigned pos = __ballot_sync(kFull, w > 0);
    const int src = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    const int sel = __shfl_sync(kFull, e, src < 0 ? 0 : src);
    if (lane == 0) {
      const int tok = src < 0 ? -1 : sel;
      emit(P, row, tok, tok < 0 ? (rp.st | kStNonFinite) : rp.st, wb);
    }
  }
  // No thread's range holds tau only when the masses are not finite.
  if (__syncthreads_or(mine) == 0 && tid == 0) emit(P, row, -1, rp.st | kStNonFinite, wb);
  if (q_row != nullptr) {
    // Debug output: q over every chunk; a cut-key member is kept when its
    // rank among the chunk's members is below kept_r.
    const float inv = 1.0f / (static_cast<float>(zs) / kMassScale);
    for (int r = 0; r < C; ++r) {
      group_sync();
      stage_own<true, NV, VEC>(P, row, r, stage, warp, lane);
      for (int j = 0; j < NV; ++j) {
        unsigned long long a;
        uint32_t t;
        above_and_ties(stage[(warp * NV + j) * 32 + lane], vec_base<true, NV>(r, warp, lane, j),
                       &a, &t);
        t = __reduce_add_sync(kFull, t);
        if (lane == 0) sm.hlo[warp * NV + j] = t;
      }
      group_sync();
      if (tid == 0) {
        uint32_t acc = 0;
        for (int q = 0; q < kWarps * NV; ++q) {
          const uint32_t t = sm.hlo[q];
          sm.hlo[q] = acc;
          acc += t;
        }
      }
      group_sync();
      const uint32_t kept_r = sm.cnt[r];
      for (int j = 0; j < NV; ++j) {
        const int e0 = vec_base<true, NV>(r, warp, lane, j);
        const uint4 v4 = stage[(warp * NV + j) * 32 + lane];
        unsigned long long a;
        uint32_t t;
        above_and_ties(v4, e0, &a, &t);
        uint32_t rank = sm.hlo[warp * NV + j] + warp_inclusive_scan(t, lane) - t;
        for_vec_c<true>(v4, e0, [&](float x, int e) {
          if (e < V) {
            const uint32_t i = A - key16(x);
            bool in = i < static_cast<uint32_t>(is);
            if (i == static_cast<uint32_t>(is)) in = rank++ < kept_r;
            q_row[e] = in ? weight(x, m, rp.c2) * inv : 0.0f;
          }
        });
      }
    }
  }
  return true;
}

// ----------------------------------------------------------------- candidate finish (T)

// The chunks' candidate lists hold every element of the row at or above
// thr, the largest of the chunks' bounds.  The entries at or above thr are
// gathered from the workspace as packed keys (order key of the value above,
// the complement of the index below: a larger key comes first in (value
// desc, index asc)).  When the top-p cut lies among them (their mass
// reaches p * Z), S_p is a prefix of that order.  Its end is found without
// sorting: the entries' masses are summed in 256 buckets of equal width
// over the values [thr, m] (a bucket index that never falls as the value
// rises), a suffix scan over the buckets finds the one holding the cut, and
// only that bucket's entries are ranked exactly, so the tied members of the
// cut value enter in index order.  S is S_p less the weights below min_p.
// The draw is in index order: the mass of S per index bucket (256 over
// [0, V)) and one prefix find the bucket holding floor(u * Z_S); inside it
// entry t owns [c_t, c_t + w_t), c_t the mass of the bucket's entries of S
// with a smaller index, so the intervals tile [0, Z_S) exactly.  Returns
// false, having emitted nothing, when a list overflowed, the gathered
// entries exceed the capacity, the cut lies below thr or a resolved bucket
// holds more than kBuckets entries; the caller then runs the exact fallback.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ bool finish_cand(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                            unsigned char* scratch, const ChunkSlot* recs,
                                            unsigned long long* keys, int row,
                                            const RowParams& rp, float m, const WriteBack& wb,
                                            float* q_row) {
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  // ---- warp 0: the row's total mass from the warp records, the list
  // offsets (sm.cnt), their total, the largest bound and overflow (C <= 32).
  if (warp == 0) {
    float z = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * lane + j;
      if (e < C * kWarps) {
        const float wmax = recs[e / kWarps].wm[e % kWarps];
        if (wmax > -INFINITY) z += recs[e / kWarps].wz[e % kWarps] * ex2((wmax - m) * rp.c2);
      }
    }
    z = warp_sum(z);
    const bool v = lane < C;
    const int n = v ? recs[lane].s.i0 : 0;
    float th = v ? recs[lane].s.f0 : -INFINITY;
    const bool over = __any_sync(kFull, v && n < 0);
    const int nn = n < 0 ? 0 : n;
    const int incl = warp_inclusive_scan(nn, lane);
    const int all_n = __shfl_sync(kFull, incl, 31);
    if (v) sm.cnt[lane] = static_cast<uint32_t>(incl - nn);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) th = fmaxf(th, __shfl_xor_sync(kFull, th, o));
    if (lane == 0) {
      sm.bi[0] = over ? -1 : all_n;
      sm.bi[1] = 0;   // entries gathered
      sm.bi[3] = -1;  // the cut's value bucket (none: all of the entries)
      sm.bi[4] = -1;  // the draw's index bucket
      sm.bi[5] = 0;   // entries of a resolved bucket
      sm.bf4[0] = th;
      sm.bf4[2] = z;
    }
  }
  unsigned long long* hmass = sm.scan;  // per bucket (kBuckets == kThreads)
  hmass[tid] = 0ull;
  group_sync();
  const int total = sm.bi[0];
  const float thr = sm.bf4[0];
  const float zrow = sm.bf4[2];
  if (total < 0) return false;
  if (!rp.use_p && thr > -INFINITY && weight(thr, m, rp.c2) >= rp.minp) {
    return false;  // min_p alone keeps elements below the lists' bound
  }
  // ---- gather the entries >= thr from the workspace: flat position f of
  // the concatenated lists, four loads in flight per thread, appends
  // aggregated per warp.
  const uint32_t kthr = thr > -INFINITY ? float_key(thr) : 0u;
  const ChunkSlot* wrec = ws_records(P) + static_cast<size_t>(row) * C;
  auto entry_at = [&](int f) {
    int r = 0;  // the last list starting at or before f (C <= 16)
#pragma unroll
    for (int step = kMaxChunks / 2; step > 0; step >>= 1) {
      if (r + step < C && static_cast<int>(sm.cnt[r + step]) <= f) r += step;
    }
    return __ldcg(slot_cands(const_cast<ChunkSlot*>(wrec + r)) + (f - static_cast<int>(sm.cnt[r])));
  };
  for (int f0 = 0; f0 < total; f0 += 4 * kThreads) {
    unsigned long long e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int f = f0 + q * kThreads + tid;
      e[q] = f < total ? entry_at(f) : 0ull;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int f = f0 + q * kThreads + tid;
      const uint32_t kx = static_cast<uint32_t>(e[q] >> 32);
      const bool take = f < total && kx >= kthr;
      const unsigned bal = __ballot_sync(kFull, take);
      int at0 = 0;
      if (lane == 0 && bal != 0u) at0 = atomicAdd(&sm.bi[1], __popc(bal));
      const int at = __shfl_sync(kFull, at0, 0) + __popc(bal & ((1u << lane) - 1u));
      if (take && at < kFinListCap) {
        keys[at] = (static_cast<unsigned long long>(kx) << 32) |
                   static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(e[q]));
      }
    }
  }
  group_sync();
  const int n = sm.bi[1];
  if (n < 1 || n > kFinListCap) return false;
  // ---- per entry: mass, value bucket; per value bucket: mass.  The records
  // are consumed, so their space holds the per-entry arrays.
  unsigned long long* sw = reinterpret_cast<unsigned long long*>(scratch);          // [kFinListCap]
  uint8_t* vb = scratch + kFinListCap * 8;                                          // [kFinListCap]
  uint8_t* in_cut = vb + kFinListCap;  // kept members of the cut bucket              [kFinListCap]
  // A span too small for a finite scale puts every entry in bucket 0 (they
  // are then ranked exactly, or the row takes the exact path).
  const float span = m - thr;
  const float scale =
      (thr > -INFINITY && span > 1e-30f) ? static_cast<float>(kBuckets) / span : 0.0f;
  auto vbucket = [&](float x) {
    const float b = (x - thr) * scale;  // >= 0, non-decreasing in x
    return b < static_cast<float>(kBuckets - 1) ? static_cast<int>(b) : kBuckets - 1;
  };
  for (int t = tid; t < n; t += kThreads) {
    const float x = key_float(static_cast<uint32_t>(keys[t] >> 32));
    const unsigned long long w = mass_fx(weight(x, m, rp.c2));
    const int b = vbucket(x);
    sw[t] = w;
    vb[t] = static_cast<uint8_t>(b);
    in_cut[t] = 0;
    atomicAdd(&hmass[b], w);
  }
  group_sync();
  // ---- the bucket holding the top-p cut: the mass of the buckets above
  // it is below target, with it target or more (one owner).
  int bc = -1;
  unsigned long long rem = 0;
  if (rp.use_p) {
    unsigned long long target = mul_fx(fx40(zrow), rp.p, true);
    if (target < 1ull) target = 1ull;
    const unsigned long long hm = hmass[tid];
    const unsigned long long incl = block_suffix_scan<unsigned long long>(hm, sm.wl, lane, warp);
    unsigned long long all = 0;  // the warps' totals stay in sm.wl after the scan
#pragma unroll 1
    for (int w = 0; w < kWarps; ++w) all += sm.wl[w];
    if (all < target) return false;  // the cut lies below the lists' bound
    const unsigned long long above = incl - hm;
    if (above < target && incl >= target) {
      sm.bi[3] = tid;
      sm.bl[6] = target - above;
    }
    group_sync();
    bc = sm.bi[3];
    rem = sm.bl[6];
  }
  // ---- rank the cut bucket's entries; the first j of them (mass from
  // below rem to rem or more) are kept.
  uint32_t* memb = sm.hlo;  // entry positions, then ranks in sm.hhi
  if (bc >= 0) {
    for (int t0b = warp * 32; t0b < n; t0b += kWarps * 32) {
      const int t = t0b + lane;
      const bool in = t < n && vb[t] == bc;
      const unsigned bal = __ballot_sync(kFull, in);
      int at0 = 0;
      if (lane == 0 && bal != 0u) at0 = atomicAdd(&sm.bi[5], __popc(bal));
      const int at = __shfl_sync(kFull, at0, 0) + __popc(bal & ((1u << lane) - 1u));
      if (in && at < kBuckets) memb[at] = static_cast<uint32_t>(t);
    }
    group_sync();
    const int nb = sm.bi[5];
    if (nb > kBuckets) return false;
    unsigned long long* rw = sm.scan;  // masses in rank order (the bucket masses are consumed)
    int rank = -1;
    if (tid < nb) {
      const unsigned long long ki = keys[memb[tid]];
      rank = 0;
#pragma unroll 1
      for (int q = 0; q < nb; ++q) rank += keys[memb[q]] > ki ? 1 : 0;
      sm.hhi[tid] = static_cast<uint32_t>(rank);
    }
    group_sync();
    if (tid < nb) rw[rank] = sw[memb[tid]];
    if (tid == 0) {
      sm.bi[5] = 0;
      sm.bi[6] = nb;  // kept members (all, should the sums not reach rem)
    }
    group_sync();
    const unsigned long long wr = tid < nb ? rw[tid] : 0ull;
    unsigned long long tot;
    const unsigned long long bef = block_exclusive_scan<unsigned long long>(wr, sm.wl, lane, warp, &tot);
    if (tid < nb && bef < rem && bef + wr >= rem) sm.bi[6] = tid + 1;
    group_sync();
    const int jkeep = sm.bi[6];
    if (tid < nb && static_cast<int>(sm.hhi[tid]) < jkeep) in_cut[memb[tid]] = 1;
    group_sync();
  }
  auto in_s = [&](int t) {
    const int b = vb[t];
    if (bc >= 0 && (b < bc || (b == bc && in_cut[t] == 0))) return false;
    return rp.minp <= 0.0f ||
           weight(key_float(static_cast<uint32_t>(keys[t] >> 32)), m, rp.c2) >= rp.minp;
  };
  // ---- the draw: the mass of S per index bucket, the bucket holding it.
  auto ibucket = [&](int idx) {
    return static_cast<int>((static_cast<unsigned long long>(idx) * kBuckets) /
                            static_cast<unsigned long long>(V));
  };
  unsigned long long* bmass = sm.scan;
  bmass[tid] = 0ull;
  group_sync();
  for (int t = tid; t < n; t += kThreads) {
    if (in_s(t)) {
      atomicAdd(&bmass[ibucket(static_cast<int>(0xffffffffu - static_cast<uint32_t>(keys[t])))],
                sw[t]);
    }
  }
  group_sync();
  const unsigned long long mb = bmass[tid];
  unsigned long long zs;
  const unsigned long long bb = block_exclusive_scan<unsigned long long>(mb, sm.wl, lane, warp, &zs);
  if (zs == 0ull) {
    if (tid == 0) emit(P, row, -1, rp.st | kStNonFinite, wb);
    return true;
  }
  unsigned long long tdraw = mul_fx(zs, rp.u, false);
  if (tdraw >= zs) tdraw = zs - 1ull;
  if (mb > 0ull && tdraw >= bb && tdraw < bb + mb) {
    sm.bi[4] = tid;
    sm.bl[7] = tdraw - bb;
  }
  group_sync();
  const int bstar = sm.bi[4];
  const unsigned long long rest = sm.bl[7];
  // ---- the drawn bucket's entries of S (aggregated appends), then the owner.
  for (int t0b = warp * 32; t0b < n; t0b += kWarps * 32) {
    const int t = t0b + lane;
    bool in = false;
    if (t < n) {
      const int xi = static_cast<int>(0xffffffffu - static_cast<uint32_t>(keys[t]));
      in = ibucket(xi) == bstar && in_s(t);
    }
    const unsigned bal = __ballot_sync(kFull, in);
    int at0 = 0;
    if (lane == 0 && bal != 0u) at0 = atomicAdd(&sm.bi[5], __popc(bal));
    const int at = __shfl_sync(kFull, at0, 0) + __popc(bal & ((1u << lane) - 1u));
    if (in && at < kBuckets) memb[at] = static_cast<uint32_t>(t);
  }
  group_sync();
  const int nm = sm.bi[5];
  if (nm > kBuckets) return false;
  bool owner = false;
  if (tid < nm) {
    const int t = static_cast<int>(memb[tid]);
    const int xi = static_cast<int>(0xffffffffu - static_cast<uint32_t>(keys[t]));
    const unsigned long long w = sw[t];
    unsigned long long cum = 0;
#pragma unroll 1
    for (int q = 0; q < nm; ++q) {
      const int tq = static_cast<int>(memb[q]);
      const int xq = static_cast<int>(0xffffffffu - static_cast<uint32_t>(keys[tq]));
      cum += xq < xi ? sw[tq] : 0ull;
    }
    if (w > 0ull && rest >= cum && rest < cum + w) {
      owner = true;
      emit(P, row, xi, rp.st, wb);
    }
  }
  if (__syncthreads_or(owner) == 0 && tid == 0) emit(P, row, -1, rp.st | kStNonFinite, wb);
  if (q_row != nullptr) {
    const float inv = 1.0f / (static_cast<float>(zs) / kMassScale);
    for (int t = tid; t < n; t += kThreads) {
      if (in_s(t)) {
        const unsigned long long kk = keys[t];
        q_row[0xffffffffu - static_cast<uint32_t>(kk)] =
            weight(key_float(static_cast<uint32_t>(kk >> 32)), m, rp.c2) * inv;
      }
    }
  }
  return true;
}

// ----------------------------------------------------------------- the finish kernel

// One CTA of kThreads threads per row.  Launched as a programmatic dependent
// of the stream kernel: griddepcontrol.wait returns once that grid has
// completed and its writes are visible.
template <bool BF16, int NV, bool VEC>
__global__ void __launch_bounds__(kThreads, 2) finish_kernel(const __grid_constant__ SampleParams P) {
  __shared__ SampleSmem sm;
  __shared__ __align__(8) unsigned long long rec_bar;
  extern __shared__ __align__(128) unsigned char dyn[];
  ChunkSlot* recs = reinterpret_cast<ChunkSlot*>(dyn);
  float* l_val = reinterpret_cast<float*>(dyn + kFinOffList);
  int32_t* l_idx = reinterpret_cast<int32_t*>(dyn + kFinOffList + kFinListCap * 4);
  unsigned long long* table = reinterpret_cast<unsigned long long*>(dyn + kFinOffTable);

  if (static_cast<int>(blockIdx.x) >= P.B) {
    // Fused page allocation and table fill: independent of the stream
    // kernel's output, so these CTAs start at once (no griddepcontrol.wait).
    fill::page_fill_cta<kThreads>(P.fill, reinterpret_cast<int32_t*>(dyn),
                                  static_cast<int>(blockIdx.x) - P.B, P.fill_ctas, threadIdx.x,
                                  []() { __syncthreads(); });
    return;
  }
  const int C = P.chunks;
  const int V = P.V;
  Ctx c;
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  c.crank = 0;
  c.csize = static_cast<uint32_t>(C);
  const int tid = c.tid;
  uint64_t* bar = reinterpret_cast<uint64_t*>(&rec_bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // The row's parameters and write-back coordinates are inputs, not the
  // stream kernel's output: they load before the wait.
  const int row = static_cast<int>(blockIdx.x);
  const RowParams rp = row_params<BF16, NV>(P, row, C);
  const WriteBack wb = load_write_back(P, row);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The parts of the row's records that its kind reads, one bulk copy per
  // (chunk, part), issued by the lanes of warp 0 and completing on rec_bar:
  // the header (summary and warp words) always, the thread maxima for
  // greedy and top-k rows and the count histogram for count-histogram rows
  // (candidate rows read their lists from the workspace directly).
  {
    constexpr uint32_t kHead = static_cast<uint32_t>(offsetof(ChunkSlot, tmax));
    constexpr uint32_t kHistOff = static_cast<uint32_t>(offsetof(ChunkSlot, hist));
    uint32_t len0 = kHead, len1 = 0;  // [0, len0) and [kHistOff, kHistOff + len1)
    if (rp.kind == kKindG || rp.kind == kKindK) {
      len0 = kHistOff;
    } else if (rp.kind == kKindH) {
      len1 = static_cast<uint32_t>(kChunkSlotBytes) - kHistOff;
    }
    if (c.warp == 0) {
      if (c.lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(C) * (len0 + len1));
      __syncwarp();
      if (c.lane < C) {
        const char* src = reinterpret_cast<const char*>(ws_records(P) +
                                                        static_cast<size_t>(row) * C + c.lane);
        unsigned char* dst = dyn + static_cast<size_t>(c.lane) * kChunkSlotBytes;
        bulk_copy_g2s(dst, src, len0, bar);
        if (len1 != 0u) bulk_copy_g2s(dst + kHistOff, src + kHistOff, len1, bar);
      }
    }
  }
  const uint32_t seq = __ldcg(&ws_header(P)->calls);  // the stream kernel's call number
  float* q_row = P.probs_out != nullptr ? P.probs_out + static_cast<size_t>(row) * V : nullptr;
  group_sync();  // the barrier's initialisation is visible to every waiter
  bool landed = mbar_try_wait(bar, 0u);
  if (!landed) {
    const long long t0 = globaltimer_ns();
    while (!(landed = mbar_try_wait(bar, 0u))) {
      if (globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  if (!__syncthreads_and(landed ? 1 : 0)) {
    // The copy did not land: nothing here is trusted, and the shared memory
    // must outlive the copy, so wait for it (bounded) before leaving.
    if (tid == 0) {
      emit(P, row, -1, rp.st | kStTimeout, wb);
      const long long t0 = globaltimer_ns();
      while (!mbar_try_wait(bar, 0u)) {
        if (globaltimer_ns() - t0 > kWaitNs) break;
      }
    }
    return;
  }
  const RowHead head = row_head(recs, C, seq, sm, c);
  if (head.stale) {
    if (tid == 0) emit(P, row, -1, rp.st | kStTimeout, wb);
    return;
  }
  const float m = head.m;
  if (rp.kind == kKindG) {
    // ---- greedy: in the first (chunk, warp) holding the row maximum, the
    // lanes whose thread maximum is m re-read their vectors (one batch of
    // loads) and the first index holding m wins.
    if (head.nan) {
      if (tid == 0) emit(P, row, -1, kStNonFinite | rp.st, wb);
      return;
    }
    const int r = head.first / kWarps, w = head.first % kWarps;
    const unsigned lanes = __ballot_sync(kFull, recs[r].tmax[w * 32 + c.lane] == m);
    const int nl = __popc(lanes);
    int idx = INT_MAX;
    for (int t = tid; t < nl * NV; t += kThreads) {
      const int l = static_cast<int>(__fns(lanes, 0u, t / NV + 1));
      const int e0 = vec_base<BF16, NV>(r, w, l, t % NV);
      uint32_t w4[4];
      load_vec<BF16, NV, VEC>(P, row, e0, w4);
      for_vec<BF16>(w4, e0, [&](float x, int e) {
        if (x == m && e < V) idx = min(idx, e);
      });
    }
    idx = block_min_int(idx, sm.wi, c.lane, c.warp);
    if (tid == 0) {
      const int tok = idx == INT_MAX ? -1 : idx;
      emit(P, row, tok, tok < 0 ? (kStNonFinite | rp.st) : rp.st, wb);
      if (q_row != nullptr && tok >= 0) q_row[tok] = 1.0f;
    }
    return;
  }
  if (head.nan || m == INFINITY || m == -INFINITY) {
    const int est = (m == -INFINITY) ? kStAllNegInf : kStNonFinite;
    if (tid == 0) emit(P, row, -1, est | rp.st, wb);
    return;
  }
  if (rp.kind == kKindP) {
    finish_plain<BF16, NV, VEC>(P, sm, c, recs, row, rp, m, wb, q_row);
    return;
  }
  if (rp.kind == kKindK) {
    if (finish_topk<BF16, NV, VEC>(P, sm, c, recs, l_val, l_idx, row, rp, m, wb, q_row)) return;
    group_sync();
  }
  if (rp.kind == kKindT) {
    if (finish_cand<BF16, NV, VEC>(P, sm, c, dyn, recs, reinterpret_cast<unsigned long long*>(l_val),
                                   row, rp, m, wb, q_row)) {
      return;
    }
    group_sync();
  }
  if constexpr (BF16) {
    if (rp.kind == kKindH) {
      if (finish_hist<NV, VEC>(P, sm, c, recs, table, reinterpret_cast<uint4*>(dyn), row, rp, m,
                               wb, q_row)) {
        return;
      }
      group_sync();
    }
  }
  leader_fallback<BF16>(P, sm, c, row, rp.k, rp.use_p, rp.p, rp.minp, rp.u, m, rp.c2, rp.st,
                        q_row);
}

}  // namespace pkv
