// Finish kernel of the batched sampler: one CTA per row reads the stream
// kernel's records of the row from the workspace and settles the token (see
// sample_common.cuh for the row kinds).
#pragma once

#include "sample_common.cuh"

namespace pkv {

// ----------------------------------------------------------------- histogram finish (H)

// Chunk r counted its elements per 16-bit key over the kHistKeys keys below
// a_r = gather[r].i0, the key of its maximum: h16[r * kHistKeys + d] is the
// count of key a_r - d.  Merged key i (0 = the row maximum, key A - i) has
// count sum_r h_r[i - (A - a_r)]; every element within kHistKeys keys of the
// row maximum is counted in its chunk (a_r <= A).
//
// The finisher settles top-k (by count) and top-p (by fixed-point mass)
// exactly on the merged keys: keys i < is are wholly in the kept set S, the
// first rs members (in index order) of key is are in it too.  It then picks
// the chunk holding the draw from per-chunk masses of S, re-reads that chunk
// into registers and finds the token with one pass of per-vector sums.
// Returns false, having emitted nothing, when a cut lies below the merged
// window; the caller then runs the exact fallback.
template <int NV, bool VEC>
__device__ __forceinline__ bool finish_hist(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                            const uint32_t* hist, unsigned long long* table,
                                            uint4* stage, int row, const RowParams& rp, float m,
                                            float zrow, float* q_row) {
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  const int k = rp.k;
  const bool topk = k < V;
  const uint16_t* h16 = reinterpret_cast<const uint16_t*>(hist);
  const uint32_t A = key16(m);

  // ---- merged counts and fixed-point weights; thread t holds keys 4t .. 4t + 3.
  uint32_t cnt[4] = {0u, 0u, 0u, 0u};
#pragma unroll 1
  for (int r = 0; r < C; ++r) {
    const uint32_t delta = A - static_cast<uint32_t>(sm.gather[r].i0);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t i = static_cast<uint32_t>(4 * tid + jj);
      if (i >= delta) cnt[jj] += h16[r * kHistKeys + (i - delta)];
    }
  }
  unsigned long long wfx[4];
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t i = static_cast<uint32_t>(4 * tid + jj);
    wfx[jj] = cnt[jj] ? mass_fx(weight(key16_float(A - i), m, rp.c2)) : 0ull;
    table[i] = wfx[jj];
  }
  // ---- top-k by count: keys i < ik are wholly in K, key ik keeps rk members.
  int ik = kHistKeys;
  unsigned long long rk = 0;
  if (topk) {
    const uint32_t local = cnt[0] + cnt[1] + cnt[2] + cnt[3];
    uint32_t total;
    const uint32_t before = block_exclusive_scan<uint32_t>(local, sm.wu, lane, warp, &total);
    if (total < static_cast<uint32_t>(k)) return false;  // the k-th value lies below the window
    int cand = INT_MAX;
    uint32_t run = before;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (run < static_cast<uint32_t>(k) && run + cnt[jj] >= static_cast<uint32_t>(k)) {
        cand = 4 * tid + jj;
        sm.bl[0] = static_cast<unsigned long long>(k) - run;  // one owner
      }
      run += cnt[jj];
    }
    ik = block_min_int(cand, sm.wi, lane, warp);
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
      target = static_cast<unsigned long long>(
          ceil(static_cast<double>(zk) * static_cast<double>(rp.p)));
      if (target > zk) target = zk;
    } else {
      target = static_cast<unsigned long long>(
          ceil(static_cast<double>(zrow) * kMassScaleD * static_cast<double>(rp.p)));
      if (zk < target) return false;  // the top-p cut lies below the window
    }
    if (target < 1) target = 1;
    int cand = INT_MAX;
    unsigned long long run = before, rem = 0, wc = 0;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (run < target && run + mk[jj] >= target) {
        cand = 4 * tid + jj;
        rem = target - run;
        wc = wfx[jj];
      }
      run += mk[jj];
    }
    if (cand != INT_MAX) {
      // Members j of the cut key are kept iff run + j * w < target (one owner).
      unsigned long long need = wc == 0 ? ~0ull : (rem + wc - 1) / wc;
      if (cand == ik && need > rk) need = rk;
      sm.bl[1] = need;
    }
    is = block_min_int(cand, sm.wi, lane, warp);
    rs = sm.bl[1];
  }
  if (is >= kHistKeys) return false;  // unreachable when the masses add up
  const unsigned long long wcut = table[is];
  // ---- per-chunk mass of S above the cut key and the cut key's members.
  for (int r = warp; r < C; r += kWarps) {
    const uint32_t delta = A - static_cast<uint32_t>(sm.gather[r].i0);
    unsigned long long part = 0;
    for (int i = lane; i < is; i += 32) {
      if (static_cast<uint32_t>(i) >= delta) part += h16[r * kHistKeys + (i - delta)] * table[i];
    }
    part = warp_sum_u64(part);
    if (lane == 0) {
      sm.cmass[r][0] = part;
      sm.ties[r] = static_cast<uint32_t>(is) >= delta ? h16[r * kHistKeys + (is - delta)] : 0u;
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
    unsigned long long tdraw =
        static_cast<unsigned long long>(static_cast<double>(rp.u) * static_cast<double>(zs));
    if (tdraw >= zs) tdraw = zs - 1;  // zs >= the row maximum's own weight > 0
    const unsigned bal = __ballot_sync(kFull, v && tdraw < incl);
    const int cstar = bal ? __ffs(bal) - 1 : C - 1;
    if (v) sm.cnt[lane] = static_cast<uint32_t>(kept);
    if (lane == cstar) {
      sm.bi[0] = cstar;
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
  // members count, later ones do not.  The histograms are consumed: the
  // chunk is staged over them.
  auto above_and_ties = [&](const uint4 v4, int e0, unsigned long long* a, uint32_t* t) {
    const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
    unsigned long long s = 0;
    uint32_t n = 0;
    for_vec<true>(w4, e0, [&](float x, int e) {
      if (e < V) {
        const uint32_t i = A - key16(x);
        if (i < static_cast<uint32_t>(is)) s += table[i];
        n += i == static_cast<uint32_t>(is) ? 1u : 0u;
      }
    });
    *a = s;
    *t = n;
  };
  stage_own<true, NV, VEC>(P, row, cstar, stage, warp, lane);
  // Per (warp, vector) sums; entry q = warp * NV + j is in index order.
#pragma unroll 1
  for (int j = 0; j < NV; ++j) {
    unsigned long long a;
    uint32_t t;
    above_and_ties(stage[(warp * NV + j) * 32 + lane], vec_base<true, NV>(cstar, warp, lane, j),
                   &a, &t);
    a = warp_sum_u64(a);
    t = __reduce_add_sync(kFull, t);
    if (lane == 0) {
      sm.scan[warp * NV + j] = a;
      sm.hlo[warp * NV + j] = t;
    }
  }
  group_sync();
  if (warp == 0) {
    constexpr int nq = kWarps * NV;
    unsigned long long carry_a = 0;
    uint32_t carry_t = 0;
    int qstar = -1;
    unsigned long long a_before = 0;
    uint32_t t_before = 0;
#pragma unroll 1
    for (int base = 0; base < nq; base += 32) {
      const int q = base + lane;
      const unsigned long long a = q < nq ? sm.scan[q] : 0ull;
      const uint32_t t = q < nq ? sm.hlo[q] : 0u;
      const unsigned long long ai = warp_inclusive_scan(a, lane) + carry_a;
      const uint32_t ti = warp_inclusive_scan(t, lane) + carry_t;
      const unsigned long long pi = ai + wcut * min(static_cast<unsigned long long>(ti),
                                                    static_cast<unsigned long long>(kept_c));
      const unsigned bal = __ballot_sync(kFull, q < nq && tau < pi);
      if (qstar < 0 && bal) {
        const int ls = __ffs(bal) - 1;
        qstar = base + ls;
        a_before = __shfl_sync(kFull, ai - a, ls);
        t_before = __shfl_sync(kFull, ti - t, ls);
      }
      carry_a = __shfl_sync(kFull, ai, 31);
      carry_t = __shfl_sync(kFull, ti, 31);
    }
    if (lane == 0) {
      sm.bi[2] = qstar;
      sm.bl[6] = a_before;
      sm.bi[3] = static_cast<int32_t>(t_before);
    }
  }
  group_sync();
  const int qstar = sm.bi[2];
  if (qstar >= 0 && warp == qstar / NV) {
    const int jstar = qstar % NV;
    const uint4 v4 = stage[(warp * NV + jstar) * 32 + lane];
    const int e0 = vec_base<true, NV>(cstar, warp, lane, jstar);
    unsigned long long a;
    uint32_t t;
    above_and_ties(v4, e0, &a, &t);
    const unsigned long long ai = warp_inclusive_scan(a, lane) + sm.bl[6];
    const uint32_t ti = warp_inclusive_scan(t, lane) + static_cast<uint32_t>(sm.bi[3]);
    const unsigned long long pi =
        ai + wcut * min(static_cast<unsigned long long>(ti), static_cast<unsigned long long>(kept_c));
    const unsigned bal = __ballot_sync(kFull, tau < pi);
    const int ls = bal ? __ffs(bal) - 1 : 31;
    int sel = -1;
    if (lane == ls) {
      // Walk the lane's elements with the mass of S before each.
      unsigned long long above = ai - a;
      uint32_t tc = ti - t;
      int last = -1;
      for_vec_c<true>(v4, e0, [&](float x, int e) {
        if (e < V) {
          const uint32_t i = A - key16(x);
          const unsigned long long pb =
              above + wcut * min(static_cast<unsigned long long>(tc),
                                 static_cast<unsigned long long>(kept_c));
          unsigned long long w = 0;
          if (i < static_cast<uint32_t>(is)) {
            w = table[i];
            above += w;
          } else if (i == static_cast<uint32_t>(is)) {
            w = tc < kept_c ? wcut : 0ull;
            ++tc;
          }
          if (w > 0) {
            last = e;
            if (sel < 0 && tau < pb + w) sel = e;
          }
        }
      });
      if (sel < 0) sel = last;
    }
    const int tok = __shfl_sync(kFull, sel, ls);
    if (lane == 0) emit_token(P, row, tok, tok < 0 ? (rp.st | kStNonFinite) : rp.st);
  }
  if (qstar < 0 && tid == 0) emit_token(P, row, -1, rp.st | kStNonFinite);
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

// ----------------------------------------------------------------- plain finish (P)

// No filter: the draw is over the whole row.  The leader picks the chunk and
// the warp from the CTAs' per-warp masses; that warp re-reads its slice of
// the chunk (one batch of loads) and finds the token.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void leader_finish_plain(const SampleParams& P, SampleSmem& sm,
                                                    const Ctx& c, int row, float u, float m,
                                                    float c2, int st, float* q_row) {
  using L = Layout<BF16>;
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  if (tid == 0) {
    auto wmass = [&](int r, int w) {
      const float mw = sm.gwm[r][w];
      return mw > -INFINITY ? sm.gwz[r][w] * ex2((mw - m) * c2) : 0.0f;
    };
    float zrow = 0.0f;
    for (int r = 0; r < C; ++r) {
      for (int w = 0; w < kWarps; ++w) zrow += wmass(r, w);
    }
    float target = u * zrow;
    if (!(target < zrow)) target = nextafterf(zrow, 0.0f);
    int rstar = -1, wstar = -1, rlast = -1, wlast = -1;
    float tau = 0.0f, cum = 0.0f;
    for (int r = 0; r < C; ++r) {
      for (int w = 0; w < kWarps; ++w) {
        const float mw = wmass(r, w);
        if (rstar < 0 && mw > 0.0f && target < cum + mw) {
          rstar = r;
          wstar = w;
          tau = target - cum;
        }
        if (mw > 0.0f) {
          rlast = r;
          wlast = w;
        }
        cum += mw;
      }
    }
    if (rstar < 0) {
      rstar = rlast;
      wstar = wlast;
      tau = INFINITY;
    }
    sm.bi[0] = rstar;
    sm.bi[1] = wstar;
    sm.bf4[0] = tau;
    sm.bf4[1] = zrow;
  }
  group_sync();
  const int rstar = sm.bi[0];
  const int wstar = sm.bi[1];
  const float tau = sm.bf4[0];
  const float zrow = sm.bf4[1];
  if (warp == wstar && rstar >= 0) {
    uint32_t d[NV][4];
    load_chunk<BF16, NV, VEC>(P, row, rstar, warp, lane, d);
    int found = -1, lastpos = -1;
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int e0 = vec_base<BF16, NV>(rstar, warp, lane, j);
      float sj = 0.0f;
      int lj = -1;
      for_vec<BF16>(d[j], e0, [&](float x, int e) {
        const float w = e < V ? weight(x, m, c2) : 0.0f;
        sj += w;
        if (w > 0.0f) lj = e;
      });
      const unsigned has = __ballot_sync(kFull, lj >= 0);
      if (has != 0u) lastpos = __shfl_sync(kFull, lj, 31 - __clz(has));
      const float incl = warp_inclusive_scan(sj, lane);
      const float tot = __shfl_sync(kFull, incl, 31);
      if (found < 0 && tau < a + tot) {
        const unsigned bal = __ballot_sync(kFull, tau < a + incl);
        const int lx = bal ? __ffs(bal) - 1 : 31;
        int sel = -1;
        if (lane == lx) {
          float run = a + incl - sj;
          for_vec<BF16>(d[j], e0, [&](float x, int e) {
            const float w = e < V ? weight(x, m, c2) : 0.0f;
            run += w;
            if (sel < 0 && w > 0.0f && tau < run) sel = e;
          });
          if (sel < 0) sel = lj;
        }
        found = __shfl_sync(kFull, sel, lx);
        if (found < 0) found = lastpos;
      }
      a += tot;
    }
    if (found < 0) found = lastpos;  // rounding: the warp's last token with mass
    if (lane == 0) emit_token(P, row, found, found < 0 ? (st | kStNonFinite) : st);
  }
  if (rstar < 0 && tid == 0) emit_token(P, row, -1, st | kStNonFinite);
  if (q_row != nullptr) {
    const float inv = 1.0f / zrow;
    for (int r = 0; r < C; ++r) {
      for_chunk<BF16, NV, VEC>(P, row, r, warp, lane, [&](float x, int e) {
        if (e < V) q_row[e] = weight(x, m, c2) * inv;
      });
    }
  }
}

// ----------------------------------------------------------------- the finish kernel

// One CTA of kThreads threads per row.  Launched as a programmatic dependent
// of the stream kernel: griddepcontrol.wait returns once that grid has
// completed and its writes are visible.
template <bool BF16, int NV, bool VEC>
__global__ void __launch_bounds__(kThreads, 2) finish_kernel(const __grid_constant__ SampleParams P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ SampleSmem sm;
  extern __shared__ __align__(128) unsigned char dyn[];
  float* tm = reinterpret_cast<float*>(dyn + kFinOffTm);
  uint32_t* hist = reinterpret_cast<uint32_t*>(dyn + kFinOffHist);
  float* l_val = reinterpret_cast<float*>(dyn + kFinOffList);
  int32_t* l_idx = reinterpret_cast<int32_t*>(dyn + kFinOffList + kListCap * 4);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(dyn + kFinOffCnt);
  unsigned long long* table = reinterpret_cast<unsigned long long*>(dyn + kFinOffTable);

  const int row = blockIdx.x;
  const int C = P.chunks;
  const int V = P.V;
  Ctx c;
  c.tid = threadIdx.x;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  c.crank = 0;
  c.csize = static_cast<uint32_t>(C);
  const int tid = c.tid;
  const ChunkSlot* slots = static_cast<const ChunkSlot*>(P.workspace) + static_cast<size_t>(row) * C;
  // The row's records in one batch of 16-byte asynchronous copies:
  // summaries and per-warp values into sm, thread maxima into tm, count
  // histograms into hist.  The row parameters load meanwhile.
  {
    const char* src = reinterpret_cast<const char*>(slots);
    for (int pc = tid; pc < C * kSlotPieces; pc += kThreads) {
      const int r = pc / kSlotPieces;
      const int off = (pc - r * kSlotPieces) * 16;
      char* dst;
      if (off < kSlotOffWm) {
        dst = reinterpret_cast<char*>(&sm.gather[r]);
      } else if (off < kSlotOffWz) {
        dst = reinterpret_cast<char*>(&sm.gwm[r][0]) + (off - kSlotOffWm);
      } else if (off < kSlotOffTmax) {
        dst = reinterpret_cast<char*>(&sm.gwz[r][0]) + (off - kSlotOffWz);
      } else if (off < kSlotOffHist) {
        dst = reinterpret_cast<char*>(tm + r * kThreads) + (off - kSlotOffTmax);
      } else {
        dst = reinterpret_cast<char*>(hist + r * kHistWords) + (off - kSlotOffHist);
      }
      cp_async16(dst, src + static_cast<size_t>(pc) * 16);
    }
  }
  const RowParams rp = row_params<BF16, NV>(P, row, C);
  float* q_row = P.probs_out != nullptr ? P.probs_out + static_cast<size_t>(row) * V : nullptr;
  cp_async_wait_all();
  group_sync();
  uint32_t flags = 0;
  float m = -INFINITY;
  for (int r = 0; r < C; ++r) {
    flags |= sm.gather[r].u0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) m = fmax_nan(m, sm.gwm[r][w]);
  }
  if (flags & 2u) {
    if (tid == 0) emit_token(P, row, -1, rp.st | kStTimeout);
    return;
  }
  if (rp.kind == kKindG) {
    // ---- greedy: the first (chunk, warp) in index order holding the row
    // maximum; its warp slice is re-read to find the first index.
    if (m != m) {
      if (tid == 0) emit_token(P, row, -1, kStNonFinite | rp.st);
      return;
    }
    int first = INT_MAX;
    for (int i = tid; i < C * kWarps; i += kThreads) {
      if (sm.gwm[i / kWarps][i % kWarps] == m) first = min(first, i);
    }
    first = block_min_int(first, sm.wi, c.lane, c.warp);
    if (c.warp == 0) {
      // One batch of loads for the warp's whole slice, then the first match
      // in index order (vector j, then lane, then element).
      const int r = first / kWarps, w = first % kWarps;
      uint32_t d[NV][4];
      load_chunk<BF16, NV, VEC>(P, row, r, w, c.lane, d);
      int idx = INT_MAX;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        int mine = INT_MAX;
        for_vec<BF16>(d[j], vec_base<BF16, NV>(r, w, c.lane, j), [&](float x, int e) {
          if (x == m && e < V && mine == INT_MAX) mine = e;
        });
        const int jm = __reduce_min_sync(kFull, mine);
        if (idx == INT_MAX) idx = jm;
      }
      if (c.lane == 0) {
        emit_token(P, row, idx, rp.st);
        if (q_row != nullptr) q_row[idx] = 1.0f;
      }
    }
    return;
  }
  if (m != m || m == INFINITY || m == -INFINITY) {
    const int est = (m == -INFINITY) ? kStAllNegInf : kStNonFinite;
    if (tid == 0) emit_token(P, row, -1, est | rp.st);
    return;
  }
  if (rp.kind == kKindK) {
    // ---- top-k.  theta = the k-th largest thread maximum of the row: at
    // least k elements are >= theta, so every element of the top-k is >=
    // theta and lies in a thread whose maximum is >= theta.  Those threads'
    // vectors are re-read (an L2 hit); their elements >= theta form the
    // candidate list, in index order.
    const int nT = C * kThreads;
    // theta: count the thread maxima per 16-bit key below the row maximum
    // (bucket i = key(m) - key; keys beyond 255 share the last bucket) and
    // take the key where the count from the top reaches k.  For bf16 rows
    // this is the exact k-th largest thread maximum when it lies within 256
    // values of the maximum; otherwise (and for fp32 rows) a lower bound on
    // it, which is still valid: at least k thread maxima are >= theta.
    const uint32_t km = key16(m);
    sm.hlo[tid] = 0u;
    group_sync();
    for (int i = tid; i < nT; i += kThreads) {
      const float t = tm[i];
      if (t == t) {
        const uint32_t kt = key16(t);
        atomicAdd(&sm.hlo[kt >= km ? 0u : min(km - kt, 255u)], 1u);
      }
    }
    group_sync();
    {
      // Inclusive prefix from the top: bucket tid counts keys km - tid.
      const uint32_t h = sm.hlo[tid];
      uint32_t tot;
      const uint32_t before = block_exclusive_scan<uint32_t>(h, sm.wu, c.lane, c.warp, &tot);
      if (before < static_cast<uint32_t>(rp.k) && before + h >= static_cast<uint32_t>(rp.k)) {
        sm.bi[1] = tid;
      }
      if (tid == 0 && tot < static_cast<uint32_t>(rp.k)) sm.bi[1] = -1;
    }
    group_sync();
    const int bk = sm.bi[1];
    group_sync();
    // Bucket bk < 255 holds only 16-bit key km - bk: the smallest value with
    // that key (low 16 bits of the 32-bit key cleared) is the exact k-th
    // largest for bf16 and a lower bound for fp32.  Past the last bucket the
    // exact select runs on all thread maxima.
    float theta = -INFINITY;
    if (bk >= 0 && bk < 255) {
      theta = key16_float(km - static_cast<uint32_t>(bk));
    } else if (bk == 255) {
      unsigned long long rk;
      theta = list_select<false>(tm, nT, [](int) { return true; }, [](int) { return 1ull; },
                                 static_cast<unsigned long long>(rp.k), sm, c, &rk);
    }
    // Candidate lanes of each (chunk, warp) pair q = chunk * kWarps + warp;
    // vector (q, j, lane) of a candidate lane has rank
    //   vbase[q] + j * popc(M_q) + popc(M_q below lane)
    // among the candidate vectors, which is index order.
    uint32_t* Mq = reinterpret_cast<uint32_t*>(sm.scan);     // kMaxChunks * kWarps <= 128
    uint32_t* vbase = Mq + kMaxChunks * kWarps;              // ... and their bases
    for (int q = c.warp; q < C * kWarps; q += kWarps) {
      const unsigned mq = __ballot_sync(kFull, tm[q * 32 + c.lane] >= theta);
      if (c.lane == 0) Mq[q] = mq;
    }
    group_sync();
    if (tid == 0) {
      uint32_t acc = 0;
      for (int q = 0; q < C * kWarps; ++q) {
        vbase[q] = acc;
        acc += static_cast<uint32_t>(__popc(Mq[q])) * NV;
      }
      sm.bi[0] = static_cast<int32_t>(acc);
    }
    group_sync();
    const int nvec = sm.bi[0];
    if (nvec <= kMaxCandVecs && theta > -INFINITY) {
      // Each thread takes candidate vectors v = tid + r * kThreads (at most
      // kKeep kept in registers; more are re-read).
      constexpr int kKeep = 4;
      uint32_t keepv[kKeep][4];
      auto decode = [&](int v, uint32_t (&w4)[4]) -> int {
        // The pair q with vbase[q] <= v < vbase[q + 1] (binary search), then
        // the vector j and the candidate lane within it.
        int lo = 0, hi = C * kWarps - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (vbase[mid] <= static_cast<uint32_t>(v)) lo = mid;
          else hi = mid - 1;
        }
        const int q = lo;
        const uint32_t mq = Mq[q];
        const int pc = __popc(mq);
        const int off = v - static_cast<int>(vbase[q]);
        const int j = off / pc;
        const int lane_q = static_cast<int>(__fns(mq, 0u, off % pc + 1));
        const int e0 = vec_base<BF16, NV>(q / kWarps, q % kWarps, lane_q, j);
        load_vec<BF16, NV, VEC>(P, row, e0, w4);
        return e0;
      };
      int keep_e0[kKeep];
      auto count_vec = [&](int v, uint32_t (&w4)[4], int* e0_out) {
        const int e0 = decode(v, w4);
        uint32_t nc = 0;
        for_vec<BF16>(w4, e0, [&](float x, int e) { nc += (e < V && x >= theta) ? 1u : 0u; });
        cnt[v] = nc;
        *e0_out = e0;
      };
#pragma unroll
      for (int r = 0; r < kKeep; ++r) {
        const int v = tid + r * kThreads;
        if (v < nvec) count_vec(v, keepv[r], &keep_e0[r]);
      }
      for (int v = tid + kKeep * kThreads; v < nvec; v += kThreads) {
        uint32_t w4[4];
        int e0;
        count_vec(v, w4, &e0);
      }
      group_sync();
      // Exclusive prefix of the counts in vector order: contiguous segments.
      const int per = (nvec + kThreads - 1) / kThreads;
      const int i0 = min(nvec, tid * per), i1 = min(nvec, i0 + per);
      uint32_t seg = 0;
      for (int i = i0; i < i1; ++i) seg += cnt[i];
      uint32_t total;
      uint32_t run = block_exclusive_scan<uint32_t>(seg, sm.wu, c.lane, c.warp, &total);
      for (int i = i0; i < i1; ++i) {
        const uint32_t t = cnt[i];
        cnt[i] = run;
        run += t;
      }
      group_sync();
      if (total <= static_cast<uint32_t>(kListCap)) {
        auto place = [&](int v, const uint32_t (&w4)[4], int e0) {
          uint32_t pos = cnt[v];
          for_vec<BF16>(w4, e0, [&](float x, int e) {
            if (e < V && x >= theta) {
              l_val[pos] = x;
              l_idx[pos] = e;
              ++pos;
            }
          });
        };
#pragma unroll
        for (int r = 0; r < kKeep; ++r) {
          const int v = tid + r * kThreads;
          if (v < nvec) place(v, keepv[r], keep_e0[r]);
        }
        for (int v = tid + kKeep * kThreads; v < nvec; v += kThreads) {
          uint32_t w4[4];
          const int e0 = decode(v, w4);
          place(v, w4, e0);
        }
        group_sync();
        leader_finish_list(P, sm, c, l_val, l_idx, static_cast<int>(total), row, rp.k, rp.use_p,
                           rp.p, m, rp.c2, rp.u, rp.st, q_row);
        return;
      }
    }
    // Pathological ties or -inf rows: more candidates than the list holds.
  }
  if (rp.kind == kKindP) {
    leader_finish_plain<BF16, NV, VEC>(P, sm, c, row, rp.u, m, rp.c2, rp.st, q_row);
    return;
  }
  if constexpr (BF16) {
    if (rp.kind == kKindH) {
      float zrow = 0.0f;
      if (rp.k == V) {
        for (int r = 0; r < C; ++r) {
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            const float mw = sm.gwm[r][w];
            if (mw > -INFINITY) zrow += sm.gwz[r][w] * ex2((mw - m) * rp.c2);
          }
        }
      }
      if (finish_hist<NV, VEC>(P, sm, c, hist, table, reinterpret_cast<uint4*>(dyn), row, rp, m,
                               zrow, q_row)) {
        return;
      }
    }
  }
  leader_fallback<BF16>(P, sm, c, row, rp.k, rp.use_p, rp.p, rp.u, m, rp.c2, rp.st, q_row);
}

}  // namespace pkv
