// Finish kernel of the batched sampler: one CTA per row reads the stream
// kernel's records of the row from the workspace and settles the token (see
// sample_common.cuh for the row kinds).
#pragma once

#include "sample_common.cuh"

namespace pkv {

// ----------------------------------------------------------------- histogram finish (H)

// The leader merges the C count histograms (CTA r counted its elements per
// 16-bit key over the kHistKeys keys below a_r = gather[r].i0, the key of its
// maximum), settles top-k and top-p exactly, picks the chunk holding the draw,
// re-reads it and finds the token.  Returns false, having emitted nothing,
// when a cut lies below the merged window; the caller then runs the exact
// fallback.
template <int NV, bool VEC>
__device__ __forceinline__ bool leader_finish_hist(const SampleParams& P, SampleSmem& sm,
                                                  const Ctx& c, const uint32_t* hist, uint4* stage,
                                                  unsigned long long* table, int row,
                                                int k, bool use_p, float p, float u, float m,
                                                float zrow, float c2, int st, float* q_row) {
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int C = static_cast<int>(c.csize);
  const int V = P.V;
  const bool topk = k < V;
  const uint32_t A = key16(m);
  // Count of CTA r at merged key i (key A - i); 0 above the CTA's maximum.
  auto count_at = [&](int r, uint32_t i) -> uint32_t {
    const uint32_t delta = A - static_cast<uint32_t>(sm.gather[r].i0);
    if (i > A || i < delta) return 0u;
    const uint32_t idx = i - delta;
    return (hist[r * kHistWords + (idx >> 1)] >> ((idx & 1u) * 16u)) & 0xffffu;
  };
  // Merged key i (0 = the row maximum); thread t holds keys 4t .. 4t + 3.
  uint32_t cnt[4];
  unsigned long long wfx[4];
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t i = static_cast<uint32_t>(4 * tid + jj);
    uint32_t n = 0;
    for (int r = 0; r < C; ++r) n += count_at(r, i);
    cnt[jj] = n;
    wfx[jj] = n ? mass_fx(weight(key16_float(A - i), m, c2)) : 0ull;
    table[i] = wfx[jj];
  }
  // ---- top-k by count: keys i < ik are wholly in K, key ik keeps rk members.
  int ik = kHistKeys;
  unsigned long long rk = 0;
  if (topk) {
    const uint32_t local = cnt[0] + cnt[1] + cnt[2] + cnt[3];
    uint32_t total;
    const uint32_t before = block_exclusive_scan<uint32_t>(local, sm.wu, lane, warp, &total);
    if (total < static_cast<uint32_t>(k)) return false;  // k-th value below the window
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
    group_sync();
  }
  unsigned long long mk[4];  // mass of K at each key
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int i = 4 * tid + jj;
    mk[jj] = i < ik ? cnt[jj] * wfx[jj] : (i == ik ? rk * wfx[jj] : 0ull);
  }
  // ---- top-p inside K by mass: keys i < is wholly in S, key is keeps rs.
  int is = ik;
  unsigned long long rs = rk;
  if (use_p) {
    const unsigned long long local = mk[0] + mk[1] + mk[2] + mk[3];
    unsigned long long zk;
    const unsigned long long before =
        block_exclusive_scan<unsigned long long>(local, sm.wl, lane, warp, &zk);
    unsigned long long target;
    if (topk) {
      target =
          static_cast<unsigned long long>(ceil(static_cast<double>(zk) * static_cast<double>(p)));
      if (target > zk) target = zk;
    } else {
      target = static_cast<unsigned long long>(
          ceil(static_cast<double>(zrow) * kMassScaleD * static_cast<double>(p)));
      if (zk < target) return false;  // the top-p cut lies below the window
    }
    if (target < 1) target = 1;
    int cand = INT_MAX;
    unsigned long long run = before;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (run < target && run + mk[jj] >= target) {
        cand = 4 * tid + jj;
        // Members j of the cut key are kept iff run + j * w < target.
        const unsigned long long rem = target - run;
        unsigned long long rp = wfx[jj] == 0 ? ~0ull : (rem + wfx[jj] - 1) / wfx[jj];
        if (cand == ik && rp > rk) rp = rk;
        sm.bl[1] = rp;  // one owner
      }
      run += mk[jj];
    }
    is = block_min_int(cand, sm.wi, lane, warp);
    rs = sm.bl[1];
    group_sync();
  }
  if (is >= kHistKeys) return false;  // unreachable when the masses add up
  // ---- per-chunk masses of S: keys above the cut wholly (warp w sums chunks
  // w, w + 8), then the cut key's members in chunk order (chunks are in index
  // order).
  for (int r = warp; r < C; r += kWarps) {
    unsigned long long part = 0;
    for (int i = lane; i < is; i += 32) {
      part += count_at(r, static_cast<uint32_t>(i)) * table[i];
    }
    part = warp_sum(part);
    if (lane == 0) sm.cmass[r][0] = part;
  }
  group_sync();
  if (tid == 0) {
    const unsigned long long wcut = table[is];
    unsigned long long zs = 0, ties_before = 0;
    for (int r = 0; r < C; ++r) {
      unsigned long long mr = sm.cmass[r][0];
      const uint32_t ties = count_at(r, static_cast<uint32_t>(is));
      unsigned long long kept = 0;
      if (ties_before < rs) kept = min(static_cast<unsigned long long>(ties), rs - ties_before);
      ties_before += ties;
      sm.cnt[r] = static_cast<uint32_t>(kept);
      sm.ties[r] = ties;
      mr += kept * wcut;
      sm.cmass[r][0] = mr;
      zs += mr;
    }
    const unsigned long long tdraw =
        static_cast<unsigned long long>(static_cast<double>(u) * static_cast<double>(zs));
    unsigned long long cum = 0, tau = 0;
    int cstar = -1, clast = -1;
    for (int r = 0; r < C; ++r) {
      const unsigned long long mr = sm.cmass[r][0];
      if (cstar < 0 && mr > 0 && tdraw < cum + mr) {
        cstar = r;
        tau = tdraw - cum;
      }
      if (mr > 0) clast = r;
      cum += mr;
    }
    if (cstar < 0) {
      cstar = clast;
      tau = ~0ull;  // the chunk's last token with mass
    }
    sm.bi[0] = cstar;
    sm.bl[3] = tau;
    sm.bl[5] = zs;
  }
  group_sync();
  const int cstar = sm.bi[0];
  const unsigned long long tau = sm.bl[3];
  const unsigned long long zs = sm.bl[5];
  const uint32_t ks = A - static_cast<uint32_t>(is);  // the cut key
  group_sync();
  // The histograms are consumed: the staging area may overwrite them.
  // Members of the cut key kept in chunk r (staged): all, none, or those
  // with index below the returned cut (the first sm.cnt[r]).
  auto chunk_cut = [&](int r) -> int {
    const uint32_t kept = sm.cnt[r];
    if (kept >= sm.ties[r]) return INT_MAX;
    if (kept == 0) return INT_MIN;
    return staged_search<true, NV, unsigned long long>(
               stage, r,
               [&](float x, int e) { return (e < V && key16(x) == ks) ? 1ull : 0ull; },
               static_cast<unsigned long long>(kept) - 1ull, sm, tid, lane, warp) + 1;
  };
  int tok = -1;
  if (cstar >= 0) {
    stage_chunk<true, NV, VEC>(P, row, cstar, stage, warp, lane);
    const int ecut = chunk_cut(cstar);
    tok = staged_search<true, NV, unsigned long long>(
        stage, cstar,
        [&](float x, int e) {
          const uint32_t i = A - key16(x);  // merged key index; >= is for keys below the cut
          const bool in = e < V && (static_cast<int>(i) < is || (static_cast<int>(i) == is && e < ecut));
          return in ? table[i] : 0ull;
        },
        tau, sm, tid, lane, warp);
  }
  if (tid == 0) emit_token(P, row, tok, tok < 0 ? (st | kStNonFinite) : st);
  if (q_row != nullptr) {
    const float inv = 1.0f / (static_cast<float>(zs) / kMassScale);
    for (int r = 0; r < C; ++r) {
      group_sync();
      stage_chunk<true, NV, VEC>(P, row, r, stage, warp, lane);
      const int ecut = chunk_cut(r);
      for_staged<true, NV>(stage, r, warp, lane, [&](float x, int e) {
        if (e < V) {
          const uint32_t kx = key16(x);
          const bool in = kx > ks || (kx == ks && e < ecut);
          q_row[e] = in ? weight(x, m, c2) * inv : 0.0f;
        }
      });
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
__global__ void __launch_bounds__(kThreads) finish_kernel(const __grid_constant__ SampleParams P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ SampleSmem sm;
  extern __shared__ __align__(128) unsigned char dyn[];
  float* l_val = reinterpret_cast<float*>(dyn);
  int32_t* l_idx = reinterpret_cast<int32_t*>(dyn + kListCap * 4);
  uint32_t* hist = reinterpret_cast<uint32_t*>(dyn);
  uint4* stage = reinterpret_cast<uint4*>(dyn);
  unsigned long long* table =
      reinterpret_cast<unsigned long long*>(dyn + finish_table_offset<NV>());

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
  const RowParams rp = row_params<BF16, NV>(P, row, C);
  float* q_row = P.probs_out != nullptr ? P.probs_out + static_cast<size_t>(row) * V : nullptr;
  // Per-warp maxima of every chunk (NaN-propagating), summaries, flags.
  for (int i = tid; i < C * kWarps; i += kThreads) {
    sm.gwm[i / kWarps][i % kWarps] = slots[i / kWarps].wm[i % kWarps];
    sm.gwz[i / kWarps][i % kWarps] = slots[i / kWarps].wz[i % kWarps];
  }
  if (tid < C) sm.gather[tid] = slots[tid].s;
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
    using L = Layout<BF16>;
    float* tm = reinterpret_cast<float*>(dyn + kFinOffTm);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(dyn + kFinOffCnt);
    const int nT = C * kThreads;
    for (int i = tid; i < nT; i += kThreads) tm[i] = slots[i / kThreads].tmax[i % kThreads];
    group_sync();
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
      for (int r = 0; r < C; ++r) {
        const uint32_t* h = slots[r].hist;
        hist[r * kHistWords + tid] = h[tid];
        hist[r * kHistWords + tid + kThreads] = h[tid + kThreads];
      }
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
      group_sync();
      if (leader_finish_hist<NV, VEC>(P, sm, c, hist, stage, table, row, rp.k, rp.use_p, rp.p,
                                      rp.u, m, zrow, rp.c2, rp.st, q_row)) {
        return;
      }
    }
  }
  leader_fallback<BF16>(P, sm, c, row, rp.k, rp.use_p, rp.p, rp.u, m, rp.c2, rp.st, q_row);
}

}  // namespace pkv
