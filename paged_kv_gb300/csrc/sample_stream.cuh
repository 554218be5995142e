// Stream kernel of the batched sampler: persistent CTAs of kGroups groups of
// kThreads threads.  Group g of CTA b works through the items (row, chunk)
// it = b * kGroups + g + n * (gridDim.x * kGroups), n = 0, 1, ...; a chunk is
// kThreads * NV 16-byte vectors of one row.  Aligned rows arrive through a
// per-group ring of kStages shared-memory stages filled by 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier), issued kStages items
// ahead, so the next chunk is in flight while the current one is reduced.
// Each item reduces its chunk, held in registers, to the workspace record
// the finish kernel needs (see sample_common.cuh for the row kinds).
#pragma once

#include "sample_common.cuh"

namespace pkv {

// Ring depth per group: two stages while they fit next to the other group's.
template <int NV>
constexpr int stream_stages() {
  return NV <= 10 ? 2 : 1;
}

template <int NV>
constexpr int stream_stage_bytes() {
  return kThreads * NV * 16;
}

template <int NV>
constexpr int stream_dyn_bytes() {
  return kGroups * stream_stages<NV>() * stream_stage_bytes<NV>() + kGroups * kHistWords * 4;
}

// Reduces one chunk (registers d, the kernel's layout) to its workspace
// record.  All threads of the group call it.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void reduce_chunk(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                             uint32_t* hist, ChunkSlot* slot, int row, int chunk,
                                             const uint32_t (&d)[NV][4]) {
  using L = Layout<BF16>;
  constexpr int CHUNK = kThreads * NV * L::VW;
  constexpr int kWarpSpan = 32 * NV * L::VW;
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int V = P.V;
  const int C = static_cast<int>(c.csize);
  const int cta_begin = chunk * CHUNK;
  const bool has_pad = cta_begin + CHUNK > V;
  const RowParams rp = row_params<BF16, NV>(P, row, C);
  const int k = rp.k;
  const float c2 = rp.c2;

  if (P.probs_out != nullptr) {
    float* q_row = P.probs_out + static_cast<size_t>(row) * V;
    for_regs<BF16, NV>(d, chunk, warp, lane, [&](float, int e) {
      if (e < V) q_row[e] = 0.0f;
    });
  }
  const float tmax = regs_max<BF16, NV>(d);
  Summary mine = {};

  if (rp.kind == kKindG) {
    // ---- greedy: each warp finds its maximum and that value's first index
    // (first vector j, then lane, holding it; then its first element); one
    // barrier combines the warps.
    const float wmax = warp_max_nan(tmax);
    int widx = INT_MAX;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const unsigned mj = __ballot_sync(kFull, vec_max<BF16>(d[j]) == wmax);
      if (widx == INT_MAX && mj != 0u) {  // warp-uniform
        const int L0 = __ffs(mj) - 1;
        int first = INT_MAX;
        if (lane == L0) {
          for_vec<BF16>(d[j], vec_base<BF16, NV>(chunk, warp, lane, j), [&](float x, int e) {
            if (x == wmax && first == INT_MAX) first = e;
          });
        }
        widx = __shfl_sync(kFull, first, L0);
      }
    }
    if (lane == 0) {
      sm.wf[warp] = wmax;
      sm.wi[warp] = widx;
    }
    group_sync();
    float cmax = sm.wf[0];
    int idx = sm.wi[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      const float v = sm.wf[w];
      if (v > cmax || (v == cmax && sm.wi[w] < idx) || v != v) {
        idx = (v != v) ? idx : sm.wi[w];
        cmax = fmax_nan(cmax, v);
      }
    }
    mine.f0 = cmax;
    mine.i0 = idx;
    mine.u0 = cmax != cmax ? 1u : 0u;
  } else if (rp.kind == kKindK) {
    // ---- top-k: candidates >= theta_c, the chunk-local bound.
    const int nfull_cta = max(0, min(kWarps, (V - cta_begin) / kWarpSpan));
    const int kw = (k + nfull_cta - 1) / nfull_cta;
    const bool full = cta_begin + (warp + 1) * kWarpSpan <= V;
    // kw-th largest thread maximum of the warp (bf16 values: the low 16 key
    // bits are 0 for positive and all ones for negative values).
    const uint32_t kth = BF16 ? (warp_kth_largest_key(float_key(tmax) >> 16, kw, 15, 0) << 16)
                              : warp_kth_largest_key(float_key(tmax), kw, 31, 0);
    const float tw = full ? (BF16 ? key16_float(kth >> 16) : key_float(kth)) : INFINITY;
    const float wmax = warp_max_nan(tmax);
    if (lane == 0) {
      sm.wt[warp] = tw;
      sm.wf[warp] = wmax;
    }
    group_sync();
    float theta = INFINITY, cmax = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      theta = fminf(theta, sm.wt[w]);
      cmax = fmax_nan(cmax, sm.wf[w]);
    }
    const bool cnan = cmax != cmax;
    // Candidate bitmask: bit b is element b of the thread (vector b / VW).
    constexpr int kElems = NV * L::VW;
    constexpr int kMaskWords = (kElems + 31) / 32;
    uint32_t mask[kMaskWords];
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) mask[w] = 0u;
    if (tmax >= theta) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int h = 0; h < L::EPW; ++h) {
            const int b = (j * 4 + q) * L::EPW + h;
            if (elem<BF16>(d[j][q], h) >= theta) mask[b >> 5] |= 1u << (b & 31);
          }
        }
      }
      if (has_pad && theta == -INFINITY) {
        // Padding reads as -inf: it is a candidate only when theta is -inf.
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const int e0 = vec_base<BF16, NV>(chunk, warp, lane, j);
#pragma unroll
          for (int b = 0; b < L::VW; ++b) {
            const int bb = j * L::VW + b;
            if (e0 + b >= V) mask[bb >> 5] &= ~(1u << (bb & 31));
          }
        }
      }
    }
    auto totals = [&](uint32_t* wbase, uint32_t* total) -> uint32_t {
      uint32_t cnt = 0;
#pragma unroll
      for (int w = 0; w < kMaskWords; ++w) cnt += __popc(mask[w]);
      const uint32_t wc = __reduce_add_sync(kFull, cnt);
      if (lane == 0) sm.wu[warp] = wc;
      group_sync();
      uint32_t b = 0, t = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) b += sm.wu[w];
        t += sm.wu[w];
      }
      group_sync();
      *wbase = b;
      *total = t;
      return wc;
    };
    uint32_t wbase, total;
    uint32_t wc = totals(&wbase, &total);
    if (total > static_cast<uint32_t>(kListRegion) && !cnan) {
      // Ties (or a loose bound) push the count past the region: keep exactly
      // the chunk's top-k (k <= kListRegion).
      int cloc = INT_MAX;
      const float tloc = cta_select_topk<BF16, NV, VEC>(P, sm, c, row, theta,
                                                        static_cast<unsigned long long>(k), &cloc);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int e0 = vec_base<BF16, NV>(chunk, warp, lane, j);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int h = 0; h < L::EPW; ++h) {
            const int b = (j * 4 + q) * L::EPW + h;
            const int e = e0 + q * L::EPW + h;
            const float x = elem<BF16>(d[j][q], h);
            if (!(x > tloc || (x == tloc && e < cloc))) mask[b >> 5] &= ~(1u << (b & 31));
          }
        }
      }
      wc = totals(&wbase, &total);
    }
    // Write the candidates, in index order, into the record: element (j,
    // lane, b) goes to wbase + (warp's candidates in vectors < j) + (lanes <
    // lane in vector j) + (rank of b in the lane's vector).  The per-vector
    // lane prefixes come from warp scans of packed 10-bit counts (3 per word).
    if (wc != 0) {
      constexpr int kPack = (NV + 2) / 3;
      uint32_t pk[kPack];
#pragma unroll
      for (int w = 0; w < kPack; ++w) pk[w] = 0u;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int b0 = j * L::VW;
        const uint32_t vb = (mask[b0 >> 5] >> (b0 & 31)) & ((1u << L::VW) - 1u);
        pk[j / 3] |= static_cast<uint32_t>(__popc(vb)) << (10 * (j % 3));
      }
      uint32_t ex[kPack], tot[kPack];
#pragma unroll
      for (int w = 0; w < kPack; ++w) {
        const uint32_t incl = warp_inclusive_scan(pk[w], lane);
        ex[w] = incl - pk[w];
        tot[w] = __shfl_sync(kFull, incl, 31);
      }
      uint32_t before_j = wbase;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int b0 = j * L::VW;
        uint32_t bits = (mask[b0 >> 5] >> (b0 & 31)) & ((1u << L::VW) - 1u);
        uint32_t pos = before_j + ((ex[j / 3] >> (10 * (j % 3))) & 0x3ffu);
        const int e0 = vec_base<BF16, NV>(chunk, warp, lane, j);
        while (bits != 0u) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1u;
          const int q = b / L::EPW;
          const uint32_t word =
              q == 0 ? d[j][0] : (q == 1 ? d[j][1] : (q == 2 ? d[j][2] : d[j][3]));
          if (pos < static_cast<uint32_t>(kListRegion)) {
            slot->payload[pos] = __float_as_uint(elem<BF16>(word, b % L::EPW));
            slot->payload[kListRegion + pos] = static_cast<uint32_t>(e0 + b);
          }
          ++pos;
        }
        before_j += (tot[j / 3] >> (10 * (j % 3))) & 0x3ffu;
      }
    }
    mine.f0 = cmax;
    mine.i0 = static_cast<int32_t>(min(total, static_cast<uint32_t>(kListRegion)));
    mine.u0 = cnan ? 1u : 0u;
  } else if (rp.kind == kKindP || (rp.kind == kKindH && k == V)) {
    // ---- chunk max and mass (online: relative to each thread's maximum).
    float zt = 0.0f;
    if (tmax > -INFINITY) {
      // (x - tmax) * c2, not an fma with tmax * c2: for large c2 (T -> 0)
      // the rounding of tmax * c2 would move the exponent by whole units.
      for_regs<BF16, NV>(d, chunk, warp, lane, [&](float x, int) { zt += weight(x, tmax, c2); });
    }
    const float wmax = warp_max_nan(tmax);
    const float zw = warp_sum(tmax > -INFINITY ? zt * ex2((tmax - wmax) * c2) : 0.0f);
    if (lane == 0) {
      sm.wf[warp] = wmax;
      sm.wz[warp] = zw;
    }
    group_sync();
    float cm = -INFINITY, cz = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) cm = fmax_nan(cm, sm.wf[w]);
    if (cm > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (sm.wf[w] > -INFINITY) cz += sm.wz[w] * ex2((sm.wf[w] - cm) * c2);
      }
    }
    mine.f0 = cm;
    mine.f1 = cz;
    mine.u0 = cm != cm ? 1u : 0u;
    if (rp.kind == kKindP && tid < kWarps) {
      slot->wm[tid] = sm.wf[tid];
      slot->wz[tid] = sm.wz[tid];
    }
  } else {
    // ---- H with top-k (no mass needed) and F: chunk max only.
    const float wmax = warp_max_nan(tmax);
    if (lane == 0) sm.wf[warp] = wmax;
    group_sync();
    float cm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) cm = fmax_nan(cm, sm.wf[w]);
    mine.f0 = cm;
    mine.u0 = cm != cm ? 1u : 0u;
  }
  if constexpr (BF16) {
    if (rp.kind == kKindH) {
      // ---- counts per 16-bit key over the window [a - kHistKeys + 1, a].
      const float cm = mine.f0;
      const bool finite = cm == cm && cm != INFINITY && cm != -INFINITY;
      const uint32_t a = finite ? key16(cm) : 0u;
      hist[tid] = 0u;
      hist[tid + kThreads] = 0u;
      group_sync();
      if (finite) {
        for_regs<true, NV>(d, chunk, warp, lane, [&](float x, int e) {
          const uint32_t idx = a - key16(x);
          if (idx < static_cast<uint32_t>(kHistKeys) && (!has_pad || e < V)) {
            atomicAdd(&hist[idx >> 1], 1u << ((idx & 1u) * 16u));
          }
        });
      }
      group_sync();
      mine.i0 = static_cast<int32_t>(a);
      reinterpret_cast<uint2*>(slot->payload)[tid] = make_uint2(hist[2 * tid], hist[2 * tid + 1]);
    }
  }
  if (tid == 0) slot->s = mine;
}

template <bool BF16, int NV, bool VEC>
__global__ void __launch_bounds__(kThreads * kGroups, 1)
    stream_kernel(const __grid_constant__ SampleParams P) {
  using L = Layout<BF16>;
  constexpr int CHUNK = kThreads * NV * L::VW;
  constexpr int kStages = stream_stages<NV>();
  constexpr int kStageBytes = stream_stage_bytes<NV>();
  __shared__ SampleSmem smg[kGroups];
  __shared__ __align__(8) unsigned long long full[kGroups][kStages];
  extern __shared__ __align__(128) unsigned char dyn[];

  // The finish kernel may be scheduled as soon as our CTAs retire.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int group = threadIdx.x / kThreads;
  Ctx c;
  c.tid = threadIdx.x % kThreads;
  c.lane = c.tid & 31;
  c.warp = c.tid >> 5;
  const int C = P.chunks;
  c.csize = static_cast<uint32_t>(C);
  SampleSmem& sm = smg[group];
  unsigned char* ring = dyn + group * kStages * kStageBytes;
  uint32_t* hist =
      reinterpret_cast<uint32_t*>(dyn + kGroups * kStages * kStageBytes) + group * kHistWords;
  uint64_t* bars = reinterpret_cast<uint64_t*>(full[group]);
  const int V = P.V;
  const int items = P.B * C;
  const int G = gridDim.x * kGroups;
  const int gid = blockIdx.x * kGroups + group;
  ChunkSlot* ws = static_cast<ChunkSlot*>(P.workspace);
  const char* logits = static_cast<const char*>(P.logits);

  // Bulk copy of item `it` into stage s: the chunk's bytes up to the row end
  // (V * elt is a multiple of 16 on this path), in pieces of at most 16 KB.
  auto issue = [&](int it, int s) {
    const int r = it / C, ch = it % C;
    const int e0 = ch * CHUNK;
    // Every chunk starts inside the row (the launch never makes an empty one).
    const uint32_t bytes = static_cast<uint32_t>(max(0, min(CHUNK, V - e0))) * L::ELT;
    const char* src = logits + (static_cast<size_t>(r) * static_cast<size_t>(P.row_stride) +
                                static_cast<size_t>(e0)) * L::ELT;
    mbar_arrive_expect_tx(&bars[s], bytes);
    for (uint32_t off = 0; off < bytes; off += 16384u) {
      bulk_copy_g2s(ring + s * kStageBytes + off, src + off, min(16384u, bytes - off), &bars[s]);
    }
  };

  if constexpr (VEC) {
    if (c.tid == 0) {
#pragma unroll
      for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
      fence_mbar_init();
    }
    group_sync();
    if (c.tid == 0) {
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        const int it = gid + s * G;
        if (it < items) issue(it, s);
      }
    }
  }

  // Per stage, the parity of its next completion (thread 0 of the group).
  uint32_t next_parity = 0u;  // bit s
  bool timed_out = false;
  for (int n = 0;; ++n) {
    const int it = gid + n * G;
    if (it >= items) break;
    const int row = it / C, chunk = it % C;
    c.crank = static_cast<uint32_t>(chunk);
    ChunkSlot* slot = ws + it;
    uint32_t d[NV][4];
    if constexpr (VEC) {
      const int s = n % kStages;
      const uint32_t parity = static_cast<uint32_t>(n / kStages) & 1u;
      if (c.tid == 0) {
        const long long t0 = globaltimer_ns();
        bool ok = false;
        while (!(ok = mbar_try_wait(&bars[s], parity))) {
          if (globaltimer_ns() - t0 > kWaitNs) break;
        }
        sm.bi[7] = ok ? 1 : 0;
      }
      group_sync();
      if (sm.bi[7] == 0) {
        // The copy did not arrive: flag the item and stop issuing.
        if (c.tid == 0) {
          Summary bad = {};
          bad.u0 = 2u;
          slot->s = bad;
        }
        timed_out = true;
        break;
      }
      next_parity ^= 1u << s;
      const uint4* sv = reinterpret_cast<const uint4*>(ring + s * kStageBytes);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int e0 = vec_base<BF16, NV>(chunk, c.warp, c.lane, j);
        if (e0 < V) {
          const uint4 v = sv[(c.warp * NV + j) * 32 + c.lane];
          d[j][0] = v.x;
          d[j][1] = v.y;
          d[j][2] = v.z;
          d[j][3] = v.w;
        } else {
          const uint32_t ninf = BF16 ? 0xff80ff80u : 0xff800000u;
          d[j][0] = d[j][1] = d[j][2] = d[j][3] = ninf;
        }
      }
      group_sync();  // the stage is consumed
      if (c.tid == 0) {
        const int next = it + kStages * G;
        if (next < items) {
          fence_proxy_async_smem();
          issue(next, s);
        }
      }
    } else {
      load_chunk<BF16, NV, false>(P, row, chunk, c.warp, c.lane, d);
    }
    reduce_chunk<BF16, NV, VEC>(P, sm, c, hist, slot, row, chunk, d);
  }
  if constexpr (VEC) {
    // After a timeout, copies may still be in flight into this group's ring:
    // wait for them (bounded) before the CTA's shared memory goes away.
    if (timed_out && c.tid == 0) {
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        const long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&bars[s], (next_parity >> s) & 1u)) {
          if (globaltimer_ns() - t0 > kWaitNs) break;
        }
      }
    }
  }
}

}  // namespace pkv
