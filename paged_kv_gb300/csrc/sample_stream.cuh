// Stream kernel of the batched sampler: persistent CTAs of kGroups groups of
// kThreads threads.  The items (row, chunk) are ranked with the rows in
// falling cost order (build_order) and handed out one at a time from ticket
// counters in the workspace header.  A chunk is kThreads * NV 16-byte
// vectors of one row.  Aligned rows arrive through a
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
  return kGroups * stream_stages<NV>() * stream_stage_bytes<NV>() + kGroups * kWarps * kHistWords * 4;
}

// Reduces one chunk (registers d, the kernel's layout) to its workspace
// record.  All threads of the group call it.  Every warp records its maximum;
// plain rows add the warp's mass, greedy and top-k rows the thread maxima,
// top-p rows a count histogram of the chunk and one of each warp's slice.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void reduce_chunk(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                             uint32_t* hist, ChunkSlot* slot, int row, int chunk,
                                             const RowParams& rp, const uint32_t (&d)[NV][4]) {
  using L = Layout<BF16>;
  constexpr int CHUNK = kThreads * NV * L::VW;
  constexpr int kWarpSpan = 32 * NV * L::VW;
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  const int V = P.V;
  const int cta_begin = chunk * CHUNK;
  const bool has_pad = cta_begin + CHUNK > V;
  const int k = rp.k;
  const float c2 = rp.c2;

  if (P.probs_out != nullptr) {
    float* q_row = P.probs_out + static_cast<size_t>(row) * V;
    for_regs<BF16, NV>(d, chunk, warp, lane, [&](float, int e) {
      if (e < V) q_row[e] = 0.0f;
    });
  }
  const float tmax = regs_max<BF16, NV>(d);
  const float wmax = warp_max_nan(tmax);
  if (lane == 0) slot->wm[warp] = wmax;
  if (tid == 0 && rp.kind != kKindH && rp.kind != kKindT) slot->s = Summary{};

  if (rp.kind == kKindP || rp.kind == kKindT || (rp.kind == kKindH && k == V)) {
    // ---- the warp's mass relative to its maximum (online: each thread
    // relative to its own maximum, then rescaled).  (x - tmax) * c2, not an
    // fma with tmax * c2: for large c2 (T -> 0) the rounding of tmax * c2
    // would move the exponent by whole units.
    float zt = 0.0f;
    if (tmax > -INFINITY) {
      for_regs<BF16, NV>(d, chunk, warp, lane, [&](float x, int) { zt += weight(x, tmax, c2); });
    }
    const float zw = warp_sum(tmax > -INFINITY ? zt * ex2((tmax - wmax) * c2) : 0.0f);
    if (lane == 0) slot->wz[warp] = zw;
  } else if (rp.kind == kKindK || rp.kind == kKindG) {
    // ---- top-k: the thread maxima; the finisher bounds the row's k-th
    // value by the k-th largest of them and re-reads the few threads above.
    // Greedy: the finisher re-reads the threads holding the row maximum.
    slot->tmax[tid] = tmax;
  }
  if (rp.kind == kKindT) {
    // ---- the chunk's candidate list: a bound theta with at least kCandMin
    // thread maxima at or above it, then every element >= theta.  The thread
    // maxima are counted in 256 buckets of 1/8 logit below the chunk maximum
    // (the last one open); theta is the smallest thread maximum in the
    // buckets that first hold kCandMin of them.  The finisher trusts the list
    // for the elements at or above the largest bound of the row's chunks.
    if (lane == 0) sm.wf[warp] = wmax;
    uint32_t* bucket = hist;                  // 256 counts, then the list length
    bucket[tid] = 0u;
    if (tid == 0) bucket[kBuckets] = 0u;
    group_sync();
    float cm = sm.wf[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) cm = fmax_nan(cm, sm.wf[w]);
    const bool finite = cm == cm && cm != INFINITY && cm != -INFINITY;
    int b = kBuckets;  // no bucket
    if (finite && tmax > -INFINITY) {
      const float dist = cm - tmax;  // >= 0
      b = dist < 32.0f ? min(static_cast<int>(dist * 8.0f), kBuckets - 1) : kBuckets - 1;
      atomicAdd(&bucket[b], 1u);
    }
    group_sync();
    {
      const uint32_t h = bucket[tid];
      uint32_t tot;
      const uint32_t before = block_exclusive_scan<uint32_t>(h, sm.wu, lane, warp, &tot);
      if (tid == 0) sm.bi[6] = kBuckets - 1;
      group_sync();
      if (tid < kBuckets - 1 && before < static_cast<uint32_t>(kCandMin) &&
          before + h >= static_cast<uint32_t>(kCandMin)) {
        sm.bi[6] = tid;
      }
      group_sync();
    }
    const int bk = sm.bi[6];
    uint32_t kmin = __reduce_min_sync(kFull, b <= bk ? float_key(tmax) : 0xffffffffu);
    if (lane == 0) sm.wu[warp] = kmin;
    group_sync();
#pragma unroll
    for (int w = 0; w < kWarps; ++w) kmin = min(kmin, sm.wu[w]);
    const float theta = (finite && kmin != 0xffffffffu) ? key_float(kmin) : -INFINITY;
    unsigned long long* cand = slot_cands(slot);
    if (cm == cm) {
      for_regs<BF16, NV>(d, chunk, warp, lane, [&](float x, int e) {
        if (x >= theta && (!has_pad || e < V)) {
          const uint32_t at = atomicAdd(&bucket[kBuckets], 1u);
          if (at < static_cast<uint32_t>(kCandCap)) {
            cand[at] = (static_cast<unsigned long long>(float_key(x)) << 32) |
                       static_cast<unsigned long long>(static_cast<uint32_t>(e));
          }
        }
      });
    }
    group_sync();
    if (tid == 0) {
      const uint32_t n = bucket[kBuckets];
      Summary sm0 = {};
      sm0.f0 = theta;
      sm0.i0 = (cm == cm && n <= static_cast<uint32_t>(kCandCap)) ? static_cast<int32_t>(n) : -1;
      slot->s = sm0;
    }
    // Every thread has read the counts before the group's next item clears them.
    group_sync();
  }
  if constexpr (BF16) {
    if (rp.kind == kKindH) {
      // ---- counts per 16-bit key over the window [a - kHistKeys + 1, a],
      // a the key of the chunk maximum: one histogram per warp (its slice of
      // NV vectors), summed into the chunk's.  hist holds kWarps blocks of
      // kHistWords words.
      if (lane == 0) sm.wf[warp] = wmax;
      uint4* h4 = reinterpret_cast<uint4*>(hist);
      constexpr int kH4 = kWarps * kHistWords / 4;  // 16-byte words of all blocks
#pragma unroll
      for (int k = 0; k < kH4 / kThreads; ++k) h4[tid + k * kThreads] = make_uint4(0u, 0u, 0u, 0u);
      group_sync();
      float cm = sm.wf[0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) cm = fmax_nan(cm, sm.wf[w]);
      const bool finite = cm == cm && cm != INFINITY && cm != -INFINITY;
      const uint32_t a = finite ? key16(cm) : 0u;
      if (finite) {
        for_regs<true, NV>(d, chunk, warp, lane, [&](float x, int e) {
          const uint32_t idx = a - key16(x);
          if (idx < static_cast<uint32_t>(kHistKeys) && (!has_pad || e < V)) {
            atomicAdd(&hist[warp * kHistWords + (idx >> 1)], 1u << ((idx & 1u) * 16u));
          }
        });
      }
      group_sync();
      // Sums of packed counts: a key's chunk count is at most the chunk's
      // length (< 65536), so the 16-bit halves never carry.
      uint32_t s0 = 0u, s1 = 0u;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        s0 += hist[w * kHistWords + 2 * tid];
        s1 += hist[w * kHistWords + 2 * tid + 1];
      }
      reinterpret_cast<uint2*>(slot->hist)[tid] = make_uint2(s0, s1);
      uint4* sh = ws_slice_hist(P, row, chunk);
#pragma unroll
      for (int k = 0; k < kH4 / kThreads; ++k) sh[tid + k * kThreads] = h4[tid + k * kThreads];
      if (tid == 0) {
        Summary s = {};
        s.i0 = static_cast<int32_t>(a);
        slot->s = s;
      }
      // Every warp has read the histograms before the group's next item
      // clears them (there is no group barrier between items otherwise).
      group_sync();
    }
  }
}

// Threads of a stream CTA: kGroups consumer groups of kThreads, then one
// producer warp per group.
constexpr int kStreamThreads = kGroups * (kThreads + 32);

// Batches of up to kOrderRows rows (sample_params.h) are ordered by cost (one
// 16-bit entry per row in shared memory); larger batches go in row order.
constexpr int kOrderPerThread = (kOrderRows + kStreamThreads - 1) / kStreamThreads;

// Cost class of a row's parameters: 0 for the count-histogram, candidate
// and fallback rows (the most work in both kernels), 1 for top-k rows (long
// in the finish kernel), 2 for plain rows (one exp per element in the
// stream kernel), 3 for greedy rows.  Classes 0 and 1 are the finish
// kernel's heavy rows.
template <bool BF16, int NV>
__device__ __forceinline__ int row_cost_class(const RowInputs& in, int V) {
  const int kind = row_params_of<BF16, NV>(in, V).kind;
  return (kind == kKindH || kind == kKindF || kind == kKindT)
             ? 0
             : (kind == kKindK ? 1 : (kind == kKindP ? 2 : 3));
}

// order[0 .. n): the rows the queues hand out, sorted by cost class, stable
// in row index: every row except the light rows below r_early (those are
// streamed as early items, see the kernel).  All threads of the CTA call it;
// it ends with a CTA barrier, after which wsum[kStreamThreads / 32] holds the
// four class counts of the rows placed.  Thread t ranks the `per` rows
// [t * per, (t + 1) * per), per = ceil(B / kStreamThreads) (so every thread
// has work and the parameter loads of all rows are in flight at once): four
// 16-bit class counts packed in a 64-bit word, one CTA-wide exclusive scan.
template <bool BF16, int NV>
__device__ __forceinline__ void build_order(const SampleParams& P, int r_early, uint16_t* order,
                                            unsigned long long* wsum) {
  constexpr int kWarpsAll = kStreamThreads / 32;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int per = (P.B + kStreamThreads - 1) / kStreamThreads;  // <= kOrderPerThread
  const int r0 = t * per;
  RowInputs in[kOrderPerThread];
#pragma unroll
  for (int j = 0; j < kOrderPerThread; ++j) {
    if (j < per && r0 + j < P.B) in[j] = load_row_inputs(P, r0 + j);
  }
  uint32_t cls = 0, placed = 0;
  unsigned long long cnt = 0;
#pragma unroll
  for (int j = 0; j < kOrderPerThread; ++j) {
    const int r = r0 + j;
    if (j < per && r < P.B) {
      const int c = row_cost_class<BF16, NV>(in[j], P.V);
      if (r < r_early && c != 0) continue;  // an early row
      cls |= static_cast<uint32_t>(c) << (2 * j);
      placed |= 1u << j;
      cnt += 1ull << (16 * c);
    }
  }
  unsigned long long incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const unsigned long long v = lane < kWarpsAll ? wsum[lane] : 0ull;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kWarpsAll) wsum[lane] = x - v;
    if (lane == 31) wsum[kWarpsAll] = x;
  }
  __syncthreads();
  const unsigned long long before = wsum[w] + (incl - cnt);
  const unsigned long long total = wsum[kWarpsAll];
  uint32_t pos[4];
  uint32_t base = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    pos[q] = base + static_cast<uint32_t>((before >> (16 * q)) & 0xffffu);
    base += static_cast<uint32_t>((total >> (16 * q)) & 0xffffu);
  }
#pragma unroll
  for (int j = 0; j < kOrderPerThread; ++j) {
    const int r = r0 + j;
    if ((placed >> j) & 1u) {
      const uint32_t c = (cls >> (2 * j)) & 3u;
      const uint32_t at = pos[c]++;
      order[at] = static_cast<uint16_t>(r);
    }
  }
  __syncthreads();
}

// Row and chunk of item rank q: ranks [0, e0) are the early items in row
// order (item e is chunk e % C of row e / C), the others map through the
// cost order when `ordered`.
__device__ __forceinline__ void item_of(int q, int C, int e0, bool ordered, const uint16_t* order,
                                        int* row, int* chunk) {
  if (q < e0) {
    *row = q / C;
    *chunk = q - (q / C) * C;
    return;
  }
  const int r = (q - e0) / C;
  *row = ordered ? static_cast<int>(order[r]) : r;
  *chunk = (q - e0) - r * C;
}

// Items are handed out one at a time from the workspace header's ticket
// counters, so a group that meets an expensive item takes fewer of the
// cheap ones.  The last CTA to finish resets the counters and advances the
// call number, which every record of this call carries (wseq): the finish
// kernel trusts a record only with the current number, so a record a group
// could not fill (a copy that timed out) or left from an earlier call is
// never read as valid.
template <bool BF16, int NV, bool VEC>
__global__ void __launch_bounds__(kStreamThreads, 1)
    stream_kernel(const __grid_constant__ SampleParams P) {
  using L = Layout<BF16>;
  constexpr int CHUNK = kThreads * NV * L::VW;
  constexpr int kStages = stream_stages<NV>();
  constexpr int kStageBytes = stream_stage_bytes<NV>();
  __shared__ SampleSmem smg[kGroups];
  __shared__ __align__(8) unsigned long long full[kGroups][kStages];
  __shared__ __align__(8) unsigned long long empty[kGroups][kStages];
  __shared__ int stage_item[kGroups][kStages];  // rank copied into the stage, -1: no more
  __shared__ int group_item[kGroups];           // rank of the group's item (element-load path)
  __shared__ int early_taken[kGroups];          // 1: the group's stage 0 holds an early item
  __shared__ int lent_seen;                     // 1: group 1 saw group 0's stage 0 land
  __shared__ uint16_t order[kOrderRows];
  __shared__ unsigned long long order_sum[kStreamThreads / 32 + 1];
  extern __shared__ __align__(128) unsigned char dyn[];

  // The finish kernel may be scheduled as soon as our CTAs retire.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const bool producer = threadIdx.x >= kGroups * kThreads;
  const int group = producer ? (threadIdx.x - kGroups * kThreads) / 32 : threadIdx.x / kThreads;
  const int C = P.chunks;
  const int V = P.V;
  const int items = P.B * C;
  WorkspaceHeader* hdr = ws_header(P);
  uint32_t seq = __ldcg(&hdr->calls) + 1u;  // never 0: 0 marks an untrusted record
  if (seq == 0u) seq = 1u;
  unsigned char* ring = dyn + group * kStages * kStageBytes;
  uint64_t* fullb = reinterpret_cast<uint64_t*>(full[group]);
  uint64_t* emptyb = reinterpret_cast<uint64_t*>(empty[group]);
  // Early items (aligned, ordered batches): producer (CTA b, group g) owns
  // item e = 2b + g of the rows [0, early_rows) in row order (chunk e % C of
  // row e / C).  If that row is light (not a count-histogram, candidate or
  // fallback row), its first stage takes the item at the kernel's start:
  // one read of the row's parameters, no ticket and no cost order needed.
  // The queues hand out every other row: the heavy rows first (early range
  // included), then the light rows from early_rows on.
  const bool ordered = P.B <= kOrderRows;
  const int early_rows =
      (VEC && ordered) ? min(P.B, static_cast<int>(gridDim.x) * kGroups / C) : 0;
  const uint32_t early = static_cast<uint32_t>(early_rows * C);  // rank offset of the queues

  // Two queues (aligned rows): ranks [early, early + heavy) are the items of
  // the count-histogram and candidate rows, bound by shared-memory work,
  // ranks [early + heavy, items) the rest, bound by HBM.  Group 0 of a CTA
  // starts on the first queue and group 1 on the second; a group that took
  // no heavy item moves to the heavy queue once its own is empty, so the
  // heavy work overlaps the streaming instead of holding every group at
  // once.  Each producer claims its next tickets before the row order is
  // built, so that the ticket round trip overlaps it.
  uint32_t first_ticket = 0;
  int first_item = -1;  // this producer's early item
  if (VEC && producer && (threadIdx.x & 31) == 0) {
    // full[s]: the producer's arrival (with the copy's bytes) completes it;
    // empty[s]: one arrival per consumer warp once its vectors are loaded.
    // Each producer initialises its own group's barriers (the consumers
    // first use them after the CTA barrier that ends build_order).
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&fullb[s], 1);
      mbar_init(&emptyb[s], kWarps);
    }
    fence_mbar_init();
    const int e = static_cast<int>(blockIdx.x) * kGroups + group;
    if (e < static_cast<int>(early) &&
        row_cost_class<BF16, NV>(load_row_inputs(P, e / C), V) != 0) {
      first_item = e;
      const int r = e / C, ch = e - (e / C) * C;
      const int e0 = ch * CHUNK;
      const uint32_t bytes = static_cast<uint32_t>(max(0, min(CHUNK, V - e0))) * L::ELT;
      const char* src = static_cast<const char*>(P.logits) +
                        (static_cast<size_t>(r) * static_cast<size_t>(P.row_stride) +
                         static_cast<size_t>(e0)) * L::ELT;
      stage_item[group][0] = e;
      mbar_arrive_expect_tx(&fullb[0], bytes);
      for (uint32_t off = 0; off < bytes; off += 16384u) {
        bulk_copy_g2s(ring + off, src + off, min(16384u, bytes - off), &fullb[0]);
      }
    }
    early_taken[group] = first_item >= 0 ? 1 : 0;  // read by the consumers after build_order
    if (group == 0) lent_seen = 0;
    first_ticket = atomicAdd(group == 0 ? &hdr->ticket_heavy : &hdr->ticket,
                             static_cast<uint32_t>(kStages - (first_item >= 0 ? 1 : 0)));
  }
  uint32_t heavy = 0;  // items of class-0 rows, ranked first
  uint32_t queued = static_cast<uint32_t>(items);  // ranks [early, queued) are the queues'
  if (ordered) {
    build_order<BF16, NV>(P, early_rows, order, order_sum);  // ends with a CTA barrier
    const unsigned long long cls = order_sum[kStreamThreads / 32];
    heavy = static_cast<uint32_t>(cls & 0xffffu) * static_cast<uint32_t>(C);
    const uint32_t placed = static_cast<uint32_t>((cls & 0xffffu) + ((cls >> 16) & 0xffffu) +
                                                  ((cls >> 32) & 0xffffu) + (cls >> 48));
    queued = early + placed * static_cast<uint32_t>(C);
  } else {
    __syncthreads();
  }

  if (producer) {
    // ---- producer warp of the group (lane 0): takes a ticket whenever a
    // stage is free, publishes its rank in stage_item and bulk-copies the
    // chunk; past the last item it publishes -1 with a plain arrival.
    if constexpr (VEC) {
      if ((threadIdx.x & 31) == 0) {
        const char* logits = static_cast<const char*>(P.logits);
        int sent = -1, last_copy[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) last_copy[s] = -1;
        int qi = group == 0 ? 0 : 1;  // the queue in use: 0 heavy, 1 the rest
        bool moved = false;           // already moved to the other queue
        bool took_heavy = false;      // has taken items of the heavy queue
        const bool stagger = heavy > 0u;
        const int n0 = first_item >= 0 ? 1 : 0;  // stage 0 already holds the early item
        if (n0 == 1) last_copy[0] = 0;
        for (int n = n0;; ++n) {
          const int s = n % kStages;
          if (n >= kStages) {
            const uint32_t parity = static_cast<uint32_t>(n / kStages - 1) & 1u;
            const long long t0 = globaltimer_ns();
            bool ok = false;
            while (!(ok = mbar_try_wait(&emptyb[s], parity))) {
              if (globaltimer_ns() - t0 > kWaitNs) break;
              __nanosleep(512);  // leave the issue slots to the consumers
            }
            if (!ok) break;  // the consumers stopped: issue nothing more
          } else if (stagger && n > 0) {
            // The count-histogram items start first: the second opening copy
            // of each group waits (bounded) until group 0's first chunk has
            // landed, so that chunk does not share the opening burst with
            // every other stage.
            const long long t0 = globaltimer_ns();
            while (!mbar_try_wait(reinterpret_cast<uint64_t*>(&full[0][0]), 0u)) {
              if (globaltimer_ns() - t0 > kWaitNs) break;
            }
          }
          int q = -1;
          for (;;) {
            const uint32_t t = (!moved && n < kStages)
                                   ? first_ticket + static_cast<uint32_t>(n - n0)
                                   : atomicAdd(qi == 0 ? &hdr->ticket_heavy : &hdr->ticket, 1u);
            const uint32_t lo = qi == 0 ? early : early + heavy;
            const uint32_t len = qi == 0 ? heavy : queued - early - heavy;
            if (t < len) {
              q = static_cast<int>(lo + t);
              took_heavy = took_heavy || qi == 0;
              break;
            }
            // Both queues are empty, or this group did heavy work: light
            // items it took now would wait in its ring behind a heavy one
            // while the other groups drain the light queue.
            if (moved || took_heavy) break;
            moved = true;
            qi ^= 1;
          }
          if (q < 0) {
            stage_item[group][s] = -1;
            mbar_arrive(&fullb[s]);
            sent = n;
            break;
          }
          int r, ch;
          item_of(q, C, static_cast<int>(early), ordered, order, &r, &ch);
          const int e0 = ch * CHUNK;
          // Every chunk starts inside the row (the launch never makes an empty one).
          const uint32_t bytes = static_cast<uint32_t>(max(0, min(CHUNK, V - e0))) * L::ELT;
          const char* src = logits + (static_cast<size_t>(r) * static_cast<size_t>(P.row_stride) +
                                      static_cast<size_t>(e0)) * L::ELT;
          stage_item[group][s] = q;
          mbar_arrive_expect_tx(&fullb[s], bytes);
          for (uint32_t off = 0; off < bytes; off += 16384u) {
            bulk_copy_g2s(ring + s * kStageBytes + off, src + off, min(16384u, bytes - off),
                          &fullb[s]);
          }
          last_copy[s] = n;
        }
        // Before the CTA's shared memory can go away, every issued copy must
        // have landed: wait (bounded) for the last copy of each stage.  The
        // stage that took the final -1 is skipped: its last copy was consumed
        // before that phase began (and a completed later phase would alias
        // the parity).
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
          if (last_copy[s] < 0 || (sent >= 0 && s == sent % kStages)) continue;
          const uint32_t parity = static_cast<uint32_t>(last_copy[s] / kStages) & 1u;
          const long long t0 = globaltimer_ns();
          while (!mbar_try_wait(&fullb[s], parity)) {
            if (globaltimer_ns() - t0 > kWaitNs) break;
          }
        }
      }
    }
  } else {
    // ---- consumers.
    Ctx c;
    c.tid = threadIdx.x % kThreads;
    c.lane = c.tid & 31;
    c.warp = c.tid >> 5;
    c.csize = static_cast<uint32_t>(C);
    SampleSmem& sm = smg[group];
    uint32_t* hist =
        reinterpret_cast<uint32_t*>(dyn + kGroups * kStages * kStageBytes) + group * kWarps * kHistWords;
    ChunkSlot* ws = ws_records(P);
    bool trusted = true;  // this warp has seen every copy land
    // When there is heavy work, group 1 consumes the early item in group 0's
    // first stage (before its own items), and group 0 starts on its first
    // ticketed item, a heavy one: the long items start first while group 0's
    // producer still keeps two stages ahead.  A stage's barriers count its
    // consumers' arrivals, not which group's warps make them.
    bool lend = false;
    if constexpr (VEC) lend = kStages >= 2 && heavy > 0u && early_taken[0] != 0;
    for (int n = 0;; ++n) {
      uint32_t d[NV][4];
      int q;
      // The stage consumed n-th: group sg's item m.
      const int sg = (lend && group == 1 && n == 0) ? 0 : group;
      const int m = lend ? (group == 0 ? n + 1 : (n == 0 ? 0 : n - 1)) : n;
      if constexpr (VEC) {
        // Each warp waits for the stage on its own (bounded), reads the rank,
        // loads its vectors and signals the producer; no group-wide barrier
        // on the data path.  After a timeout the warp still reads the rank
        // (written long before) and goes on, so that the group's barriers
        // stay matched, but its records are marked untrusted.
        const int s = m % kStages;
        const uint32_t parity = static_cast<uint32_t>(m / kStages) & 1u;
        uint64_t* full_s = reinterpret_cast<uint64_t*>(&full[sg][s]);
        if (lend && group == 0 && m == kStages) {
          // The first phase of this stage went to group 1: a parity test for
          // the second is only meaningful once the first has completed.
          const long long t0 = globaltimer_ns();
          while (*static_cast<volatile int*>(&lent_seen) == 0) {
            if (globaltimer_ns() - t0 > kWaitNs) {
              trusted = false;
              break;
            }
          }
        }
        bool ok = mbar_try_wait(full_s, parity);
        if (!ok) {
          const long long t0 = globaltimer_ns();
          while (!(ok = mbar_try_wait(full_s, parity))) {
            if (globaltimer_ns() - t0 > kWaitNs) break;
          }
        }
        if (!ok) trusted = false;
        if (sg != group && ok && c.lane == 0) *static_cast<volatile int*>(&lent_seen) = 1;
        q = *static_cast<volatile int*>(&stage_item[sg][s]);
        if (q < 0) break;
        int row, chunk;
        item_of(q, C, static_cast<int>(early), ordered, order, &row, &chunk);
        const uint4* sv =
            reinterpret_cast<const uint4*>(dyn + (sg * kStages + s) * kStageBytes);
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
        __syncwarp();
        if (c.lane == 0) mbar_arrive(reinterpret_cast<uint64_t*>(&empty[sg][s]));
      } else {
        // Element loads: thread 0 of the group takes the ticket.
        if (c.tid == 0) {
          const uint32_t t = atomicAdd(&hdr->ticket, 1u);
          group_item[group] = t >= static_cast<uint32_t>(items) ? items : static_cast<int>(t);
        }
        group_sync();
        q = group_item[group];
        group_sync();
        if (q >= items) break;
        int row, chunk;
        item_of(q, C, static_cast<int>(early), ordered, order, &row, &chunk);
        load_chunk<BF16, NV, false>(P, row, chunk, c.warp, c.lane, d);
      }
      int row, chunk;
      item_of(q, C, static_cast<int>(early), ordered, order, &row, &chunk);
      c.crank = static_cast<uint32_t>(chunk);
      ChunkSlot* slot = ws + (static_cast<size_t>(row) * C + chunk);
      const RowParams rp = row_params<BF16, NV>(P, row, C);
      reduce_chunk<BF16, NV, VEC>(P, sm, c, hist, slot, row, chunk, rp, d);
      if (c.lane == 0) slot->wseq[c.warp] = trusted ? seq : 0u;
    }
  }
  // ---- the last CTA out resets the counters for the next call (the next
  // kernel on the stream sees them once this grid has completed).
  __syncthreads();
  if (threadIdx.x == 0 && atomicAdd(&hdr->done, 1u) == gridDim.x - 1) {
    hdr->ticket = 0u;
    hdr->ticket_heavy = 0u;
    hdr->done = 0u;
    hdr->calls = seq;
  }
}

}  // namespace pkv
