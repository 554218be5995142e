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
//   * One thread-block cluster of C CTAs per row (grid = C x B).  CTA r of the
//     cluster owns the contiguous slice [r*chunk, (r+1)*chunk) of the row and
//     keeps it in REGISTERS for the whole kernel: the logits are read from HBM
//     exactly once, with 16-byte streaming loads, each warp reading 512
//     contiguous bytes per instruction.  Within a CTA every warp owns a
//     contiguous sub-slice, so index order is (warp, vector j, lane, element).
//   * Every cross-CTA step is a cluster barrier plus reads of the other CTAs'
//     shared memory (DSMEM): row maximum / argmax, radix-select histograms,
//     tie counts and the partial sums of the inverse-CDF scan.  No global
//     scratch memory is used and nothing is sorted.
//   * top-k: radix select (8-bit digits, 2 levels for bf16, 4 for fp32) on an
//     order-preserving integer key with exact integer counts, then the tied
//     elements at the threshold are cut by index (lowest first).
//   * top-p: the same radix select weighted by probability mass.  Masses are
//     accumulated as 2^-40 fixed-point integers, so bucket sums are exact and
//     independent of the order of the shared-memory atomics (deterministic).
//   * inverse CDF: per-warp partial sums -> per-CTA sums exchanged across the
//     cluster -> the CTA, warp, 256-element slab, lane and element where the
//     cumulative mass first exceeds u * Z_S.  The one warp that searches copies
//     its slice to shared memory and walks it with runtime loops, which keeps
//     the register budget of the other phases intact.
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
constexpr float kMassScale = 1099511627776.0f;  // 2^40: fixed-point unit of probability mass

constexpr int kStNonFinite = 1;
constexpr int kStAllNegInf = 2;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStBadUniform = 16;

// Values one CTA publishes for the others to read through DSMEM.  Two copies
// alternate between consecutive cluster phases: a copy is rewritten only after
// the next cluster barrier, which every CTA reaches after finishing its reads.
struct Exchange {
  float f;
  int32_t i;
  uint32_t u;
  uint32_t pad;
  union {
    uint32_t cnt[kBuckets];
    unsigned long long mass[kBuckets];
  } hist;
};

struct SampleSmem {
  Exchange ex[2];
  unsigned long long scan[kBuckets];
  unsigned long long wl[kWarps];
  float wf[kWarps];
  uint32_t wu[kWarps];
  int32_t wi[kWarps];
  float bf[4];
  int32_t bi[4];
  uint32_t bu[4];
  unsigned long long bl[2];
};

// ----------------------------------------------------------------- element access
//
// Thread storage: d[j][c] is 32-bit word c of the thread's j-th 16-byte vector.
// fp32: one element per word; bf16: two per word (low half first).  Element
// index of (j, c, h) = lane_base + j*32*VW + c*EPW + h.

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

// f(x, e) for every element held by the thread, in ascending index order.
template <bool BF16, int NV, typename F>
__device__ __forceinline__ void for_each(const uint32_t (&d)[NV][4], int lane_base, F&& f) {
  using L = Layout<BF16>;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int h = 0; h < L::EPW; ++h) {
        f(elem<BF16>(d[j][c], h), lane_base + j * 32 * L::VW + c * L::EPW + h);
      }
    }
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

// Copies the warp's register slice to shared memory (slab j, lane l at
// s[j*32 + l]) so that one warp can search it with runtime loops.
template <int NV>
__device__ __forceinline__ void dump_slice(const uint32_t (&d)[NV][4], uint4* s, int lane) {
#pragma unroll
  for (int j = 0; j < NV; ++j) s[j * 32 + lane] = make_uint4(d[j][0], d[j][1], d[j][2], d[j][3]);
  __syncwarp();
}

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
      for (int c = 0; c < 4; ++c) {
        if constexpr (BF16) {
          const int e = e0 + 2 * c;
          const uint32_t lo = e < V ? reinterpret_cast<const uint16_t*>(rp)[e] : 0xff80u;
          const uint32_t hi = e + 1 < V ? reinterpret_cast<const uint16_t*>(rp)[e + 1] : 0xff80u;
          d[j][c] = lo | (hi << 16);
        } else {
          const int e = e0 + c;
          d[j][c] = e < V ? reinterpret_cast<const uint32_t*>(rp)[e] : 0xff800000u;
        }
      }
    }
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

// Radix-select step: thread t holds the cluster-wide weight `tot` of bucket t.
// Returns the highest bucket b whose suffix weight S(b) = sum_{t >= b} tot_t
// reaches `rem`, and S(b + 1) (the weight strictly above it) in *above.
template <typename T>
__device__ __forceinline__ int select_bucket(T tot, T rem, SampleSmem& sm, T* above, int tid,
                                             int lane, int warp) {
  const unsigned long long S = block_suffix_scan<unsigned long long>(tot, sm.wl, lane, warp);
  sm.scan[tid] = S;
  int b = block_max_int(S >= rem ? tid : -1, sm.wi, lane, warp);
  if (b < 0) b = 0;  // unreachable: the caller keeps rem <= S(0)
  *above = (b + 1 < kBuckets) ? static_cast<T>(sm.scan[b + 1]) : T(0);
  __syncthreads();
  return b;
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

// ----------------------------------------------------------------- tie cutoff
//
// Among the elements satisfying `member` across the whole cluster, the first
// r in index order are kept.  Returns this CTA's cutoff: its members with
// index < cutoff are the kept ones.  One cluster phase.
template <bool BF16, int NV, typename M>
__device__ __forceinline__ int tie_cutoff(const uint32_t (&d)[NV][4], int lane_base, M&& member,
                                          unsigned long long r, SampleSmem& sm, uint4* s_slice,
                                          int& ph, uint32_t crank, uint32_t csize, int tid,
                                          int lane, int warp) {
  using L = Layout<BF16>;
  uint32_t cnt = 0;
  for_each<BF16>(d, lane_base, [&](float x, int e) { cnt += member(x, e) ? 1u : 0u; });
  const uint32_t wc = __reduce_add_sync(kFull, cnt);
  if (lane == 0) sm.wu[warp] = wc;
  __syncthreads();
  Exchange& ex = sm.ex[ph & 1];
  if (tid == 0) {
    uint32_t s = 0;
    for (int w = 0; w < kWarps; ++w) s += sm.wu[w];
    ex.u = s;
  }
  cluster_sync();
  ++ph;
  if (warp == 0) {
    const uint32_t c = lane < static_cast<int>(csize) ? ld_dsmem_u32(dsmem(&ex.u, lane)) : 0u;
    const uint32_t incl = warp_inclusive_scan(c, lane);
    const uint32_t before = __shfl_sync(kFull, incl - c, crank);
    const uint32_t mine = __shfl_sync(kFull, c, crank);
    if (lane == 0) {
      unsigned long long rl = r > before ? r - before : 0ull;
      if (rl > mine) rl = mine;
      sm.bu[0] = static_cast<uint32_t>(rl);
      sm.bu[1] = mine;
    }
  }
  __syncthreads();
  const uint32_t rl = sm.bu[0];
  const uint32_t mine = sm.bu[1];
  int cut;
  if (rl == 0) {
    cut = INT_MIN;
  } else if (rl >= mine) {
    cut = INT_MAX;
  } else {
    // The warp holding the rl-th member of this CTA.
    uint32_t cum = 0;
    int wstar = kWarps - 1;
    uint32_t rw = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (cum + sm.wu[w] >= rl) {
        wstar = w;
        rw = rl - cum;
        break;
      }
      cum += sm.wu[w];
    }
    if (warp == wstar) {
      dump_slice(d, s_slice, lane);
      uint32_t acc = 0;
      int found = INT_MAX;
#pragma unroll 1
      for (int j = 0; j < NV; ++j) {
        const uint4 v = s_slice[j * 32 + lane];
        const int e0 = lane_base + j * 32 * L::VW;
        uint32_t cj = 0;
        for_vector<BF16>(v, e0, [&](float x, int e) { cj += member(x, e) ? 1u : 0u; });
        const uint32_t incl = warp_inclusive_scan(cj, lane);
        const uint32_t stot = __shfl_sync(kFull, incl, 31);
        if (acc + stot >= rw) {
          const unsigned bal = __ballot_sync(kFull, acc + incl >= rw);
          const int lx = __ffs(bal) - 1;
          int sel = INT_MAX;
          if (lane == lx) {
            uint32_t need = rw - (acc + incl - cj);  // 1-based rank inside this lane's vector
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
      if (lane == 0) sm.bi[0] = found == INT_MAX ? INT_MAX : found + 1;
    }
    __syncthreads();
    cut = sm.bi[0];
  }
  __syncthreads();
  return cut;
}

// ----------------------------------------------------------------- the kernel

template <bool BF16, int NV, bool VEC, bool ALL_GREEDY>
__global__ void __launch_bounds__(kThreads, 2) sample_kernel(const SampleParams P) {
  using L = Layout<BF16>;
  constexpr int NLEV = BF16 ? 2 : 4;  // 8-bit radix levels covering the key
  __shared__ SampleSmem sm;
  __shared__ uint4 s_slice[NV * 32];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const uint32_t csize = cluster_size();
  const int row = blockIdx.y;
  const int V = P.V;
  const int cta_begin = static_cast<int>(crank) * P.cta_chunk;
  const int lane_base = cta_begin + warp * (32 * NV * L::VW) + lane * L::VW;

  uint32_t d[NV][4];
  load_slice<BF16, NV, VEC>(P, row, lane_base, d);

  const bool greedy = ALL_GREEDY || !(P.temperature[row] > 0.0f);

  // ---- phase 1: row maximum (NaN-propagating), argmax for greedy rows.
  float tmax;
  if constexpr (BF16) {
    uint32_t a0 = d[0][0], a1 = d[0][1], a2 = d[0][2], a3 = d[0][3];
#pragma unroll
    for (int j = 1; j < NV; ++j) {
      a0 = bf16x2_max_nan(a0, d[j][0]);
      a1 = bf16x2_max_nan(a1, d[j][1]);
      a2 = bf16x2_max_nan(a2, d[j][2]);
      a3 = bf16x2_max_nan(a3, d[j][3]);
    }
    const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(a0, a1), bf16x2_max_nan(a2, a3));
    tmax = fmax_nan(elem<true>(m2, 0), elem<true>(m2, 1));
  } else {
    float a0 = elem<false>(d[0][0], 0), a1 = elem<false>(d[0][1], 0);
    float a2 = elem<false>(d[0][2], 0), a3 = elem<false>(d[0][3], 0);
#pragma unroll
    for (int j = 1; j < NV; ++j) {
      a0 = fmax_nan(a0, elem<false>(d[j][0], 0));
      a1 = fmax_nan(a1, elem<false>(d[j][1], 0));
      a2 = fmax_nan(a2, elem<false>(d[j][2], 0));
      a3 = fmax_nan(a3, elem<false>(d[j][3], 0));
    }
    tmax = fmax_nan(fmax_nan(a0, a1), fmax_nan(a2, a3));
  }
  int tidx = INT_MAX;
  if (greedy) {
    // Lowest index holding the thread maximum: walk downwards, keep the last hit.
#pragma unroll
    for (int j = NV - 1; j >= 0; --j) {
#pragma unroll
      for (int c = 3; c >= 0; --c) {
#pragma unroll
        for (int h = L::EPW - 1; h >= 0; --h) {
          if (elem<BF16>(d[j][c], h) == tmax) tidx = lane_base + j * 32 * L::VW + c * L::EPW + h;
        }
      }
    }
  }
  const int nan_any = __any_sync(kFull, tmax != tmax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFull, tmax, o);
    const int oi = __shfl_xor_sync(kFull, tidx, o);
    if (ov > tmax || (ov == tmax && oi < tidx)) {
      tmax = ov;
      tidx = oi;
    }
  }
  if (lane == 0) {
    sm.wf[warp] = tmax;
    sm.wi[warp] = tidx;
    sm.wu[warp] = nan_any;
  }
  __syncthreads();
  int ph = 0;
  {
    Exchange& ex = sm.ex[ph & 1];
    if (tid == 0) {
      float v = sm.wf[0];
      int i = sm.wi[0];
      uint32_t n = sm.wu[0];
      for (int w = 1; w < kWarps; ++w) {
        if (sm.wf[w] > v || (sm.wf[w] == v && sm.wi[w] < i)) {
          v = sm.wf[w];
          i = sm.wi[w];
        }
        n |= sm.wu[w];
      }
      ex.f = v;
      ex.i = i;
      ex.u = n;
    }
    cluster_sync();
    ++ph;
    if (warp == 0) {
      float v = -INFINITY;
      int i = INT_MAX;
      uint32_t n = 0;
      if (lane < static_cast<int>(csize)) {
        v = ld_dsmem_f32(dsmem(&ex.f, lane));
        i = static_cast<int>(ld_dsmem_u32(dsmem(&ex.i, lane)));
        n = ld_dsmem_u32(dsmem(&ex.u, lane));
      }
      n = __reduce_or_sync(kFull, n);
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
        sm.bf[0] = v;
        sm.bi[0] = i;
        sm.bu[0] = n;
      }
    }
    __syncthreads();
  }
  const float m = sm.bf[0];
  const int gidx = sm.bi[0];
  const bool nan_row = sm.bu[0] != 0;
  __syncthreads();

  if (greedy) {
    const int tok = nan_row ? -1 : gidx;
    if (crank == 0 && tid == 0) emit_token(P, row, tok, nan_row ? kStNonFinite : 0);
    if (P.probs_out != nullptr) {
      float* q = P.probs_out + static_cast<size_t>(row) * V;
      for_each<BF16>(d, lane_base, [&](float, int e) {
        if (e < V) q[e] = (e == tok) ? 1.0f : 0.0f;
      });
    }
    cluster_sync();
    return;
  }

  if constexpr (!ALL_GREEDY) {
    // ---- parameters (Sampler.prepare's normalisation, applied per row).
    const float T = fmaxf(P.temperature[row], 1e-6f);
    int k = P.top_k != nullptr ? P.top_k[row] : -1;
    if (k < 1 || k >= V) k = V;
    const float p = P.top_p != nullptr ? fminf(fmaxf(P.top_p[row], 1e-6f), 1.0f) : 1.0f;
    float u = P.uniform[row];
    int st = 0;
    if (!(u >= 0.0f && u < 1.0f)) {
      st |= kStBadUniform;
      u = (u != u) ? 0.0f : fminf(fmaxf(u, 0.0f), 0x1.fffffep-1f);
    }
    if (nan_row || m == INFINITY || m == -INFINITY) {
      st = (m == -INFINITY && !nan_row) ? kStAllNegInf : kStNonFinite;
      if (crank == 0 && tid == 0) emit_token(P, row, -1, st);
      if (P.probs_out != nullptr) {
        float* q = P.probs_out + static_cast<size_t>(row) * V;
        for_each<BF16>(d, lane_base, [&](float, int e) {
          if (e < V) q[e] = 0.0f;
        });
      }
      cluster_sync();
      return;
    }
    const float c2 = 1.4426950408889634f / T;  // log2(e) / T

    // ---- top-k: radix select of the k-th key, then the index cutoff of ties.
    float tk = -INFINITY;
    int ck = INT_MAX;
    if (k < V) {
      uint32_t prefix = 0, pmask = 0;
      uint32_t rem = static_cast<uint32_t>(k);
#pragma unroll 1
      for (int lvl = 0; lvl < NLEV; ++lvl) {
        const int shift = 24 - 8 * lvl;
        Exchange& ex = sm.ex[ph & 1];
        ex.hist.cnt[tid] = 0u;
        __syncthreads();
        for_each<BF16>(d, lane_base, [&](float x, int) {
          const uint32_t key = float_key(x);
          if ((key & pmask) == prefix) atomicAdd(&ex.hist.cnt[(key >> shift) & 0xffu], 1u);
        });
        cluster_sync();
        ++ph;
        uint32_t tot = 0;
        for (uint32_t r = 0; r < csize; ++r) tot += ld_dsmem_u32(dsmem(&ex.hist.cnt[tid], r));
        uint32_t above;
        const int b = select_bucket<uint32_t>(tot, rem, sm, &above, tid, lane, warp);
        rem -= above;
        prefix |= static_cast<uint32_t>(b) << shift;
        pmask |= 0xffu << shift;
      }
      if (BF16 && !(prefix & 0x80000000u)) prefix |= 0xffffu;  // bf16 negatives: low bits all ones
      tk = key_float(prefix);
      const float tkv = tk;
      ck = tie_cutoff<BF16>(d, lane_base, [&](float x, int) { return x == tkv; },
                            static_cast<unsigned long long>(rem), sm, s_slice, ph, crank, csize,
                            tid, lane, warp);
    }
    auto in_k = [&](float x, int e) { return x > tk || (x == tk && e < ck); };

    // ---- top-p, first mass-histogram level over K (digit = key bits 31..24).
    const bool use_p = p < 1.0f;
    if (use_p) {
      Exchange& ex = sm.ex[ph & 1];
      ex.hist.mass[tid] = 0ull;
      __syncthreads();
      for_each<BF16>(d, lane_base, [&](float x, int e) {
        if (in_k(x, e)) {
          const float w = ex2((x - m) * c2);
          atomicAdd(&ex.hist.mass[float_key(x) >> 24],
                    static_cast<unsigned long long>(__float2ull_rz(w * kMassScale)));
        }
      });
      cluster_sync();
      ++ph;
    }

    // ---- top-p: mass-weighted radix select inside K, then the tie cutoff.
    float tp = tk;
    int cp = ck;
    if (use_p) {
      uint32_t prefix = 0, pmask = 0;
      unsigned long long rem = 0;
#pragma unroll 1
      for (int lvl = 0; lvl < NLEV; ++lvl) {
        const int shift = 24 - 8 * lvl;
        Exchange* hx = &sm.ex[(ph - 1) & 1];  // level 0 was filled above
        if (lvl > 0) {
          Exchange& ex = sm.ex[ph & 1];
          ex.hist.mass[tid] = 0ull;
          __syncthreads();
          for_each<BF16>(d, lane_base, [&](float x, int e) {
            const uint32_t key = float_key(x);
            if ((key & pmask) == prefix && in_k(x, e)) {
              const float w = ex2((x - m) * c2);
              atomicAdd(&ex.hist.mass[(key >> shift) & 0xffu],
                        static_cast<unsigned long long>(__float2ull_rz(w * kMassScale)));
            }
          });
          cluster_sync();
          ++ph;
          hx = &ex;
        }
        unsigned long long tot = 0;
        for (uint32_t r = 0; r < csize; ++r) tot += ld_dsmem_u64(dsmem(&hx->hist.mass[tid], r));
        if (lvl == 0) {
          // Target: keep while (mass before) < p * Z, Z the exact fixed-point total.
          const unsigned long long z_fx =
              block_suffix_scan<unsigned long long>(tot, sm.wl, lane, warp);
          if (tid == 0) sm.bl[0] = z_fx;
          __syncthreads();
          const double target = static_cast<double>(sm.bl[0]) * static_cast<double>(p);
          rem = static_cast<unsigned long long>(ceil(target));
          if (rem < 1) rem = 1;
          if (rem > sm.bl[0]) rem = sm.bl[0];
          __syncthreads();
        }
        unsigned long long above;
        const int b = select_bucket<unsigned long long>(tot, rem, sm, &above, tid, lane, warp);
        rem -= above;
        prefix |= static_cast<uint32_t>(b) << shift;
        pmask |= 0xffu << shift;
      }
      if (BF16 && !(prefix & 0x80000000u)) prefix |= 0xffffu;
      tp = key_float(prefix);
      // Members of the threshold group share one weight wt: member j (index
      // order) is kept iff above + j * wt < target, i.e. j < ceil(rem / wt).
      const unsigned long long wt =
          static_cast<unsigned long long>(__float2ull_rz(ex2((tp - m) * c2) * kMassScale));
      const unsigned long long rp = wt == 0 ? ~0ull : (rem + wt - 1) / wt;
      const float tpv = tp;
      cp = tie_cutoff<BF16>(d, lane_base, [&](float x, int e) { return x == tpv && in_k(x, e); },
                            rp, sm, s_slice, ph, crank, csize, tid, lane, warp);
      // The cut counted only K members; when both thresholds fall in the same
      // tie group, members past the top-k cutoff are outside K and stay out.
      if (tp == tk && ck < cp) cp = ck;
    }
    auto in_s = [&](float x, int e) { return x > tp || (x == tp && e < cp); };

    // ---- inverse CDF over S in vocab order.
    float ts = 0.0f;
    for_each<BF16>(d, lane_base, [&](float x, int e) {
      if (in_s(x, e)) ts += ex2((x - m) * c2);
    });
    const float wsum = warp_sum(ts);
    if (lane == 0) sm.wf[warp] = wsum;
    __syncthreads();
    {
      Exchange& ex = sm.ex[ph & 1];
      if (tid == 0) {
        float s = 0.0f;
        for (int w = 0; w < kWarps; ++w) s += sm.wf[w];
        ex.f = s;
      }
      cluster_sync();
      ++ph;
      if (warp == 0) {
        const float t = lane < static_cast<int>(csize) ? ld_dsmem_f32(dsmem(&ex.f, lane)) : 0.0f;
        const float cum = warp_inclusive_scan(t, lane);
        const float Z = __shfl_sync(kFull, cum, 31);
        const float target = u * Z;
        const unsigned hit = __ballot_sync(kFull, lane < static_cast<int>(csize) && target < cum);
        int rstar;
        float tloc;
        if (hit != 0) {
          rstar = __ffs(hit) - 1;
          tloc = target - __shfl_sync(kFull, cum - t, rstar);
        } else {
          const unsigned pos = __ballot_sync(kFull, lane < static_cast<int>(csize) && t > 0.0f);
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
    }
    const int rstar = sm.bi[0];
    const float tloc = sm.bf[0];
    const float zs_all = sm.bf[1];
    if (crank == static_cast<uint32_t>(rstar)) {
      // Warp holding the crossing (sequential cumulative over warp sums).
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
        dump_slice(d, s_slice, lane);
        float acc = 0.0f;
        int found = -1;
        int lastpos = -1;
#pragma unroll 1
        for (int j = 0; j < NV; ++j) {
          const uint4 v = s_slice[j * 32 + lane];
          const int e0 = lane_base + j * 32 * L::VW;
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
    if (P.probs_out != nullptr) {
      float* q = P.probs_out + static_cast<size_t>(row) * V;
      const float inv = 1.0f / zs_all;
      for_each<BF16>(d, lane_base, [&](float x, int e) {
        if (e < V) q[e] = in_s(x, e) ? ex2((x - m) * c2) * inv : 0.0f;
      });
    }
    cluster_sync();
  }
}

}  // namespace pkv
