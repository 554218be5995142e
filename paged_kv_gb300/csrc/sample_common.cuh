// Shared pieces of the batched sampler for sm_103a: constants, the
// per-chunk workspace slot, element access on 16-byte vectors, block helpers
// (one 256-thread group = 8 warps synchronises on its own named barrier),
// the candidate-list selects, the CTA-local top-k, chunk searches and the
// exact fallback over global memory.
//
// Operation ("mini-sglang from Scratch", page "The engine and the sampler",
// section "The sampler": Sampler.sample / sample_torch): greedy rows return
// the argmax (lowest index on ties); other rows are scaled by 1/T, filtered
// top-k first and then top-p on the renormalised top-k distribution (keep a
// token while the mass ranked before it is < p), renormalised, and a token is
// drawn by inverse CDF in ascending vocab index against the supplied uniform.
// Order between equal logits is by ascending index everywhere.
//
// Two kernels (sample_stream.cuh, sample_finish.cuh):
//   * stream: persistent CTAs, two groups of 8 warps each; every group works
//     through its (row, chunk) items, fed by a ring of 1-D bulk copies
//     (cp.async.bulk + mbarrier) from global into shared memory, so the next
//     chunk is in flight while the current one is reduced.  Each item leaves
//     a small record in the workspace: a summary and per-warp maxima, with
//     per-warp masses (plain and top-p rows), the thread maxima (greedy and
//     top-k rows), a count histogram (bf16 top-p rows) or a candidate list
//     (fp32 top-p rows).
//   * finish: one CTA per row (programmatic dependent launch) reads the
//     records of its row and settles the token exactly.
// Row kinds:
//   G  greedy: (max, first index) per chunk.
//   K  top-k with k <= 256: the chunk's thread maxima; the finisher bounds
//      the row's k-th value by the k-th largest of the row's thread maxima
//      and re-reads the few threads at or above it.
//   P  plain (no filter): chunk and per-warp (max, mass); the finisher picks
//      the warp of the draw and re-reads that warp's slice.
//   H  top-p, or top-k with k > 256, on bf16 rows: all elements with one bf16
//      value share one weight, so exact counts per value give exact masses;
//      each chunk counts its elements per value over the 1024 values below
//      its maximum.
//   T  top-p (or min_p) without top-k on fp32 rows: each chunk lists its
//      elements at or above a bound below which at least 64 of its thread
//      maxima lie; the lists hold every element above the largest bound, and
//      when the top-p cut falls there the finisher settles the row from the
//      lists alone (masses per value bucket for the cut and per index bucket
//      for the draw, each resolved exactly inside one bucket).
//   F  whatever the above cannot settle (a cut below the window or the
//      lists; fp32 rows with k > 256): radix passes over the row in global
//      memory.
// No tensor cores (nothing here is a contraction); exp is MUFU.EX2.
#pragma once

#include <climits>
#include <cstddef>
#include <cstdint>

#include "device_common.cuh"
#include "sample_params.h"

namespace pkv {

constexpr int kThreads = 256;                  // threads of one group (and of a finish CTA)
constexpr int kWarps = kThreads / 32;
constexpr int kGroups = 2;                     // groups per stream CTA
constexpr int kBuckets = 256;
constexpr int kMaxChunks = 16;                 // chunks per row
constexpr int kHistKeys = 1024;                // values counted below a chunk's maximum (H rows)
constexpr int kHistWords = kHistKeys / 2;      // two 16-bit counts per word
constexpr int kMaxK = 256;                     // largest k of a K row
static_assert(kHistKeys == 4 * kThreads, "four merged histogram keys per finisher thread");
static_assert(kHistWords == 2 * kThreads, "two histogram words per thread");


// Dynamic shared memory of the finish kernel (offsets 16-byte aligned): the
// parts of the row's records its kind reads, the K rows' candidate list (T
// rows: their gathered sort keys) and the H rows' fixed-point mass per
// merged key.  Once the records are consumed, an H row stages its draw
// slice histograms and a T row its per-entry masses from offset 0.
constexpr int kFinListCap = 2048;
constexpr int kFinRecBytes = kMaxChunks * static_cast<int>(kChunkSlotBytes);
constexpr int kFinOffList = kFinRecBytes;
constexpr int kFinOffTable = kFinOffList + kFinListCap * 8;
constexpr int kFinishDynBytes = kFinOffTable + kHistKeys * 8;
static_assert(kFinRecBytes % 16 == 0, "aligned regions");
static_assert(kThreads * 16 * 16 <= kFinOffTable, "a staged chunk (NV <= 16) below the mass table");
static_assert(kFinListCap * 2 >= kMaxChunks * kThreads, "the thread maxima fit the list region");
static_assert(kFinishDynBytes >= static_cast<int>((64 + 3 * kMaxFillBatch + 1) * 4),
              "a fused page-fill CTA's scan fits the finish kernel's shared memory");
constexpr float kMassScale = 1099511627776.0f;  // 2^40: fixed-point unit of probability mass
constexpr long long kWaitNs = 500000000ll;      // bound of every wait on a bulk copy (0.5 s)

constexpr int kStNonFinite = 1;
constexpr int kStAllNegInf = 2;
constexpr int kStRowOOB = 4;
constexpr int kStColOOB = 8;
constexpr int kStBadUniform = 16;
constexpr int kStTimeout = 64;

enum RowKind { kKindG = 0, kKindK = 1, kKindP = 2, kKindH = 3, kKindF = 4, kKindT = 5 };

// T rows: a chunk's bound leaves at least kCandMin of its thread maxima at
// or above it; its list of (order key, index) entries takes the space of
// the thread maxima and the histogram (kCandCap entries).
constexpr int kCandMin = 64;

// One chunk's summary.
struct __align__(16) Summary {
  float f0;     // T: the chunk's bound (every element at or above it is listed)
  float f1;     // unused
  int32_t i0;   // H: 16-bit key of the chunk maximum (the histogram's anchor); T: list
                // length, -1 when the list overflowed
  uint32_t u0;  // unused
};

// The workspace record of one (row, chunk): written by the stream kernel,
// read by the finish kernel.  Warp w of the chunk owns wm[w] (its maximum,
// NaN if it saw a NaN) and wz[w] (P rows and H rows without top-k: its mass
// relative to wm[w]); thread t owns tmax[t] (K rows: its maximum); H rows
// keep their count histogram in hist.
struct __align__(16) ChunkSlot {
  Summary s;
  float wm[kWarps];
  float wz[kWarps];
  uint32_t wseq[kWarps];  // per warp: the call's record number, 0 when its data is not trusted
  uint32_t pad[kWarps];
  float tmax[kThreads];
  uint32_t hist[kHistWords];
};
// T rows: the candidate list over tmax and hist (contiguous).
static_assert(offsetof(ChunkSlot, hist) == offsetof(ChunkSlot, tmax) + sizeof(float) * kThreads,
              "the candidate list spans tmax and hist");
constexpr int kCandCap = static_cast<int>((sizeof(float) * kThreads + 4 * kHistWords) / 8);
__device__ __forceinline__ unsigned long long* slot_cands(ChunkSlot* s) {
  return reinterpret_cast<unsigned long long*>(s->tmax);
}
__device__ __forceinline__ const unsigned long long* slot_cands(const ChunkSlot* s) {
  return reinterpret_cast<const unsigned long long*>(s->tmax);
}

struct SampleSmem {
  Summary gather[kMaxChunks];
  uint32_t cnt[kMaxChunks];
  uint32_t ties[kMaxChunks];
  unsigned long long cmass[kMaxChunks][kWarps];
  unsigned long long scan[kBuckets];
  uint32_t hlo[kBuckets];  // histograms of the list and fallback selects
  uint32_t hhi[kBuckets];
  unsigned long long wl[kWarps];
  float wf[kWarps];
  uint32_t wu[kWarps];
  int32_t wi[kWarps];
  float wt[kWarps];
  float wz[kWarps];
  int32_t bi[8];
  float bf4[4];
  unsigned long long bl[8];
};

static_assert(sizeof(Summary) == 16, "one 16-byte record");
static_assert(sizeof(ChunkSlot) == kChunkSlotBytes, "workspace record size");
// Byte offsets of the record's parts (the finisher copies them in 16-byte pieces).
static_assert(offsetof(ChunkSlot, tmax) % 16 == 0 && offsetof(ChunkSlot, hist) % 16 == 0 &&
                  kChunkSlotBytes % 16 == 0,
              "records move by 16-byte bulk copies");

__device__ __forceinline__ WorkspaceHeader* ws_header(const SampleParams& P) {
  return static_cast<WorkspaceHeader*>(P.workspace);
}
__device__ __forceinline__ ChunkSlot* ws_records(const SampleParams& P) {
  return reinterpret_cast<ChunkSlot*>(static_cast<char*>(P.workspace) + kRecordsOffset);
}
// Slice histograms of (row, chunk): kWarps blocks of kHistWords words (two
// 16-bit counts each), block w for consumer warp w's slice of the chunk.
static_assert(kSliceHistBytes == static_cast<size_t>(kWarps) * kHistWords * 4,
              "one histogram per consumer warp");
__device__ __forceinline__ uint4* ws_slice_hist(const SampleParams& P, int row, int chunk) {
  char* base = reinterpret_cast<char*>(ws_records(P) + static_cast<size_t>(P.B) * P.chunks);
  return reinterpret_cast<uint4*>(base + (static_cast<size_t>(row) * P.chunks + chunk) * kSliceHistBytes);
}

// Barrier of the calling thread's group of kThreads threads (named barrier
// 1 + group); a finish CTA is one group.
__device__ __forceinline__ void group_sync() {
  asm volatile("bar.sync %0, %1;" :: "r"(1 + (threadIdx.x / kThreads)), "n"(kThreads)
               : "memory");
}

// ----------------------------------------------------------------- element access

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
__device__ __forceinline__ void for_vec(const uint32_t (&w)[4], int e0, F&& f) {
  using L = Layout<BF16>;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int h = 0; h < L::EPW; ++h) f(elem<BF16>(w[q], h), e0 + q * L::EPW + h);
  }
}

// for_vec as a loop that is not unrolled (one copy of f's code), for code
// that runs once per row: there instruction fetch, not issue, sets the pace.
template <bool BF16, typename F>
__device__ __forceinline__ void for_vec_c(const uint4 v, int e0, F&& f) {
  using L = Layout<BF16>;
#pragma unroll 1
  for (int t = 0; t < L::VW; ++t) {
    const int q = t / L::EPW;
    const uint32_t w = q < 2 ? (q == 0 ? v.x : v.y) : (q == 2 ? v.z : v.w);
    f(elem<BF16>(w, t % L::EPW), e0 + t);
  }
}

struct Ctx {
  int tid, lane, warp;  // within the group
  uint32_t crank;       // chunk of the row
  uint32_t csize;       // chunks per row
};

// Row index of the first element of vector j of (warp, lane) in chunk `chunk`.
template <bool BF16, int NV>
__device__ __forceinline__ int vec_base(int chunk, int warp, int lane, int j) {
  using L = Layout<BF16>;
  return chunk * (kThreads * NV * L::VW) + ((warp * NV + j) * 32 + lane) * L::VW;
}

// f(x, e) for every element of the thread's registers (chunk `chunk`).
template <bool BF16, int NV, typename F>
__device__ __forceinline__ void for_regs(const uint32_t (&d)[NV][4], int chunk, int warp,
                                         int lane, F&& f) {
#pragma unroll
  for (int j = 0; j < NV; ++j) for_vec<BF16>(d[j], vec_base<BF16, NV>(chunk, warp, lane, j), f);
}

// Loads the thread's NV vectors of chunk `chunk` of `row`.  Elements past V
// read as -inf.  VEC: the row start and V * elt are 16-byte aligned, so a
// whole vector loads with one instruction; otherwise (and for the vector that
// straddles V) elements load one by one.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void load_chunk(const SampleParams& P, int row, int chunk, int warp,
                                           int lane, uint32_t (&d)[NV][4]) {
  using L = Layout<BF16>;
  const char* rp = static_cast<const char*>(P.logits) +
                   static_cast<size_t>(row) * static_cast<size_t>(P.row_stride) * L::ELT;
  const int V = P.V;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e0 = vec_base<BF16, NV>(chunk, warp, lane, j);
    if (VEC && e0 + L::VW <= V) {
      const uint4 v = ld_stream_v4(rp + static_cast<size_t>(e0) * L::ELT);
      d[j][0] = v.x;
      d[j][1] = v.y;
      d[j][2] = v.z;
      d[j][3] = v.w;
    } else {
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

// NaN-propagating maximum of the thread's registers.
template <bool BF16, int NV>
__device__ __forceinline__ float regs_max(const uint32_t (&d)[NV][4]) {
  // Four independent chains (one per word of a vector) keep the dependency
  // chain short.
  if constexpr (BF16) {
    uint32_t m2[4] = {d[0][0], d[0][1], d[0][2], d[0][3]};
#pragma unroll
    for (int j = 1; j < NV; ++j) {
#pragma unroll
      for (int q = 0; q < 4; ++q) m2[q] = bf16x2_max_nan(m2[q], d[j][q]);
    }
    const uint32_t r = bf16x2_max_nan(bf16x2_max_nan(m2[0], m2[1]), bf16x2_max_nan(m2[2], m2[3]));
    return fmax_nan(elem<true>(r, 0), elem<true>(r, 1));
  } else {
    float m[4] = {__uint_as_float(d[0][0]), __uint_as_float(d[0][1]), __uint_as_float(d[0][2]),
                  __uint_as_float(d[0][3])};
#pragma unroll
    for (int j = 1; j < NV; ++j) {
#pragma unroll
      for (int q = 0; q < 4; ++q) m[q] = fmax_nan(m[q], __uint_as_float(d[j][q]));
    }
    return fmax_nan(fmax_nan(m[0], m[1]), fmax_nan(m[2], m[3]));
  }
}

// 16-bit order-preserving key of a bf16 value held as a float (-0 folded).
__device__ __forceinline__ uint32_t key16(float x) { return float_key(x) >> 16; }

__device__ __forceinline__ float key16_float(uint32_t k) { return key_float(k << 16); }

// Weight of logit x relative to the row maximum m: 2^((x - m) * log2(e) / T).
// The one formula used wherever two results must agree to the last bit.
__device__ __forceinline__ float weight(float x, float m, float c2) {
  return ex2(__fmul_rn(__fsub_rn(x, m), c2));
}

// Fixed-point arithmetic without FP64 or 64-bit float<->integer conversion
// instructions (on this GPU both run at a few hundred cycles each).

// floor(x * 2^40) for a finite x in [0, 2^23), by shifting its significand.
__device__ __forceinline__ unsigned long long fx40(float x) {
  const uint32_t b = __float_as_uint(x);
  const int e = static_cast<int>((b >> 23) & 0xffu);
  if (e == 0 || (b >> 31)) return 0ull;  // zero, subnormal (below 2^-126) or negative
  if (e >= 127 + 23) return ~0ull;        // outside the domain (not reached for weights)
  const unsigned long long mnt = static_cast<unsigned long long>((b & 0x7fffffu) | 0x800000u);
  const int sh = e - 127 - 23 + 40;      // x * 2^40 = mnt * 2^sh
  if (sh >= 0) return mnt << sh;
  return sh > -32 ? (mnt >> -sh) : 0ull;
}

// The fixed-point mass of a weight w in [0, 1]: floor(w * 2^40).
__device__ __forceinline__ unsigned long long mass_fx(float w) { return fx40(w); }

// ceil(z * f) (up = true) or floor(z * f) for z < 2^60 and a finite f in
// [0, 1], exactly: f = mnt * 2^-s with a 24-bit mnt, the product in 128 bits.
__device__ __forceinline__ unsigned long long mul_fx(unsigned long long z, float f, bool up) {
  const uint32_t b = __float_as_uint(f);
  const int e = static_cast<int>((b >> 23) & 0xffu);
  if (e == 0 || (b >> 31) || z == 0) return 0ull;
  const unsigned long long mnt = static_cast<unsigned long long>((b & 0x7fffffu) | 0x800000u);
  const int s = 127 + 23 - e;  // f = mnt * 2^-s, s >= 23 for f <= 1
  const unsigned long long lo = z * mnt;
  const unsigned long long hi = __umul64hi(z, mnt);
  if (s >= 64) {
    // z * f < 2^60 * 2^-40: the quotient is hi >> (s - 64) (s < 128 here).
    const int t = s - 64;
    const unsigned long long q = t < 64 ? (hi >> t) : 0ull;
    const bool frac = lo != 0 || (t < 64 ? (hi & ((1ull << t) - 1ull)) != 0 : hi != 0);
    return q + ((up && frac) ? 1ull : 0ull);
  }
  const unsigned long long q = (hi << (64 - s)) | (lo >> s);
  const bool frac = (lo & ((1ull << s) - 1ull)) != 0;
  return q + ((up && frac) ? 1ull : 0ull);
}

// ceil(rem / w) for w > 0 and a quotient at most `bound` (< 2^21), by
// bisection on j * w >= rem (integer multiplies only).
__device__ __forceinline__ unsigned long long ceil_div_small(unsigned long long rem,
                                                             unsigned long long w,
                                                             unsigned long long bound) {
  unsigned long long lo = 0, hi = bound;
  while (lo < hi) {
    const unsigned long long mid = (lo + hi) >> 1;
    if (mid * w >= rem) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// ----------------------------------------------------------------- block helpers

// These run once per row in the finish paths, where instruction fetch sets
// the pace: their loops stay rolled (one copy of the body's code).

template <typename T>
__device__ __forceinline__ T block_suffix_scan(T v, T* s_w, int lane, int warp) {
  v = warp_suffix_scan(v, lane);
  if (lane == 0) s_w[warp] = v;
  group_sync();
  T add = 0;
#pragma unroll 1
  for (int w = warp + 1; w < kWarps; ++w) add += s_w[w];
  group_sync();
  return v + add;
}

// Exclusive prefix over threads in tid order; *total receives the block sum.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* s_w, int lane, int warp, T* total) {
  const T incl = warp_inclusive_scan(v, lane);
  if (lane == 31) s_w[warp] = incl;
  group_sync();
  T before = 0, all = 0;
#pragma unroll 1
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += s_w[w];
    all += s_w[w];
  }
  group_sync();
  *total = all;
  return before + incl - v;
}

template <typename T>
__device__ __forceinline__ T block_sum(T v, T* s_w, int lane, int warp) {
  v = warp_sum(v);
  if (lane == 0) s_w[warp] = v;
  group_sync();
  T r = 0;
#pragma unroll 1
  for (int w = 0; w < kWarps; ++w) r += s_w[w];
  group_sync();
  return r;
}

__device__ __forceinline__ int block_max_int(int v, int32_t* s_w, int lane, int warp) {
  v = __reduce_max_sync(kFull, v);
  if (lane == 0) s_w[warp] = v;
  group_sync();
  int r = s_w[0];
#pragma unroll 1
  for (int w = 1; w < kWarps; ++w) r = max(r, s_w[w]);
  group_sync();
  return r;
}

__device__ __forceinline__ int block_min_int(int v, int32_t* s_w, int lane, int warp) {
  v = __reduce_min_sync(kFull, v);
  if (lane == 0) s_w[warp] = v;
  group_sync();
  int r = s_w[0];
#pragma unroll 1
  for (int w = 1; w < kWarps; ++w) r = min(r, s_w[w]);
  group_sync();
  return r;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(kFull, v, o));
  return v;
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
  group_sync();
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

// ----------------------------------------------------------------- chunk search
//
// These re-read a chunk from global memory (an L2 hit: the chunk was just
// streamed) one vector at a time, so they hold no register copy of it.

// Loads vector j of (warp, lane) in chunk `chunk` of `row` (see load_chunk).
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void load_vec(const SampleParams& P, int row, int e0,
                                         uint32_t (&w)[4]) {
  using L = Layout<BF16>;
  const char* rp = static_cast<const char*>(P.logits) +
                   static_cast<size_t>(row) * static_cast<size_t>(P.row_stride) * L::ELT;
  const int V = P.V;
  if (VEC && e0 + L::VW <= V) {
    const uint4 v = *reinterpret_cast<const uint4*>(rp + static_cast<size_t>(e0) * L::ELT);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (BF16) {
        const int e = e0 + 2 * q;
        const uint32_t lo = e < V ? reinterpret_cast<const uint16_t*>(rp)[e] : 0xff80u;
        const uint32_t hi = e + 1 < V ? reinterpret_cast<const uint16_t*>(rp)[e + 1] : 0xff80u;
        w[q] = lo | (hi << 16);
      } else {
        const int e = e0 + q;
        w[q] = e < V ? reinterpret_cast<const uint32_t*>(rp)[e] : 0xff800000u;
      }
    }
  }
}

// Stages this thread's NV vectors of chunk `chunk` of `row` in shared memory,
// in the register layout of load_chunk: vector j of (warp, lane) at
// sv[(warp * NV + j) * 32 + lane].  Vectors inside an aligned row move by
// 16-byte asynchronous copies, the rest by element loads (-inf past V).  On
// return the thread's own vectors are in place (no barrier: each thread
// reads back only what it staged).  A loop, not unrolled: the finisher runs
// it once per row, so its code size matters more than its issue rate.
template <bool BF16, int NV, bool VEC>
__device__ __forceinline__ void stage_own(const SampleParams& P, int row, int chunk, uint4* sv,
                                          int warp, int lane) {
  using L = Layout<BF16>;
  const char* rp = static_cast<const char*>(P.logits) +
                   static_cast<size_t>(row) * static_cast<size_t>(P.row_stride) * L::ELT;
  const int V = P.V;
#pragma unroll 1
  for (int j = 0; j < NV; ++j) {
    const int e0 = vec_base<BF16, NV>(chunk, warp, lane, j);
    uint4* dst = sv + (warp * NV + j) * 32 + lane;
    if (VEC && e0 + L::VW <= V) {
      cp_async16(dst, rp + static_cast<size_t>(e0) * L::ELT);
    } else {
      uint32_t w[4];
      load_vec<BF16, NV, false>(P, row, e0, w);
      *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  cp_async_wait_all();
}

// ----------------------------------------------------------------- list selects
//
// The leader's list holds n entries (value, row index) in ascending index
// order.  These run in one CTA with __syncthreads only.

// Radix select over a list of n entries with 32-bit keys key_of(i): the key
// t such that the weight of entries with key > t is < target <= the weight
// with key >= t.  weight_of(i) is 1 (count) or a fixed-point mass; entries
// with keep(i) false weigh nothing.  Returns t and the weight still needed
// from the entries equal to t in *rem.  Only the key bits on which the kept
// entries differ are examined, 8 at a time.  Runs on one group.
template <bool MASS, typename KeyOf, typename K, typename W>
__device__ __forceinline__ uint32_t list_select_key(KeyOf&& key_of, int n, K&& keep, W&& weight_of,
                                                    unsigned long long target, SampleSmem& sm,
                                                    const Ctx& c, unsigned long long* rem_out) {
  uint32_t kand = 0xffffffffu, kor = 0u;
  for (int i = c.tid; i < n; i += kThreads) {
    if (keep(i)) {
      const uint32_t k = key_of(i);
      kand &= k;
      kor |= k;
    }
  }
  kand = __reduce_and_sync(kFull, kand);
  kor = __reduce_or_sync(kFull, kor);
  if (c.lane == 0) {
    sm.wu[c.warp] = kand;
    sm.wi[c.warp] = static_cast<int32_t>(kor);
  }
  group_sync();
  uint32_t a = 0xffffffffu, o = 0u;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    a &= sm.wu[w];
    o |= static_cast<uint32_t>(sm.wi[w]);
  }
  unsigned long long rem = target;
  const uint32_t diff = a ^ o;  // bits on which the kept keys differ
  if (diff == 0u) {
    group_sync();
    *rem_out = rem;
    return a;
  }
  const int top = 31 - __clz(diff);
  const int bottom = __ffs(diff) - 1;
  // Bits above `top` and below `bottom` are the same in every kept key.
  uint32_t prefix = a & (top == 31 ? 0u : (0xffffffffu << (top + 1)));
  prefix |= a & ((1u << bottom) - 1u);
  for (int hi = top; hi >= bottom; hi -= 8) {
    const int lo = max(hi - 7, bottom);
    const uint32_t dmask = (1u << (hi - lo + 1)) - 1u;
    const uint32_t amask = hi == 31 ? 0u : (0xffffffffu << (hi + 1));  // bits above the digit
    sm.hlo[c.tid] = 0u;
    if constexpr (MASS) sm.hhi[c.tid] = 0u;
    group_sync();
    for (int i = c.tid; i < n; i += kThreads) {
      if (!keep(i)) continue;
      const uint32_t key = key_of(i);
      if ((key & amask) != (prefix & amask)) continue;
      const uint32_t dg = (key >> lo) & dmask;
      if constexpr (MASS) {
        atomic_add_u64_split(&sm.hlo[dg], &sm.hhi[dg], weight_of(i));
      } else {
        atomicAdd(&sm.hlo[dg], 1u);
      }
    }
    group_sync();
    const unsigned long long tot =
        MASS ? ((static_cast<unsigned long long>(sm.hhi[c.tid]) << 32) | sm.hlo[c.tid])
             : static_cast<unsigned long long>(sm.hlo[c.tid]);
    // Suffix sums S(t) over buckets; the bucket b with S(b + 1) < rem <= S(b).
    const unsigned long long sw = warp_suffix_scan(tot, c.lane);
    if (c.lane == 0) sm.wl[c.warp] = sw;
    group_sync();
    unsigned long long S = sw;
    for (int w = c.warp + 1; w < kWarps; ++w) S += sm.wl[w];
    if (S >= rem && S - tot < rem) {
      sm.bi[4] = c.tid;
      sm.bl[6] = S - tot;
    }
    group_sync();
    const int b = sm.bi[4];
    rem -= sm.bl[6];
    prefix |= static_cast<uint32_t>(b) << lo;
  }
  group_sync();
  *rem_out = rem;
  return prefix;
}

// list_select_key over the order keys of float values val[0 .. n): returns
// the value of the selected key.
template <bool MASS, typename K, typename W>
__device__ __forceinline__ float list_select(const float* val, int n, K&& keep, W&& weight_of,
                                             unsigned long long target, SampleSmem& sm,
                                             const Ctx& c, unsigned long long* rem_out) {
  return key_float(list_select_key<MASS>([&](int i) { return float_key(val[i]); }, n, keep,
                                         weight_of, target, sm, c, rem_out));
}

// ----------------------------------------------------------------- exact fallback (F)
//
// The leader alone settles the row by radix passes over the row in global
// memory (elements read one by one; used only when the fast kinds cannot).
// Same decisions as the list and histogram paths: 2^-40 fixed-point masses,
// ties by index.

template <bool BF16>
__device__ __forceinline__ float load_elem(const SampleParams& P, int row, int e) {
  const char* rp = static_cast<const char*>(P.logits) +
                   static_cast<size_t>(row) * static_cast<size_t>(P.row_stride) * (BF16 ? 2 : 4);
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(rp)[e]) << 16);
  } else {
    return reinterpret_cast<const float*>(rp)[e];
  }
}

// Among the elements of the row with member(x, e), the position after the
// r-th in index order (INT_MAX if there are fewer than r; r >= 1).
template <bool BF16, typename M>
__device__ __forceinline__ int row_tie_cut(const SampleParams& P, int row, M&& member,
                                           unsigned long long r, SampleSmem& sm, const Ctx& c) {
  const int V = P.V;
  const int per = (V + kThreads - 1) / kThreads;
  const int i0 = min(V, c.tid * per);
  const int i1 = min(V, i0 + per);
  unsigned long long cnt = 0;
  for (int e = i0; e < i1; ++e) cnt += member(load_elem<BF16>(P, row, e), e) ? 1ull : 0ull;
  unsigned long long total;
  const unsigned long long before =
      block_exclusive_scan<unsigned long long>(cnt, sm.wl, c.lane, c.warp, &total);
  if (c.tid == 0) sm.bi[3] = INT_MAX;
  group_sync();
  if (r <= total && before < r && r <= before + cnt) {
    unsigned long long need = r - before;
    for (int e = i0; e < i1; ++e) {
      if (member(load_elem<BF16>(P, row, e), e) && --need == 0) {
        sm.bi[3] = e + 1;
        break;
      }
    }
  }
  group_sync();
  const int cut = sm.bi[3];
  group_sync();
  return cut;
}

// Radix select over the row: the key t with W(key > t) < target <= W(key >= t),
// W the sum of wfx(x, e) over elements with keep(x, e).  *rem receives target
// - W(key > t).
template <bool BF16, bool MASS, typename K, typename W>
__device__ __forceinline__ float row_select(const SampleParams& P, int row, K&& keep, W&& wfx,
                                            unsigned long long target, SampleSmem& sm,
                                            const Ctx& c, unsigned long long* rem_out) {
  const int V = P.V;
  uint32_t prefix = 0, pmask = 0;
  unsigned long long rem = target;
  for (int lvl = 0; lvl < 4; ++lvl) {
    const int shift = 24 - 8 * lvl;
    sm.hlo[c.tid] = 0u;
    sm.hhi[c.tid] = 0u;
    group_sync();
    for (int e = c.tid; e < V; e += kThreads) {
      const float x = load_elem<BF16>(P, row, e);
      if (!keep(x, e)) continue;
      const uint32_t key = float_key(x);
      if ((key & pmask) != prefix) continue;
      const uint32_t dg = (key >> shift) & 0xffu;
      if constexpr (MASS) {
        atomic_add_u64_split(&sm.hlo[dg], &sm.hhi[dg], wfx(x, e));
      } else {
        atomicAdd(&sm.hlo[dg], 1u);
      }
    }
    group_sync();
    const unsigned long long tot =
        MASS ? ((static_cast<unsigned long long>(sm.hhi[c.tid]) << 32) | sm.hlo[c.tid])
             : static_cast<unsigned long long>(sm.hlo[c.tid]);
    unsigned long long above;
    const int b = select_bucket(tot, rem, sm, &above, c.tid, c.lane, c.warp);
    rem -= above;
    prefix |= static_cast<uint32_t>(b) << shift;
    pmask |= 0xffu << shift;
  }
  *rem_out = rem;
  return key_float(prefix);
}

template <bool BF16>
__device__ __noinline__ void leader_fallback(const SampleParams& P, SampleSmem& sm, const Ctx& c,
                                             int row, int k, bool use_p, float p, float minp,
                                             float u, float m, float c2, int st, float* q_row) {
  const int V = P.V;
  const int tid = c.tid, lane = c.lane, warp = c.warp;
  // ---- top-k: the k-th key by count, ties cut by index.
  float tk = -INFINITY;
  int ck = INT_MAX;
  if (k < V) {
    unsigned long long rk;
    tk = row_select<BF16, false>(P, row, [](float, int) { return true; },
                                 [](float, int) { return 1ull; },
                                 static_cast<unsigned long long>(k), sm, c, &rk);
    const float tkv = tk;
    ck = row_tie_cut<BF16>(P, row, [&](float x, int) { return x == tkv; }, rk, sm, c);
  }
  const float tkf = tk;
  const int ckf = ck;
  auto in_k = [&](float x, int e) { return x > tkf || (x == tkf && e < ckf); };
  auto wfx = [&](float x, int) { return mass_fx(weight(x, m, c2)); };
  // ---- top-p inside K: mass select on fixed-point weights.
  float tp = tk;
  int cp = ck;
  if (use_p) {
    unsigned long long z = 0;
    for (int e = tid; e < V; e += kThreads) {
      const float x = load_elem<BF16>(P, row, e);
      if (in_k(x, e)) z += wfx(x, e);
    }
    z = block_sum<unsigned long long>(z, sm.wl, lane, warp);
    unsigned long long target = mul_fx(z, p, true);
    if (target < 1) target = 1;
    if (target > z) target = z;
    unsigned long long rem;
    tp = row_select<BF16, true>(P, row, in_k, wfx, target, sm, c, &rem);
    const unsigned long long wt = mass_fx(weight(tp, m, c2));
    const unsigned long long rp = wt == 0 ? ~0ull : ceil_div_small(rem, wt, 1ull << 21);
    const float tpv = tp;
    cp = row_tie_cut<BF16>(P, row, [&](float x, int e) { return x == tpv && in_k(x, e); }, rp, sm,
                           c);
    if (tp == tk && ck < cp) cp = ck;
  }
  const float tpf = tp;
  const int cpf = cp;
  // min_p: a token stays when its probability is at least minp times the
  // largest one, weight(x) = 2^((x - m) * c2) >= minp (the row maximum m has
  // weight 1, so the set never empties).
  auto in_s = [&](float x, int e) {
    return in_k(x, e) && (x > tpf || (x == tpf && e < cpf)) &&
           (minp <= 0.0f || weight(x, m, c2) >= minp);
  };
  // ---- draw in index order over contiguous segments.
  const int per = (V + kThreads - 1) / kThreads;
  const int i0 = min(V, tid * per);
  const int i1 = min(V, i0 + per);
  unsigned long long seg = 0;
  int last = -1;
  for (int e = i0; e < i1; ++e) {
    const float x = load_elem<BF16>(P, row, e);
    if (in_s(x, e)) {
      const unsigned long long w = wfx(x, e);
      seg += w;
      if (w > 0) last = e;
    }
  }
  unsigned long long zs;
  const unsigned long long before =
      block_exclusive_scan<unsigned long long>(seg, sm.wl, lane, warp, &zs);
  const unsigned long long tdraw = mul_fx(zs, u, false);
  const int lastpos = block_max_int(last, sm.wi, lane, warp);
  if (tid == 0) sm.bi[2] = lastpos;
  group_sync();
  if (seg > 0 && tdraw >= before && tdraw < before + seg) {
    unsigned long long run = before;
    int sel = last;
    for (int e = i0; e < i1; ++e) {
      const float x = load_elem<BF16>(P, row, e);
      if (in_s(x, e)) {
        run += wfx(x, e);
        if (tdraw < run) {
          sel = e;
          break;
        }
      }
    }
    sm.bi[2] = sel;
  }
  group_sync();
  const int tok = sm.bi[2];
  if (tid == 0) emit_token(P, row, tok, tok < 0 ? (st | kStNonFinite) : st);
  if (q_row != nullptr) {
    const float inv = 1.0f / (static_cast<float>(zs) / kMassScale);
    for (int e = tid; e < V; e += kThreads) {
      const float x = load_elem<BF16>(P, row, e);
      q_row[e] = in_s(x, e) ? weight(x, m, c2) * inv : 0.0f;
    }
  }
}

// ----------------------------------------------------------------- row parameters

// Sampler.prepare's normalisation of one row, and the row's kind (the same
// decision in both kernels).
struct RowParams {
  float T, p, u, c2;
  float minp;  // 0 when min_p is off, else in (0, 1]
  int k;     // V when top-k is off
  int st;    // status bits found so far (a bad uniform)
  int kind;
  bool use_p;
};

// A row's raw parameters.  All five loads are issued at once (none depends
// on another), so a thread that ranks several rows pays one round trip.
struct RowInputs {
  float t, p, u, mp;
  int k;
};

__device__ __forceinline__ RowInputs load_row_inputs(const SampleParams& P, int row) {
  RowInputs in;
  in.t = P.temperature != nullptr ? P.temperature[row] : 0.0f;
  in.k = P.top_k != nullptr ? P.top_k[row] : -1;
  in.p = P.top_p != nullptr ? P.top_p[row] : 1.0f;
  in.u = P.uniform != nullptr ? P.uniform[row] : 0.0f;
  in.mp = P.min_p != nullptr ? P.min_p[row] : 0.0f;
  return in;
}

template <bool BF16, int NV>
__device__ __forceinline__ RowParams row_params_of(const RowInputs& in, int V) {
  using L = Layout<BF16>;
  RowParams r;
  r.T = 1.0f;
  r.p = 1.0f;
  r.u = 0.0f;
  r.k = V;
  r.st = 0;
  r.kind = kKindG;
  r.minp = 0.0f;
  const bool greedy = !(in.t > 0.0f);  // no temperature tensor reads as 0
  if (!greedy) {
    r.T = fmaxf(in.t, 1e-6f);
    int k = in.k;
    if (k < 1 || k >= V) k = V;
    r.k = k;
    r.p = fminf(fmaxf(in.p, 1e-6f), 1.0f);
    float u = in.u;
    if (!(u >= 0.0f && u < 1.0f)) {
      r.st |= kStBadUniform;
      u = (u != u) ? 0.0f : fminf(fmaxf(u, 0.0f), 0x1.fffffep-1f);
    }
    r.u = u;
    // K bounds the k-th value by the k-th largest thread maximum: it needs
    // at least k threads whose elements all lie inside the row.
    const int full_threads = V / (NV * L::VW);
    // min_p (off when <= 0 or NaN, at most 1) is one more cut on the kept
    // set of every filtered kind; a row with no other filter is filtered.
    r.minp = in.mp > 0.0f ? fminf(in.mp, 1.0f) : 0.0f;
    if (k < V && k <= kMaxK && full_threads >= k) {
      r.kind = kKindK;
    } else if (k == V && !(r.p < 1.0f) && !(r.minp > 0.0f)) {
      r.kind = kKindP;
    } else if (BF16) {
      r.kind = kKindH;
    } else {
      r.kind = k == V ? kKindT : kKindF;
    }
  }
  r.use_p = r.p < 1.0f;
  r.c2 = 1.4426950408889634f / r.T;  // log2(e) / T
  return r;
}

template <bool BF16, int NV>
__device__ __forceinline__ RowParams row_params(const SampleParams& P, int row, int C) {
  (void)C;
  return row_params_of<BF16, NV>(load_row_inputs(P, row), P.V);
}

}  // namespace pkv
