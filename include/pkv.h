/*
 * pkv.h -- C ABI of the decode-step tail: batched per-request sampling with
 * fused token write-back, and paged-KV page allocation / page-table fill;
 * plus the step before the model, device uniforms, min_p and the free path.
 *
 * The operations follow "mini-sglang from Scratch":
 *   - sampling: page "The engine and the sampler", section "The sampler"
 *     (Sampler.prepare, Sampler.sample, sample_torch), and its exercise 2
 *     (min_p);
 *   - token write-back and the step before the model: page "The scheduler
 *     skeleton and the offline interface", section "Preparing a batch"
 *     (_prepare_batch, _make_write_tuple, Scheduler._forward);
 *   - page allocation, page-table fill and the free path: page
 *     "CacheManager: allocation, release and admission control", sections
 *     "The free-page list", "Allocating pages for this step's tokens"
 *     (_allocate, allocate_paged, _write_page_table), "Freeing, and freeing
 *     lazily", "The integrity check";
 *   - device uniforms: page "The scheduler's IO and multi-rank
 *     synchronization", section "Sending results" (one seed for every rank).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller unless the comment says
 *     "host".  The library never allocates, frees or copies caller memory and
 *     never synchronises: every call is enqueued on `stream` and returns.
 *   - Host-detectable errors return a negative pkv_status and launch nothing.
 *     pkv_last_error() then describes the problem (per calling thread).
 *   - Device-detectable problems set bits in the caller's int32 status word
 *     (zeroed by the caller; bits are OR-ed in, never cleared), write -1 for
 *     the affected token and skip the affected write.  No kernel traps.
 *   - Integers are int32 except lengths of device buffers and pool / table
 *     coordinates, which are int64.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,       /* bad argument: NULL pointer, size, stride, dtype */
  PKV_ENOSPC = -2,       /* not enough free pages (pkv_alloc_pages)          */
  PKV_ECUDA = -3,        /* a CUDA call failed (launch or attribute)         */
  PKV_EUNSUPPORTED = -4  /* valid but outside what the kernels handle        */
} pkv_status;

typedef enum { PKV_FP32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Bits of the device status word. */
#define PKV_ST_NONFINITE 1     /* NaN in a row, or +inf in a sampled row       */
#define PKV_ST_ALL_NEG_INF 2   /* sampled row whose logits are all -inf        */
#define PKV_ST_ROW_OOB 4       /* write-back / page-table row out of range     */
#define PKV_ST_COL_OOB 8       /* write-back / page-table column out of range  */
#define PKV_ST_BAD_UNIFORM 16  /* uniform outside [0,1): clamped, still drawn  */
#define PKV_ST_NOSPC 32        /* page fill: more pages needed than are free   */
#define PKV_ST_TIMEOUT 64      /* a row's records are missing or untrusted (a
                                  copy did not land in time, or the workspace
                                  was not initialised); the token is -1       */
#define PKV_ST_TOKEN_CAP 128   /* prepare step: more tokens than max_tokens    */

/* Largest vocabulary the sampler handles for each dtype. */
#define PKV_MAX_VOCAB_BF16 524288
#define PKV_MAX_VOCAB_FP32 262144
/* Largest batch of pkv_fill_page_table (its per-request scan lives in shared memory). */
#define PKV_MAX_FILL_BATCH 4096

/* Text of the last host-side error on this thread ("" if none). */
const char* pkv_last_error(void);

/* Library version, 100 * major + minor. */
int pkv_version(void);

/*
 * Device bytes of the workspace pkv_sample_batch needs for (B, V, dtype), or
 * 0 for invalid arguments.  The sampler runs as two kernels: the first splits
 * every row into chunks, hands the chunks out to its CTAs from counters in
 * the workspace header and leaves one record per (row, chunk) in the
 * workspace (about 3 KB each, plus 16 KB of per-slice counts on bf16 rows
 * for top-p); the second settles each row from its records.  The caller owns the workspace.  Before its first use it must be
 * initialised once, by pkv_sample_workspace_init or by zeroing it; every
 * call then leaves it ready for the next call on the same stream.  A
 * workspace must not be used by two calls that may run concurrently.
 */
size_t pkv_sample_workspace_bytes(int B, int V, pkv_dtype dt);

/*
 * pkv_sample_workspace_init -- enqueues on `stream` the zeroing of the
 * workspace header (the first 256 bytes).  workspace: device pointer, 16-byte
 * aligned, workspace_bytes >= 256.  Errors: PKV_EINVAL (NULL, too small,
 * unaligned), PKV_ECUDA.
 */
int pkv_sample_workspace_init(void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_sample_batch -- one token per row of a [B, V] logits matrix.
 *
 * Follows Sampler.sample / sample_torch ("The engine and the sampler",
 * section "The sampler") with torch.multinomial replaced by an inverse CDF
 * against a caller-supplied uniform:
 *   - temperature == NULL: the whole batch is greedy (torch.argmax);
 *   - a row with temperature <= 0 is greedy and returns the exact argmax;
 *   - otherwise T = max(temperature, 1e-6); top_k < 1 or >= V means no top-k;
 *     top_p is clamped into [1e-6, 1] (NULL top_k / top_p: off for all rows);
 *     the row is filtered top-k first, then top-p on the renormalised top-k
 *     distribution (a token is kept while the mass before it is < top_p), and
 *     the kept set is renormalised and walked in ascending vocab index: the
 *     token is the first i with uniform < cumulative probability.
 * Ties anywhere (argmax, the k-th and the top-p boundary) go to the lowest
 * index.  Arithmetic is fp32 (bf16 logits are widened exactly).
 *
 *   logits      [B, row_stride] fp32 or bf16, row-major; only the first V
 *               entries of each row are read.  Rows whose start and length
 *               are 16-byte aligned (base, row_stride * element size and
 *               V * element size) are fetched with bulk copies; others with
 *               element loads.
 *   temperature [B] fp32 or NULL      top_k [B] int32 or NULL
 *   top_p       [B] fp32 or NULL      uniform [B] fp32, required unless
 *                                     temperature is NULL
 *   out_tokens  [B] int32, written (-1 for a row with a device error)
 *   token_pool  [pool_rows, pool_cols] int32 or NULL.  When given, the fused
 *               write-back does token_pool[wb_rows[b], wb_cols[b]] = token for
 *               every row with wb_cols[b] >= 0 and token >= 0 (the write
 *               tuple's column -1 means "do not write").
 *   wb_rows     [B] int32, wb_cols [B] int64 (required with token_pool)
 *   probs_out   [B, V] fp32 or NULL: debug output of the kept-set
 *               probabilities (one-hot for greedy rows); leave NULL when timing.
 *   status      device int32 status word or NULL.
 *   workspace   device memory of at least pkv_sample_workspace_bytes(B, V, dt)
 *               bytes (workspace_bytes), 16-byte aligned, initialised once
 *               before its first use (pkv_sample_workspace_init); not to be
 *               shared by calls that may run concurrently.
 * Errors: PKV_EINVAL (NULL required pointer, B < 1, B > 65535, V < 1,
 * row_stride < V, bad dtype, pool sizes < 1, workspace missing, too small or
 * unaligned), PKV_EUNSUPPORTED (V above PKV_MAX_VOCAB_*), PKV_ECUDA (launch
 * failure).
 */
int pkv_sample_batch(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                     const float* temperature, const int32_t* top_k, const float* top_p,
                     const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                     int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                     const int64_t* wb_cols, float* probs_out, int32_t* status,
                     void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_sample_batch_ex -- pkv_sample_batch with a min_p filter ("The engine and
 * the sampler", exercise 2 and its answer): in a sampled row, a token stays
 * only if its probability is at least min_p[b] times the row's largest
 * probability (on the full distribution after temperature scaling), a mask
 * intersected with the top-k / top-p set before the renormalisation and the
 * draw.  min_p [B] float (device) or NULL (off for every row); a value <= 0
 * or NaN is off, above 1 is 1.  Greedy rows ignore it.  A sampled row with
 * no other filter becomes a filtered row (slower than a plain one).  All
 * other arguments, the meaning and the errors are those of
 * pkv_sample_batch, which equals this call with min_p NULL.
 */
int pkv_sample_batch_ex(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                        const float* temperature, const int32_t* top_k, const float* top_p,
                        const float* min_p, const float* uniform, int32_t* out_tokens,
                        int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                        const int32_t* wb_rows, const int64_t* wb_cols, float* probs_out,
                        int32_t* status, void* workspace, size_t workspace_bytes,
                        pkv_stream_t stream);

/*
 * pkv_sample_batch_noalloc -- pkv_sample_batch without a caller workspace.
 * The source pages have no counterpart: this entry point exists for callers
 * that cannot allocate device memory at the point where they sample.  Such
 * callers include a decode loop that must never stall (cudaMalloc can
 * synchronise the device and has no latency bound), code running while a
 * stream is being captured into a CUDA graph (allocation is not allowed
 * there), and engines that handed nearly all free memory to the KV pool at
 * start-up and have no headroom left.  The call itself uses the CUDA runtime
 * (it looks up the array and launches kernels), so it is made from ordinary
 * host code, never from inside a host callback on a stream.
 *
 * Same arguments, meaning and errors as pkv_sample_batch, minus the
 * workspace: the sampler's scratch is a 64 MiB device array inside the
 * library (one per device, zero at load time, left ready by every call), so
 * the call allocates nothing anywhere.  The first call on a device looks up
 * that array's device address (cudaGetSymbolAddress) and caches it, so make
 * that first call before any stream capture.  Calls on one device share the
 * array: calls that overlap on the GPU (different streams without ordering)
 * race on it and must be avoided.
 * Errors: those of pkv_sample_batch, plus PKV_EUNSUPPORTED when
 * pkv_sample_workspace_bytes(B, V, dt) exceeds 64 MiB (e.g. B=1024,
 * V=256000), and PKV_ECUDA when the array's address cannot be read.
 */
int pkv_sample_batch_noalloc(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                             const float* temperature, const int32_t* top_k, const float* top_p,
                             const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                             int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                             const int64_t* wb_cols, float* probs_out, int32_t* status,
                             pkv_stream_t stream);

/*
 * pkv_decode_tail -- the whole decode-step tail in one call: pkv_sample_batch
 * (with its fused write-back) and pkv_fill_page_table for the same step.
 *
 * The page fill has no dependence on the sampled tokens, so it runs in extra
 * CTAs of the sampler's second kernel while the rows are being settled.  The
 * arguments are those of the two calls (the sampler's B, V, logits ... and
 * the fill's cached_len ... with its own batch size fill_B and the page
 * table); `status` is shared; there is no probs_out.  Results, status bits
 * and errors are exactly those of the two calls made one after the other.
 * Host errors of either argument set return before anything is launched.
 */
int pkv_decode_tail(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                    const float* temperature, const int32_t* top_k, const float* top_p,
                    const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                    int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                    const int64_t* wb_cols, int32_t* status, void* workspace,
                    size_t workspace_bytes, const int32_t* cached_len, const int32_t* device_len,
                    const int32_t* table_idx, int fill_B, int page_size,
                    const int32_t* free_slots, int64_t free_count, int32_t* page_table,
                    int64_t pt_rows, int64_t pt_cols, int64_t* total_out,
                    pkv_stream_t stream);

/*
 * pkv_writeback_tokens -- token_pool[rows[b], cols[b]] = tokens[b].
 *
 * The standalone form of the write-back in Scheduler._forward ("The scheduler
 * skeleton and the offline interface", section "Preparing a batch").  Rows
 * with cols[b] < 0 or tokens[b] < 0 are skipped; out-of-range rows / columns
 * set PKV_ST_ROW_OOB / PKV_ST_COL_OOB and are skipped.
 *   tokens [B] int32, rows [B] int32, cols [B] int64,
 *   token_pool [pool_rows, pool_cols] int32, status device int32 or NULL.
 * Errors: PKV_EINVAL (NULL pointer, B < 0, pool sizes < 1), PKV_ECUDA.
 * B == 0 is a no-op.
 */
int pkv_writeback_tokens(const int32_t* tokens, const int32_t* rows, const int64_t* cols,
                         int B, int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                         int32_t* status, pkv_stream_t stream);

/*
 * pkv_alloc_pages -- HOST computation of this step's page allocation
 * (CacheManager.allocate_paged, "CacheManager: allocation, release and
 * admission control", section "Allocating pages for this step's tokens").
 *
 * For request i: first_page[i] = ceil(cached_len[i] / page_size),
 * num_pages[i] = max(0, ceil(device_len[i] / page_size) - first_page[i]),
 * offset[i] = sum of num_pages[j] for j < i (pages are taken from the front of
 * the free list in batch order), *total = sum of num_pages.
 * All pointers are HOST pointers.  Returns PKV_ENOSPC when *total >
 * free_count (outputs are still filled), PKV_EINVAL for NULL pointers, B < 0,
 * page_size < 1 or a negative length.  The caller advances its free list by
 * *total.
 */
int pkv_alloc_pages(const int32_t* cached_len, const int32_t* device_len, int B,
                    int page_size, int64_t free_count, int32_t* first_page,
                    int32_t* num_pages, int64_t* offset, int64_t* total);

/*
 * pkv_fill_page_table -- device page allocation plus page-table fill
 * (_write_page_table with the page-to-token expansion, same section).
 *
 * On device: the per-request page counts of pkv_alloc_pages, their exclusive
 * scan, and for j < num_pages[i], o < page_size:
 *   page_table[table_idx[i], (first_page[i] + j) * page_size + o]
 *       = free_slots[offset[i] + j] + o
 * i.e. whole pages, even past device_len.  free_slots holds the first token
 * location of each free page; pages are taken from its front.  Nothing else
 * in page_table changes.  If the total exceeds free_count, PKV_ST_NOSPC is set,
 * *total_out is 0 and nothing is written.  A request whose table row or last
 * column is out of range sets PKV_ST_ROW_OOB / PKV_ST_COL_OOB and is skipped
 * (its pages are still counted as taken).
 *   cached_len, device_len, table_idx [B] int32; free_slots [free_count] int32;
 *   page_table [pt_rows, pt_cols] int32; total_out device int64 or NULL
 *   (receives the number of pages taken); status device int32 or NULL.
 * Errors: PKV_EINVAL (NULL pointer, B < 0, B > PKV_MAX_FILL_BATCH,
 * page_size < 1, free_count outside [0, 2^31), empty table), PKV_ECUDA.
 * B == 0 writes *total_out = 0.
 */
int pkv_fill_page_table(const int32_t* cached_len, const int32_t* device_len,
                        const int32_t* table_idx, int B, int page_size,
                        const int32_t* free_slots, int64_t free_count, int32_t* page_table,
                        int64_t pt_rows, int64_t pt_cols, int64_t* total_out,
                        int32_t* status, pkv_stream_t stream);

/*
 * pkv_free_pages -- batched lazy free ("CacheManager: allocation, release
 * and admission control", section "Freeing, and freeing lazily":
 * lazy_free_region appends indices[::page_size] of every freed index tensor
 * and concatenates the lot onto free_slots once).
 *
 * The freed indices of request i are the slice
 * page_table[table_idx[i], begin[i] : end[i]] of its table row (cache_req,
 * section "Handing the KV to the prefix cache", frees slices of
 * page_table[table_idx, :cached_len]).  On device, in batch order, every
 * page_size-th entry of each slice starting at its first,
 *   page_table[table_idx[i], begin[i] + j * page_size],
 *   j < ceil((end[i] - begin[i]) / page_size),
 * is appended at free_slots[free_count ...].  A range with end <= begin frees
 * nothing.  A range whose row lies outside the table sets PKV_ST_ROW_OOB,
 * one with begin < 0 or end > pt_cols sets PKV_ST_COL_OOB; either frees
 * nothing.  If free_count plus the entries to append exceeds free_capacity,
 * PKV_ST_NOSPC is set, *total_out is 0 and nothing is written.
 *   table_idx, begin, end [B] int32 (device); page_table [pt_rows, pt_cols]
 *   int32 (device, read only); free_slots [free_capacity] int32 (device),
 *   entries [0, free_count) live; total_out device int64 or NULL (receives
 *   the number of entries appended; the caller's new count is free_count
 *   plus it); status device int32 or NULL.
 * Errors: PKV_EINVAL (NULL pointer, B < 0, B > PKV_MAX_FILL_BATCH,
 * page_size < 1, free_count or free_capacity outside [0, 2^31) or
 * free_count > free_capacity, empty table), PKV_ECUDA.  B == 0 writes
 * *total_out = 0.
 */
int pkv_free_pages(const int32_t* table_idx, const int32_t* begin, const int32_t* end, int B,
                   int page_size, const int32_t* page_table, int64_t pt_rows, int64_t pt_cols,
                   int32_t* free_slots, int64_t free_count, int64_t free_capacity,
                   int64_t* total_out, int32_t* status, pkv_stream_t stream);

/*
 * pkv_prepare_step -- the step before the model, in one launch ("The
 * scheduler skeleton and the offline interface", section "Preparing a batch":
 * Scheduler._prepare_batch, then the input gather of Scheduler._forward):
 *   1. the page allocation and table fill of pkv_fill_page_table (same
 *      arguments, same rules, *total_pages_out = pages taken from the front
 *      of free_slots);
 *   2. positions = the positions [cached_len[i], device_len[i]) of every
 *      request, packed in batch order (a request with device_len <=
 *      cached_len has none);
 *   3. for packed entry j of request i at position p:
 *        input_ids[j] = token_pool[table_idx[i], p],
 *        out_loc[j]   = page_table[table_idx[i], p]  (after step 1).
 * *total_tokens_out = the step's token count N (always written).  If N >
 * max_tokens, PKV_ST_TOKEN_CAP is set and nothing else is written; if the
 * pages do not fit, PKV_ST_NOSPC is set and nothing else is written.  A
 * request whose gathers would leave the pool or the table (row outside
 * either: PKV_ST_ROW_OOB; cached_len < 0, device_len past either's columns,
 * or new pages the fill skipped: PKV_ST_COL_OOB) keeps its positions and gets
 * -1 in input_ids and out_loc.
 *   cached_len, device_len, table_idx [B] int32 (device); free_slots
 *   [free_count] int32 (device); page_table [pt_rows, pt_cols] int32
 *   (device, written); token_pool [pool_rows, pool_cols] int32 (device, read
 *   only); positions, input_ids, out_loc [max_tokens] int32 (device,
 *   written); total_pages_out, total_tokens_out device int64 or NULL; status
 *   device int32 or NULL.  The caller advances free_slots by the page total.
 * Errors: those of pkv_fill_page_table, plus PKV_EINVAL for max_tokens
 * outside [0, 2^31), a NULL or empty token pool, or a NULL output array when
 * max_tokens > 0; PKV_ECUDA.  B == 0 writes both totals as 0.
 */
int pkv_prepare_step(const int32_t* cached_len, const int32_t* device_len,
                     const int32_t* table_idx, int B, int page_size, const int32_t* free_slots,
                     int64_t free_count, int32_t* page_table, int64_t pt_rows, int64_t pt_cols,
                     const int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                     int32_t* positions, int32_t* input_ids, int32_t* out_loc, int64_t max_tokens,
                     int64_t* total_pages_out, int64_t* total_tokens_out, int32_t* status,
                     pkv_stream_t stream);

/*
 * pkv_philox_uniforms -- the uniforms of one sampler call, generated on the
 * device so the draw needs no host input.  The pages seed one generator per
 * engine (torch.manual_seed(42) in Engine) and rely on every tensor-parallel
 * rank making the same random calls ("The scheduler's IO and multi-rank
 * synchronization", section "Sending results"); a counter-based generator
 * gives each (call, row) its own number, so ranks that pass the same seed and
 * call number agree by construction.
 *
 * uniform[b] = (word 0 of Philox-4x64-10(counter = (b, offset, 0, 0),
 * key = (seed, 0))) >> 40, times 2^-24: in [0, 1), exact in fp32.  Philox
 * as published by Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3" (SC 2011).  `offset` is the caller's call number (e.g.
 * the decode step).
 *   uniform [B] float (device, written); B in [0, 65535].
 * Errors: PKV_EINVAL (B out of range, NULL uniform with B > 0), PKV_ECUDA.
 */
int pkv_philox_uniforms(uint64_t seed, uint64_t offset, int B, float* uniform,
                        pkv_stream_t stream);

/* Bits of pkv_check_free_list's result. */
#define PKV_FL_COUNT 1      /* free pages + cached pages != pool pages          */
#define PKV_FL_ALIGN 2      /* an entry is not a multiple of page_size (ps > 1) */
#define PKV_FL_RANGE 4      /* an entry outside [0, num_pages * page_size)      */
#define PKV_FL_DUPLICATE 8  /* a page listed more than once                     */

/*
 * pkv_check_free_list -- the free-list integrity check as a device reduction
 * (same page, section "The integrity check": check_integrity requires
 * len(free_slots) + cache_pages == num_pages and, for page_size > 1, every
 * entry a multiple of page_size).  Two more checks serve what the section
 * says the check is for (a page forgotten or freed twice): every entry is the
 * start of a pool page, and no page is listed twice.
 *
 * Enqueues the zeroing of *result and of the bitmap, then one kernel that
 * ORs PKV_FL_* bits into *result.  An entry failing the alignment check is
 * not checked further; one outside the pool is not checked for duplicates.
 *   free_slots [free_count] int32 (device); num_pages, cache_pages >= 0;
 *   bitmap [bitmap_words] uint32 device scratch, bitmap_words >=
 *   ceil(num_pages / 32); result device int32.
 * Errors: PKV_EINVAL (NULL pointer, free_count outside [0, 2^31), page_size
 * < 1, num_pages or cache_pages < 0, num_pages * page_size >= 2^31, bitmap
 * too small), PKV_ECUDA.
 */
int pkv_check_free_list(const int32_t* free_slots, int64_t free_count, int page_size,
                        int64_t num_pages, int64_t cache_pages, uint32_t* bitmap,
                        int64_t bitmap_words, int32_t* result, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
