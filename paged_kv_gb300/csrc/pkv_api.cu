// C ABI of the decode-step tail (declared in include/pkv.h): argument
// validation, launch-shape choice and the kernel launches.  Host-only logic
// (pkv_alloc_pages) is plain C++.  Nothing here allocates device memory or
// synchronises a stream.

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <algorithm>
#include <atomic>

#include "../../include/pkv.h"
#include "launch_config.h"
#include "page_kernels.h"
#include "sample_params.h"

namespace pkv {
cudaError_t launch_sample_bf16(const SampleParams& P, const SampleConfig& c, int num_sms,
                               cudaStream_t stream);
cudaError_t launch_sample_fp32(const SampleParams& P, const SampleConfig& c, int num_sms,
                               cudaStream_t stream);
}  // namespace pkv

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return PKV_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// SM count of the current device (cached per device; threads that race on
// the first call store the same value).
int num_sms() {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 1;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t div_ceil(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

const char* pkv_last_error(void) { return g_err; }

int pkv_version(void) { return 310; }

size_t pkv_sample_workspace_bytes(int B, int V, pkv_dtype dt) {
  if (B < 1 || V < 1 || (dt != PKV_FP32 && dt != PKV_BF16)) return 0;
  // The larger of the aligned and the element-load launch shapes.
  size_t chunks = 0;
  for (bool vec : {true, false}) {
    pkv::SampleConfig cfg;
    if (pkv::choose_sample_config(B, V, dt == PKV_BF16, vec, num_sms(), &cfg)) {
      chunks = std::max(chunks, static_cast<size_t>(cfg.chunks));
    }
  }
  return pkv::sample_workspace_need(B, static_cast<int>(chunks), dt == PKV_BF16);
}

int pkv_sample_workspace_init(void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (workspace == nullptr) return fail(PKV_EINVAL, "workspace is NULL");
  if (workspace_bytes < pkv::kWorkspaceHeaderBytes)
    return fail(PKV_EINVAL, "workspace of %zu bytes is smaller than its %zu-byte header",
                workspace_bytes, pkv::kWorkspaceHeaderBytes);
  if (!aligned16(workspace)) return fail(PKV_EINVAL, "workspace is not 16-byte aligned");
  const cudaError_t e = cudaMemsetAsync(workspace, 0, pkv::kWorkspaceHeaderBytes,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace initialisation");
  return ok();
}

}  // extern "C"

namespace {

// Host checks of pkv_sample_batch's arguments other than the workspace.
int sample_args_error(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                      const float* temperature, const float* uniform, const int32_t* out_tokens,
                      const int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                      const int32_t* wb_rows, const int64_t* wb_cols) {
  if (logits == nullptr) return fail(PKV_EINVAL, "logits is NULL");
  if (out_tokens == nullptr) return fail(PKV_EINVAL, "out_tokens is NULL");
  if (dt != PKV_FP32 && dt != PKV_BF16) return fail(PKV_EINVAL, "dtype %d is not fp32 or bf16", dt);
  if (B < 1 || B > 65535) return fail(PKV_EINVAL, "B=%d outside [1, 65535]", B);
  if (V < 1) return fail(PKV_EINVAL, "V=%d < 1", V);
  if (row_stride < V) return fail(PKV_EINVAL, "row_stride=%lld < V=%d", (long long)row_stride, V);
  if (temperature != nullptr && uniform == nullptr)
    return fail(PKV_EINVAL, "uniform is required when temperature is given");
  if (token_pool != nullptr) {
    if (wb_rows == nullptr || wb_cols == nullptr)
      return fail(PKV_EINVAL, "token_pool given without wb_rows / wb_cols");
    if (pool_rows < 1 || pool_cols < 1)
      return fail(PKV_EINVAL, "token pool shape [%lld, %lld] is empty", (long long)pool_rows,
                  (long long)pool_cols);
  }
  const int max_v = dt == PKV_BF16 ? PKV_MAX_VOCAB_BF16 : PKV_MAX_VOCAB_FP32;
  if (V > max_v) return fail(PKV_EUNSUPPORTED, "V=%d above the maximum %d", V, max_v);
  return PKV_OK;
}

// Host checks of the page-fill arguments; fills *F when they pass.
int fill_args(const int32_t* cached_len, const int32_t* device_len, const int32_t* table_idx,
              int B, int page_size, const int32_t* free_slots, int64_t free_count,
              int32_t* page_table, int64_t pt_rows, int64_t pt_cols, int64_t* total_out,
              int32_t* status, pkv::FillParams* F) {
  if (B < 0 || B > PKV_MAX_FILL_BATCH)
    return fail(PKV_EINVAL, "B=%d outside [0, %d]", B, PKV_MAX_FILL_BATCH);
  if (page_size < 1) return fail(PKV_EINVAL, "page_size=%d < 1", page_size);
  if (B > 0) {
    if (cached_len == nullptr || device_len == nullptr || table_idx == nullptr ||
        page_table == nullptr || (free_slots == nullptr && free_count > 0))
      return fail(PKV_EINVAL, "NULL pointer argument");
    if (free_count < 0 || free_count > INT32_MAX)
      return fail(PKV_EINVAL, "free_count=%lld outside [0, 2^31)", (long long)free_count);
    if (pt_rows < 1 || pt_cols < 1) return fail(PKV_EINVAL, "empty page table");
  }
  F->cached_len = cached_len;
  F->device_len = device_len;
  F->table_idx = table_idx;
  F->B = B;
  F->page_size = page_size;
  F->free_slots = free_slots;
  F->free_count = free_count;
  F->page_table = page_table;
  F->pt_rows = pt_rows;
  F->pt_cols = pt_cols;
  F->total_out = total_out;
  F->status = status;
  F->vec4 = (page_size % 4 == 0) && (pt_cols % 4 == 0) && aligned16(page_table);
  return PKV_OK;
}

// Page-fill CTAs appended to the finish kernel by pkv_decode_tail.
constexpr int kFusedFillCtas = 32;

// Scratch of pkv_sample_batch_noalloc, for callers that cannot allocate
// device memory when they sample (a decode loop that must not stall on
// cudaMalloc, a stream under graph capture, an engine whose memory went to
// the KV pool): a zero-initialised device array of the
// library (one instance per device, held until the process exits), used as
// the sampler workspace.  Every call leaves it ready for the next; calls
// that overlap on the GPU race on it.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(64) << 20;
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's address on the current device: in host code the array's name
// is only a host-side stand-in, so the device address is looked up (with
// that device current) on the first call on each device and cached.  That
// first call should come before any stream capture.
cudaError_t static_scratch(void** out) {
  static std::atomic<void*> cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    void* c = cache[dev].load(std::memory_order_acquire);
    if (c != nullptr) {
      *out = c;
      return cudaSuccess;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev].store(p, std::memory_order_release);
  *out = p;
  return cudaSuccess;
}

// pkv_sample_batch, with an optional page fill run by extra finish CTAs.
int sample_launch(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                  const float* temperature, const int32_t* top_k, const float* top_p,
                  const float* min_p, const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                  int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                  const int64_t* wb_cols, float* probs_out, int32_t* status, void* workspace,
                  size_t workspace_bytes, pkv_stream_t stream, const pkv::FillParams* fill) {
  const int bad = sample_args_error(logits, dt, B, V, row_stride, temperature, uniform,
                                    out_tokens, token_pool, pool_rows, pool_cols, wb_rows,
                                    wb_cols);
  if (bad != PKV_OK) return bad;
  const bool bf16 = dt == PKV_BF16;
  const size_t elt = bf16 ? 2 : 4;
  // The bulk-copy path needs 16-byte-aligned row starts and row lengths.
  const bool vec = aligned16(logits) && ((static_cast<uint64_t>(row_stride) * elt) % 16 == 0) &&
                   ((static_cast<uint64_t>(V) * elt) % 16 == 0);
  pkv::SampleConfig cfg;
  if (!pkv::choose_sample_config(B, V, bf16, vec, num_sms(), &cfg))
    return fail(PKV_EUNSUPPORTED, "no launch shape covers V=%d", V);
  if (static_cast<int64_t>(cfg.chunks - 1) * cfg.chunk >= V)
    return fail(PKV_EUNSUPPORTED, "launch shape with an empty chunk (V=%d)", V);
  const size_t need = pkv::sample_workspace_need(B, cfg.chunks, bf16);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(PKV_EINVAL, "workspace of %zu bytes needed (pkv_sample_workspace_bytes), got %zu",
                need, workspace == nullptr ? static_cast<size_t>(0) : workspace_bytes);
  if (!aligned16(workspace)) return fail(PKV_EINVAL, "workspace is not 16-byte aligned");

  pkv::SampleParams P;
  P.logits = logits;
  P.row_stride = row_stride;
  P.B = B;
  P.V = V;
  P.temperature = temperature;
  P.top_k = top_k;
  P.top_p = top_p;
  P.min_p = min_p;
  P.uniform = uniform;
  P.out_tokens = out_tokens;
  P.token_pool = token_pool;
  P.pool_rows = pool_rows;
  P.pool_cols = pool_cols;
  P.wb_rows = wb_rows;
  P.wb_cols = wb_cols;
  P.probs_out = probs_out;
  P.status = status;
  P.cta_chunk = cfg.chunk;
  P.chunks = cfg.chunks;
  P.workspace = workspace;
  P.fill = fill != nullptr ? *fill : pkv::FillParams{};
  P.fill_ctas = (fill != nullptr && fill->B > 0) ? kFusedFillCtas : 0;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = bf16 ? pkv::launch_sample_bf16(P, cfg, num_sms(), s)
                             : pkv::launch_sample_fp32(P, cfg, num_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "sampler launch");
  return ok();
}

}  // namespace

extern "C" {

int pkv_sample_batch(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                     const float* temperature, const int32_t* top_k, const float* top_p,
                     const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                     int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                     const int64_t* wb_cols, float* probs_out, int32_t* status,
                     void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  return sample_launch(logits, dt, B, V, row_stride, temperature, top_k, top_p, nullptr,
                       uniform, out_tokens, token_pool, pool_rows, pool_cols, wb_rows, wb_cols,
                       probs_out, status, workspace, workspace_bytes, stream, nullptr);
}

int pkv_sample_batch_ex(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                        const float* temperature, const int32_t* top_k, const float* top_p,
                        const float* min_p, const float* uniform, int32_t* out_tokens,
                        int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                        const int32_t* wb_rows, const int64_t* wb_cols, float* probs_out,
                        int32_t* status, void* workspace, size_t workspace_bytes,
                        pkv_stream_t stream) {
  return sample_launch(logits, dt, B, V, row_stride, temperature, top_k, top_p, min_p,
                       uniform, out_tokens, token_pool, pool_rows, pool_cols, wb_rows, wb_cols,
                       probs_out, status, workspace, workspace_bytes, stream, nullptr);
}

int pkv_sample_batch_noalloc(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                             const float* temperature, const int32_t* top_k, const float* top_p,
                             const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                             int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                             const int64_t* wb_cols, float* probs_out, int32_t* status,
                             pkv_stream_t stream) {
  const int bad = sample_args_error(logits, dt, B, V, row_stride, temperature, uniform,
                                    out_tokens, token_pool, pool_rows, pool_cols, wb_rows,
                                    wb_cols);
  if (bad != PKV_OK) return bad;
  const size_t need = pkv_sample_workspace_bytes(B, V, dt);
  if (need > kStaticScratchBytes)
    return fail(PKV_EUNSUPPORTED,
                "B=%d, V=%d needs %zu bytes of scratch; the static scratch holds %zu "
                "(pass a workspace to pkv_sample_batch)",
                B, V, need, kStaticScratchBytes);
  void* scratch = nullptr;
  const cudaError_t e = static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "static scratch address");
  return pkv_sample_batch(logits, dt, B, V, row_stride, temperature, top_k, top_p, uniform,
                          out_tokens, token_pool, pool_rows, pool_cols, wb_rows, wb_cols,
                          probs_out, status, scratch, kStaticScratchBytes, stream);
}

int pkv_writeback_tokens(const int32_t* tokens, const int32_t* rows, const int64_t* cols, int B,
                         int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                         int32_t* status, pkv_stream_t stream) {
  if (B < 0) return fail(PKV_EINVAL, "B=%d < 0", B);
  if (B == 0) return ok();
  if (tokens == nullptr || rows == nullptr || cols == nullptr || token_pool == nullptr)
    return fail(PKV_EINVAL, "NULL pointer argument");
  if (pool_rows < 1 || pool_cols < 1) return fail(PKV_EINVAL, "empty token pool");
  const cudaError_t e = pkv::launch_writeback(tokens, rows, cols, B, token_pool, pool_rows,
                                              pool_cols, status,
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "write-back launch");
  return ok();
}

int pkv_alloc_pages(const int32_t* cached_len, const int32_t* device_len, int B, int page_size,
                    int64_t free_count, int32_t* first_page, int32_t* num_pages,
                    int64_t* offset, int64_t* total) {
  if (B < 0) return fail(PKV_EINVAL, "B=%d < 0", B);
  if (page_size < 1) return fail(PKV_EINVAL, "page_size=%d < 1", page_size);
  if (total == nullptr) return fail(PKV_EINVAL, "total is NULL");
  if (B > 0 && (cached_len == nullptr || device_len == nullptr || first_page == nullptr ||
                num_pages == nullptr || offset == nullptr))
    return fail(PKV_EINVAL, "NULL pointer argument");
  for (int i = 0; i < B; ++i) {
    if (cached_len[i] < 0 || device_len[i] < 0)
      return fail(PKV_EINVAL, "request %d: negative length (cached_len=%d device_len=%d)", i,
                  cached_len[i], device_len[i]);
  }
  int64_t acc = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t first = div_ceil(cached_len[i], page_size);
    const int64_t last = div_ceil(device_len[i], page_size);
    const int64_t n = last > first ? last - first : 0;
    first_page[i] = static_cast<int32_t>(first);
    num_pages[i] = static_cast<int32_t>(n);
    offset[i] = acc;
    acc += n;
  }
  *total = acc;
  if (acc > free_count)
    return fail(PKV_ENOSPC, "%lld pages needed, %lld free", (long long)acc, (long long)free_count);
  return ok();
}

int pkv_fill_page_table(const int32_t* cached_len, const int32_t* device_len,
                        const int32_t* table_idx, int B, int page_size,
                        const int32_t* free_slots, int64_t free_count, int32_t* page_table,
                        int64_t pt_rows, int64_t pt_cols, int64_t* total_out, int32_t* status,
                        pkv_stream_t stream) {
  pkv::FillParams F;
  const int bad = fill_args(cached_len, device_len, table_idx, B, page_size, free_slots,
                            free_count, page_table, pt_rows, pt_cols, total_out, status, &F);
  if (bad != PKV_OK) return bad;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) {
    if (total_out != nullptr) {
      const cudaError_t e = cudaMemsetAsync(total_out, 0, sizeof(int64_t), s);
      if (e != cudaSuccess) return cuda_fail(e, "total_out reset");
    }
    return ok();
  }
  const cudaError_t e = pkv::launch_fill_page_table(F, num_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "page-fill launch");
  return ok();
}

int pkv_decode_tail(const void* logits, pkv_dtype dt, int B, int V, int64_t row_stride,
                    const float* temperature, const int32_t* top_k, const float* top_p,
                    const float* uniform, int32_t* out_tokens, int32_t* token_pool,
                    int64_t pool_rows, int64_t pool_cols, const int32_t* wb_rows,
                    const int64_t* wb_cols, int32_t* status, void* workspace,
                    size_t workspace_bytes, const int32_t* cached_len, const int32_t* device_len,
                    const int32_t* table_idx, int fill_B, int page_size,
                    const int32_t* free_slots, int64_t free_count, int32_t* page_table,
                    int64_t pt_rows, int64_t pt_cols, int64_t* total_out,
                    pkv_stream_t stream) {
  pkv::FillParams F;
  const int bad = fill_args(cached_len, device_len, table_idx, fill_B, page_size, free_slots,
                            free_count, page_table, pt_rows, pt_cols, total_out, status, &F);
  if (bad != PKV_OK) return bad;
  if (fill_B == 0 && total_out != nullptr) {
    const cudaError_t e =
        cudaMemsetAsync(total_out, 0, sizeof(int64_t), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "total_out reset");
  }
  return sample_launch(logits, dt, B, V, row_stride, temperature, top_k, top_p, nullptr,
                       uniform, out_tokens, token_pool, pool_rows, pool_cols, wb_rows, wb_cols,
                       nullptr, status, workspace, workspace_bytes, stream, &F);
}

int pkv_prepare_step(const int32_t* cached_len, const int32_t* device_len,
                     const int32_t* table_idx, int B, int page_size, const int32_t* free_slots,
                     int64_t free_count, int32_t* page_table, int64_t pt_rows, int64_t pt_cols,
                     const int32_t* token_pool, int64_t pool_rows, int64_t pool_cols,
                     int32_t* positions, int32_t* input_ids, int32_t* out_loc, int64_t max_tokens,
                     int64_t* total_pages_out, int64_t* total_tokens_out, int32_t* status,
                     pkv_stream_t stream) {
  pkv::PrepareParams Q;
  const int bad = fill_args(cached_len, device_len, table_idx, B, page_size, free_slots,
                            free_count, page_table, pt_rows, pt_cols, total_pages_out, status,
                            &Q.fill);
  if (bad != PKV_OK) return bad;
  if (max_tokens < 0 || max_tokens > INT32_MAX)
    return fail(PKV_EINVAL, "max_tokens=%lld outside [0, 2^31)", (long long)max_tokens);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) {
    for (int64_t* out : {total_pages_out, total_tokens_out}) {
      if (out == nullptr) continue;
      const cudaError_t e = cudaMemsetAsync(out, 0, sizeof(int64_t), s);
      if (e != cudaSuccess) return cuda_fail(e, "total reset");
    }
    return ok();
  }
  if (token_pool == nullptr) return fail(PKV_EINVAL, "token_pool is NULL");
  if (pool_rows < 1 || pool_cols < 1) return fail(PKV_EINVAL, "empty token pool");
  if (max_tokens > 0 && (positions == nullptr || input_ids == nullptr || out_loc == nullptr))
    return fail(PKV_EINVAL, "NULL output array");
  Q.token_pool = token_pool;
  Q.pool_rows = pool_rows;
  Q.pool_cols = pool_cols;
  Q.positions = positions;
  Q.input_ids = input_ids;
  Q.out_loc = out_loc;
  Q.max_tokens = max_tokens;
  Q.tokens_out = total_tokens_out;
  const cudaError_t e = pkv::launch_prepare_step(Q, num_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "prepare launch");
  return ok();
}

int pkv_philox_uniforms(uint64_t seed, uint64_t offset, int B, float* uniform,
                        pkv_stream_t stream) {
  if (B < 0 || B > 65535) return fail(PKV_EINVAL, "B=%d outside [0, 65535]", B);
  if (B == 0) return ok();
  if (uniform == nullptr) return fail(PKV_EINVAL, "uniform is NULL");
  const cudaError_t e =
      pkv::launch_uniforms(seed, offset, B, uniform, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "uniforms launch");
  return ok();
}

int pkv_free_pages(const int32_t* table_idx, const int32_t* begin, const int32_t* end, int B,
                   int page_size, const int32_t* page_table, int64_t pt_rows, int64_t pt_cols,
                   int32_t* free_slots, int64_t free_count, int64_t free_capacity,
                   int64_t* total_out, int32_t* status, pkv_stream_t stream) {
  if (B < 0 || B > PKV_MAX_FILL_BATCH)
    return fail(PKV_EINVAL, "B=%d outside [0, %d]", B, PKV_MAX_FILL_BATCH);
  if (page_size < 1) return fail(PKV_EINVAL, "page_size=%d < 1", page_size);
  if (free_count < 0 || free_capacity < 0 || free_capacity > INT32_MAX || free_count > free_capacity)
    return fail(PKV_EINVAL, "free_count=%lld, free_capacity=%lld: need 0 <= count <= capacity < 2^31",
                (long long)free_count, (long long)free_capacity);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) {
    if (total_out != nullptr) {
      const cudaError_t e = cudaMemsetAsync(total_out, 0, sizeof(int64_t), s);
      if (e != cudaSuccess) return cuda_fail(e, "total_out reset");
    }
    return ok();
  }
  if (table_idx == nullptr || begin == nullptr || end == nullptr || page_table == nullptr ||
      free_slots == nullptr)
    return fail(PKV_EINVAL, "NULL pointer argument");
  if (pt_rows < 1 || pt_cols < 1) return fail(PKV_EINVAL, "empty page table");
  pkv::FreeParams F;
  F.table_idx = table_idx;
  F.begin = begin;
  F.end = end;
  F.B = B;
  F.page_size = page_size;
  F.page_table = page_table;
  F.pt_rows = pt_rows;
  F.pt_cols = pt_cols;
  F.free_slots = free_slots;
  F.free_count = free_count;
  F.capacity = free_capacity;
  F.total_out = total_out;
  F.status = status;
  const cudaError_t e = pkv::launch_free_pages(F, num_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "free launch");
  return ok();
}

int pkv_check_free_list(const int32_t* free_slots, int64_t free_count, int page_size,
                        int64_t num_pages, int64_t cache_pages, uint32_t* bitmap,
                        int64_t bitmap_words, int32_t* result, pkv_stream_t stream) {
  if (result == nullptr || bitmap == nullptr || (free_slots == nullptr && free_count > 0))
    return fail(PKV_EINVAL, "NULL pointer argument");
  if (free_count < 0 || free_count > INT32_MAX)
    return fail(PKV_EINVAL, "free_count=%lld outside [0, 2^31)", (long long)free_count);
  if (page_size < 1) return fail(PKV_EINVAL, "page_size=%d < 1", page_size);
  if (num_pages < 0 || cache_pages < 0)
    return fail(PKV_EINVAL, "num_pages=%lld, cache_pages=%lld: need >= 0", (long long)num_pages,
                (long long)cache_pages);
  if (num_pages > INT32_MAX / page_size)
    return fail(PKV_EINVAL, "num_pages * page_size = %lld * %d is not below 2^31",
                (long long)num_pages, page_size);
  const int64_t words = (num_pages + 31) / 32;
  if (bitmap_words < words)
    return fail(PKV_EINVAL, "bitmap of %lld words, %lld needed", (long long)bitmap_words,
                (long long)words);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(result, 0, sizeof(int32_t), s);
  if (e == cudaSuccess && words > 0) e = cudaMemsetAsync(bitmap, 0, static_cast<size_t>(words) * 4, s);
  if (e != cudaSuccess) return cuda_fail(e, "integrity scratch reset");
  e = pkv::launch_check_free_list(free_slots, free_count, page_size, num_pages, cache_pages, bitmap,
                                  result, num_sms(), s);
  if (e != cudaSuccess) return cuda_fail(e, "integrity launch");
  return ok();
}

}  // extern "C"
