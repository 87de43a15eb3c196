// Host side of the C ABI declared in include/ds_sparse_mla.h: argument
// validation before any launch, error messages that name the offending
// parameter, the supported-shape query and the workspace-size queries.
//
// The contract follows the pages: caller-owned outputs, validation before the
// kernel launch ("[JJ] Preallocate DeepSeek V4 padded-query output", section
// "Operation contract"), a hard error instead of a fallback for missing
// support ("Batch-invariant kernels for 0-diff RL"), and a dispatch miss that
// says which of num_heads / topk / page_block_size / d_qk missed and what is
// available ("Make DSV4 sparse MLA work end-to-end", section "SM120 gate").

#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "ds_sparse_mla.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int ok() {
  g_last_error.clear();
  return DS_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_config(const char* fn, int num_heads, int topk, int page_block_size, int d_qk, int d_v,
                 int kv_dtype) {
  if (num_heads != 16 && num_heads != 32 && num_heads != 64 && num_heads != 128)
    return fail(DS_ERR_UNSUPPORTED, "%s: num_heads=%d is not supported; available: 16, 32, 64, 128",
                fn, num_heads);
  if (topk < 64 || topk > 2048 || topk % 64 != 0)
    return fail(DS_ERR_UNSUPPORTED,
                "%s: topk=%d is not supported; available: multiples of 64 in [64, 2048]", fn, topk);
  if (page_block_size != DS_PAGE_BLOCK_SIZE)
    return fail(DS_ERR_UNSUPPORTED, "%s: page_block_size=%d is not supported; available: 64", fn,
                page_block_size);
  if (d_qk != DS_D_QK)
    return fail(DS_ERR_UNSUPPORTED, "%s: d_qk=%d is not supported; available: 576", fn, d_qk);
  if (d_v != DS_D_V)
    return fail(DS_ERR_UNSUPPORTED, "%s: d_v=%d is not supported; available: 512", fn, d_v);
  if (kv_dtype != DS_KV_BF16 && kv_dtype != DS_KV_FP8_E4M3)
    return fail(DS_ERR_DTYPE, "%s: kv_dtype=%d is unknown; available: 0 (bf16), 1 (fp8 e4m3)", fn,
                kv_dtype);
  return DS_OK;
}

// The optional second entry list (a sliding window) and the sinks.
struct Window {
  const void* pages = nullptr;
  int64_t num_pages = 0;
  const int32_t* block_table = nullptr;
  int64_t bt_stride = 0;
  const int32_t* idx = nullptr;
  const int32_t* lens = nullptr;
  int width = 0;
  const float* sink = nullptr;
};

int check_window(const char* fn, const Window& w) {
  if (w.width != 0 && (w.width < 64 || w.width > 512 || w.width % 64 != 0))
    return fail(DS_ERR_UNSUPPORTED,
                "%s: swa_width=%d is not supported; available: 0 or a multiple of 64 in [64, 512]",
                fn, w.width);
  return DS_OK;
}

int attention_common(const char* fn, const void* q, const void* kv_pages, int kv_dtype,
                     int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                     int64_t num_bt_rows, const int32_t* row_req, const int32_t* idx,
                     const int32_t* lens, int64_t num_rows, int num_heads, int k, float scale,
                     void* out, float* lse, void* workspace, size_t workspace_bytes,
                     int32_t* err_flag, void* stream, const Window& win = Window()) {
  int st = check_config(fn, num_heads, k, DS_PAGE_BLOCK_SIZE, DS_D_QK, DS_D_V, kv_dtype);
  if (st != DS_OK) return st;
  st = check_window(fn, win);
  if (st != DS_OK) return st;
  if (num_rows < 0) return fail(DS_ERR_SHAPE, "%s: num_rows=%lld is negative", fn, (long long)num_rows);
  if (num_rows == 0) return ok();
  const int64_t splits = dsmla::num_splits_total(k, win.width);
  const int64_t groups = num_heads > 64 ? num_heads / 64 : 1;
  if (num_rows > (int64_t)INT32_MAX / (splits * groups) || num_rows * num_heads > (int64_t)INT32_MAX)
    return fail(DS_ERR_UNSUPPORTED, "%s: num_rows=%lld is too large for one launch (max %lld)", fn,
                (long long)num_rows, (long long)((int64_t)INT32_MAX / (splits * groups * 2)));
  if (num_pages < 1) return fail(DS_ERR_SHAPE, "%s: num_pages=%lld must be >= 1", fn, (long long)num_pages);
  if (num_pages > (int64_t)INT32_MAX / DS_PAGE_BLOCK_SIZE)
    return fail(DS_ERR_UNSUPPORTED, "%s: num_pages=%lld exceeds %lld (KV rows are indexed in 32 bits)",
                fn, (long long)num_pages, (long long)(INT32_MAX / DS_PAGE_BLOCK_SIZE));
  if (bt_stride < 1) return fail(DS_ERR_SHAPE, "%s: bt_stride=%lld must be >= 1", fn, (long long)bt_stride);
  if (num_bt_rows < 1)
    return fail(DS_ERR_SHAPE, "%s: num_requests=%lld must be >= 1", fn, (long long)num_bt_rows);
  if (!std::isfinite(scale)) return fail(DS_ERR_SHAPE, "%s: scale must be finite", fn);
  struct {
    const void* p;
    const char* name;
    uintptr_t align;
  } ptrs[] = {{q, "q", 16},           {kv_pages, "kv_pages", 16}, {block_table, "block_table", 4},
              {idx, "idx", 4},        {lens, "lens", 4},          {out, "out", 16},
              {lse, "lse", 4},        {workspace, "workspace", 256}};
  for (auto& x : ptrs) {
    if (x.p == nullptr) return fail(DS_ERR_NULL, "%s: %s is NULL", fn, x.name);
    if (!aligned(x.p, x.align))
      return fail(DS_ERR_ALIGN, "%s: %s must be %d-byte aligned", fn, x.name, (int)x.align);
  }
  if (row_req != nullptr && !aligned(row_req, 4))
    return fail(DS_ERR_ALIGN, "%s: row_req must be 4-byte aligned", fn);
  if (err_flag != nullptr && !aligned(err_flag, 4))
    return fail(DS_ERR_ALIGN, "%s: err_flag must be 4-byte aligned", fn);
  if (win.width > 0) {
    if (win.num_pages < 1)
      return fail(DS_ERR_SHAPE, "%s: swa_num_pages=%lld must be >= 1", fn, (long long)win.num_pages);
    if (win.num_pages > (int64_t)INT32_MAX / DS_PAGE_BLOCK_SIZE)
      return fail(DS_ERR_UNSUPPORTED, "%s: swa_num_pages=%lld exceeds %lld", fn,
                  (long long)win.num_pages, (long long)(INT32_MAX / DS_PAGE_BLOCK_SIZE));
    if (win.bt_stride < 1)
      return fail(DS_ERR_SHAPE, "%s: swa_bt_stride=%lld must be >= 1", fn, (long long)win.bt_stride);
    struct {
      const void* p;
      const char* name;
      uintptr_t align;
    } wp[] = {{win.pages, "swa_pages", 16}, {win.block_table, "swa_block_table", 4},
              {win.idx, "swa_idx", 4}, {win.lens, "swa_lens", 4}};
    for (auto& x : wp) {
      if (x.p == nullptr) return fail(DS_ERR_NULL, "%s: %s is NULL", fn, x.name);
      if (!aligned(x.p, x.align))
        return fail(DS_ERR_ALIGN, "%s: %s must be %d-byte aligned", fn, x.name, (int)x.align);
    }
  }
  if (win.sink != nullptr && !aligned(win.sink, 4))
    return fail(DS_ERR_ALIGN, "%s: attn_sink must be 4-byte aligned", fn);
  const size_t need = dsmla::attn_workspace_bytes(num_rows, num_heads, k, win.width);
  if (workspace_bytes < need)
    return fail(DS_ERR_WORKSPACE, "%s: workspace_bytes=%zu is smaller than the %zu bytes needed", fn,
                workspace_bytes, need);

  dsmla::AttnArgs a;
  a.q = q;
  a.kv = kv_pages;
  a.kv_dtype = kv_dtype;
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.num_bt_rows = num_bt_rows;
  a.row_req = row_req;
  a.idx = idx;
  a.lens = lens;
  a.R = num_rows;
  a.H = num_heads;
  a.k = k;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.err_flag = err_flag;
  a.kv2 = win.pages;
  a.num_pages2 = win.num_pages;
  a.block_table2 = win.block_table;
  a.bt_stride2 = win.bt_stride;
  a.idx2 = win.idx;
  a.lens2 = win.lens;
  a.k2 = win.width;
  a.sink = win.sink;
  cudaError_t e = dsmla::launch_sparse_mla(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

}  // namespace

namespace dsmla {

int report_error(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

}  // namespace dsmla

extern "C" {

const char* ds_last_error(void) { return g_last_error.c_str(); }

int ds_supported_config(int num_heads, int topk, int page_block_size, int d_qk, int d_v,
                        int kv_dtype) {
  if (check_config("ds_supported_config", num_heads, topk, page_block_size, d_qk, d_v, kv_dtype) !=
      DS_OK)
    return 0;
  ok();
  return 1;
}

size_t ds_topk_workspace_size(int64_t num_rows, int64_t row_stride, int k) {
  (void)k;
  if (num_rows < 1 || num_rows > INT32_MAX || row_stride < 1 || row_stride > (int64_t(1) << 28))
    return 0;
  return dsmla::topk_workspace_bytes(num_rows, row_stride);
}

size_t ds_sparse_mla_workspace_size(int64_t num_rows, int num_heads, int k) {
  if (num_rows < 0) return 0;
  if (check_config("ds_sparse_mla_workspace_size", num_heads, k, DS_PAGE_BLOCK_SIZE, DS_D_QK,
                   DS_D_V, DS_KV_BF16) != DS_OK)
    return 0;
  return dsmla::attn_workspace_bytes(num_rows, num_heads, k);
}

int ds_topk_per_row(const float* scores, int64_t row_stride, int64_t num_rows,
                    const int32_t* row_starts, const int32_t* row_ends, int k, int32_t* idx_out,
                    void* workspace, size_t workspace_bytes, void* stream) {
  const char* fn = "ds_topk_per_row";
  if (k < 1 || k > 16384) return fail(DS_ERR_UNSUPPORTED, "%s: k=%d must be in [1, 16384]", fn, k);
  if (row_stride < 1 || row_stride > (int64_t(1) << 28))
    return fail(DS_ERR_UNSUPPORTED, "%s: row_stride=%lld must be in [1, 2^28]", fn,
                (long long)row_stride);
  if (num_rows < 0) return fail(DS_ERR_SHAPE, "%s: num_rows=%lld is negative", fn, (long long)num_rows);
  if (num_rows > INT32_MAX)
    return fail(DS_ERR_UNSUPPORTED, "%s: num_rows=%lld exceeds 2^31-1", fn, (long long)num_rows);
  if (num_rows == 0) return ok();
  if (scores == nullptr) return fail(DS_ERR_NULL, "%s: scores is NULL", fn);
  if (row_starts == nullptr) return fail(DS_ERR_NULL, "%s: row_starts is NULL", fn);
  if (row_ends == nullptr) return fail(DS_ERR_NULL, "%s: row_ends is NULL", fn);
  if (idx_out == nullptr) return fail(DS_ERR_NULL, "%s: idx_out is NULL", fn);
  if (!aligned(scores, 4)) return fail(DS_ERR_ALIGN, "%s: scores must be 4-byte aligned", fn);
  if (!aligned(row_starts, 4) || !aligned(row_ends, 4) || !aligned(idx_out, 4))
    return fail(DS_ERR_ALIGN, "%s: row_starts, row_ends and idx_out must be 4-byte aligned", fn);
  if (workspace != nullptr && !aligned(workspace, 256))
    return fail(DS_ERR_ALIGN, "%s: workspace must be 256-byte aligned", fn);
  cudaError_t e = dsmla::launch_topk(scores, row_stride, num_rows, row_starts, row_ends, k, idx_out,
                                     workspace, workspace_bytes,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

int ds_sparse_mla_decode(const void* q, const void* kv_pages, int kv_dtype, int64_t num_pages,
                         const int32_t* block_table, int64_t bt_stride, const int32_t* idx,
                         const int32_t* lens, int64_t num_rows, int num_heads, int k, float scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, void* stream) {
  return attention_common("ds_sparse_mla_decode", q, kv_pages, kv_dtype, num_pages, block_table,
                          bt_stride, num_rows < 1 ? 1 : num_rows, nullptr, idx, lens, num_rows,
                          num_heads, k, scale, out, lse, workspace, workspace_bytes, err_flag,
                          stream);
}

int ds_sparse_mla_prefill(const void* q, const void* kv_pages, int kv_dtype, int64_t num_pages,
                          const int32_t* block_table, int64_t bt_stride, int64_t num_requests,
                          const int32_t* row_req, const int32_t* idx, const int32_t* lens,
                          int64_t num_tokens, int num_heads, int k, float scale, void* out,
                          float* lse, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                          void* stream) {
  if (num_tokens > 0 && row_req == nullptr)
    return fail(DS_ERR_NULL, "ds_sparse_mla_prefill: row_req is NULL");
  return attention_common("ds_sparse_mla_prefill", q, kv_pages, kv_dtype, num_pages, block_table,
                          bt_stride, num_requests, row_req, idx, lens, num_tokens, num_heads, k,
                          scale, out, lse, workspace, workspace_bytes, err_flag, stream);
}

int ds_kv_cache_write(const void* latent, int64_t num_rows, const int64_t* slots, int kv_dtype,
                      void* kv_pages, int64_t num_pages, int32_t* err_flag, void* stream) {
  const char* fn = "ds_kv_cache_write";
  if (kv_dtype != DS_KV_BF16 && kv_dtype != DS_KV_FP8_E4M3)
    return fail(DS_ERR_DTYPE, "%s: kv_dtype=%d must be DS_KV_BF16 (0) or DS_KV_FP8_E4M3 (1)", fn,
                kv_dtype);
  if (num_rows < 0) return fail(DS_ERR_SHAPE, "%s: num_rows=%lld must be >= 0", fn, (long long)num_rows);
  if (num_pages < 1) return fail(DS_ERR_SHAPE, "%s: num_pages=%lld must be >= 1", fn, (long long)num_pages);
  if (num_pages > INT64_MAX / (DS_PAGE_BLOCK_SIZE * (int64_t)DS_KV_ROW_BYTES_BF16))
    return fail(DS_ERR_UNSUPPORTED, "%s: num_pages=%lld is too large", fn, (long long)num_pages);
  if (num_rows == 0) return ok();
  struct {
    const void* p;
    const char* name;
    uintptr_t align;
  } ptrs[] = {{latent, "latent", 16}, {slots, "slots", 8}, {kv_pages, "kv_pages", 16}};
  for (auto& x : ptrs) {
    if (x.p == nullptr) return fail(DS_ERR_NULL, "%s: %s is NULL", fn, x.name);
    if (!aligned(x.p, x.align))
      return fail(DS_ERR_ALIGN, "%s: %s must be %d-byte aligned", fn, x.name, (int)x.align);
  }
  if (err_flag != nullptr && !aligned(err_flag, 4))
    return fail(DS_ERR_ALIGN, "%s: err_flag must be 4-byte aligned", fn);
  cudaError_t e = dsmla::launch_kv_cache_write(latent, num_rows, slots, kv_dtype, kv_pages,
                                               num_pages, err_flag,
                                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

int ds_indexer_logits(const void* q, const float* weights, const void* k_pages,
                      int64_t num_pages, const int32_t* block_table, int64_t bt_stride,
                      int64_t num_requests, const int32_t* row_req, const int32_t* lens,
                      int64_t num_rows, int num_heads, int head_dim, float* logits,
                      int64_t logits_stride, int32_t* err_flag, void* stream) {
  const char* fn = "ds_indexer_logits";
  if (num_heads != 16 && num_heads != 32 && num_heads != 64)
    return fail(DS_ERR_UNSUPPORTED, "%s: num_heads=%d is not supported; available: 16, 32, 64", fn,
                num_heads);
  if (head_dim != DS_INDEXER_HEAD_DIM)
    return fail(DS_ERR_UNSUPPORTED, "%s: head_dim=%d is not supported; available: 128", fn,
                head_dim);
  if (num_rows < 0) return fail(DS_ERR_SHAPE, "%s: num_rows=%lld is negative", fn, (long long)num_rows);
  if (num_pages < 1) return fail(DS_ERR_SHAPE, "%s: num_pages=%lld must be >= 1", fn, (long long)num_pages);
  if (num_pages > (int64_t)INT32_MAX / DS_PAGE_BLOCK_SIZE)
    return fail(DS_ERR_UNSUPPORTED, "%s: num_pages=%lld exceeds %lld (key rows are indexed in 32 bits)",
                fn, (long long)num_pages, (long long)(INT32_MAX / DS_PAGE_BLOCK_SIZE));
  if (bt_stride < 1) return fail(DS_ERR_SHAPE, "%s: bt_stride=%lld must be >= 1", fn, (long long)bt_stride);
  if (bt_stride > (int64_t)INT32_MAX / DS_PAGE_BLOCK_SIZE)
    return fail(DS_ERR_UNSUPPORTED, "%s: bt_stride=%lld is too large", fn, (long long)bt_stride);
  if (num_requests < 1)
    return fail(DS_ERR_SHAPE, "%s: num_requests=%lld must be >= 1", fn, (long long)num_requests);
  if (logits_stride < DS_PAGE_BLOCK_SIZE * bt_stride)
    return fail(DS_ERR_SHAPE,
                "%s: logits_stride=%lld must be >= 64 * bt_stride = %lld (a row scores up to that "
                "many positions)",
                fn, (long long)logits_stride, (long long)(DS_PAGE_BLOCK_SIZE * bt_stride));
  if (num_rows == 0) return ok();
  if (num_rows > (int64_t)INT32_MAX / dsmla::indexer_chunks(bt_stride))
    return fail(DS_ERR_UNSUPPORTED, "%s: num_rows=%lld is too large for one launch", fn,
                (long long)num_rows);
  struct {
    const void* p;
    const char* name;
    uintptr_t align;
  } ptrs[] = {{q, "q", 16},           {weights, "weights", 4}, {k_pages, "k_pages", 16},
              {block_table, "block_table", 4}, {lens, "lens", 4}, {logits, "logits", 4}};
  for (auto& x : ptrs) {
    if (x.p == nullptr) return fail(DS_ERR_NULL, "%s: %s is NULL", fn, x.name);
    if (!aligned(x.p, x.align))
      return fail(DS_ERR_ALIGN, "%s: %s must be %d-byte aligned", fn, x.name, (int)x.align);
  }
  if (row_req != nullptr && !aligned(row_req, 4))
    return fail(DS_ERR_ALIGN, "%s: row_req must be 4-byte aligned", fn);
  if (err_flag != nullptr && !aligned(err_flag, 4))
    return fail(DS_ERR_ALIGN, "%s: err_flag must be 4-byte aligned", fn);
  dsmla::IndexerArgs a;
  a.q = q;
  a.w = weights;
  a.k_pages = k_pages;
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.num_bt_rows = num_requests;
  a.row_req = row_req;
  a.lens = lens;
  a.R = num_rows;
  a.H = num_heads;
  a.logits = logits;
  a.logits_stride = logits_stride;
  a.err_flag = err_flag;
  cudaError_t e = dsmla::launch_indexer_logits(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DS_ERR_CUDA, "%s: launch failed: %s", fn, cudaGetErrorString(e));
  return ok();
}

size_t ds_sparse_mla_swa_workspace_size(int64_t num_rows, int num_heads, int k, int swa_width) {
  if (num_rows < 0) return 0;
  if (check_config("ds_sparse_mla_swa_workspace_size", num_heads, k, DS_PAGE_BLOCK_SIZE, DS_D_QK,
                   DS_D_V, DS_KV_BF16) != DS_OK)
    return 0;
  Window w;
  w.width = swa_width;
  if (check_window("ds_sparse_mla_swa_workspace_size", w) != DS_OK) return 0;
  return dsmla::attn_workspace_bytes(num_rows, num_heads, k, swa_width);
}

int ds_sparse_mla_decode_swa(const void* q, const void* kv_pages, int kv_dtype, int64_t num_pages,
                             const int32_t* block_table, int64_t bt_stride, const int32_t* idx,
                             const int32_t* lens, int k, const void* swa_pages,
                             int64_t swa_num_pages, const int32_t* swa_block_table,
                             int64_t swa_bt_stride, const int32_t* swa_idx,
                             const int32_t* swa_lens, int swa_width, const float* attn_sink,
                             int64_t num_rows, int num_heads, float scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t* err_flag,
                             void* stream) {
  Window w;
  w.pages = swa_pages;
  w.num_pages = swa_num_pages;
  w.block_table = swa_block_table;
  w.bt_stride = swa_bt_stride;
  w.idx = swa_idx;
  w.lens = swa_lens;
  w.width = swa_width;
  w.sink = attn_sink;
  return attention_common("ds_sparse_mla_decode_swa", q, kv_pages, kv_dtype, num_pages,
                          block_table, bt_stride, num_rows < 1 ? 1 : num_rows, nullptr, idx, lens,
                          num_rows, num_heads, k, scale, out, lse, workspace, workspace_bytes,
                          err_flag, stream, w);
}

}  // extern "C"
