// ds_sparse_mla_decode_noalloc: sparse MLA decode for callers that cannot
// hand the library a workspace.
//
// ds_sparse_mla_decode needs a caller-owned scratch buffer for its per-split
// partial results. Some callers cannot obtain one: code that runs under a
// memory manager that owns every byte of device memory and allows no side
// allocations, code that is in the middle of recording a CUDA graph (a plain
// cudaMalloc there is not part of the graph and breaks the capture), and
// latency-critical loops that must not pay for cudaMalloc's implicit device
// synchronisation. This entry point serves them: its scratch is a fixed
// file-scope device array in this library, so the call itself allocates
// nothing. The computation is exactly ds_sparse_mla_decode's; only where the
// partial results live differs.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "ds_sparse_mla.h"
#include "internal.h"

namespace {

// 32 MiB of scratch, e.g. enough for 62 decode rows at 64 heads and top-k
// 2048 (ds_sparse_mla_workspace_size() bytes). It is device memory of this
// library's module: each GPU holds it from the first time the module is
// loaded on that GPU until the process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Host code cannot use `g_decode_scratch` as a device address (on the host
// it names a stand-in object). Its device address is looked up with the
// device current and cached here once the lookup has succeeded; a failed
// lookup (for example one attempted during a stream capture) is not cached
// and is retried by the next call.
constexpr int kMaxDevices = 128;
std::atomic<void*> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" int ds_sparse_mla_decode_noalloc(const void* q, const void* kv_pages, int kv_dtype,
                                            int64_t num_pages, const int32_t* block_table,
                                            int64_t bt_stride, const int32_t* idx,
                                            const int32_t* lens, int64_t num_rows, int num_heads,
                                            int k, float scale, void* out, float* lse,
                                            int32_t* err_flag, void* stream) {
  const char* fn = "ds_sparse_mla_decode_noalloc";
  if (num_rows > 0) {
    const size_t need = ds_sparse_mla_workspace_size(num_rows, num_heads, k);
    if (need > kScratchBytes)
      return dsmla::report_error(DS_ERR_WORKSPACE,
                                 "%s: num_rows=%lld, num_heads=%d, topk=%d need %zu bytes of "
                                 "scratch, more than the built-in %zu; use ds_sparse_mla_decode "
                                 "with a caller-owned workspace",
                                 fn, (long long)num_rows, num_heads, k, need, kScratchBytes);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return dsmla::report_error(DS_ERR_CUDA, "%s: cudaGetDevice failed: %s", fn,
                               cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return dsmla::report_error(DS_ERR_UNSUPPORTED, "%s: device %d is beyond the %d supported", fn,
                               dev, kMaxDevices);
  void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (scratch == nullptr) {
    // Two threads may both get here on the first calls; both find the same
    // address.
    e = cudaGetSymbolAddress(&scratch, g_decode_scratch);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();   // not sticky: clear it so the next call can retry
      return dsmla::report_error(DS_ERR_CUDA, "%s: cudaGetSymbolAddress of the scratch failed: %s",
                                 fn, cudaGetErrorString(e));
    }
    g_scratch_addr[dev].store(scratch, std::memory_order_release);
  }
  return ds_sparse_mla_decode(q, kv_pages, kv_dtype, num_pages, block_table, bt_stride, idx, lens,
                              num_rows, num_heads, k, scale, out, lse, scratch, kScratchBytes,
                              err_flag, stream);
}
