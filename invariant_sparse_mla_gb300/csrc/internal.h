// Declarations shared by the host API (api.cu) and the kernel files.
#pragma once

#include <stdint.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <utility>

namespace dsmla {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); nullptr if the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || ptr == nullptr) {
      (void)cudaGetLastError();
      return nullptr;
    }
    f = reinterpret_cast<EncodeTiledFn>(ptr);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// Entries per attention tile and tiles per split. The split count of a call
// is ceil(k / kSplitEntries): a function of k alone, so a row's reduction
// order never depends on the batch.
constexpr int kTileEntries = 64;
constexpr int kSplitTiles = 8;
constexpr int kSplitEntries = kTileEntries * kSplitTiles;

inline int num_splits_for_k(int k) { return (k + kSplitEntries - 1) / kSplitEntries; }

// Splits of a call whose rows also attend to `k2` entries of a second list
// (a sliding window): as many as the top-k list alone needs, or more if the
// concatenation would put more than 768 entries (12 tiles) in one split. The
// concatenated tiles are spread evenly over them; with k2 = 0 this is the
// one-split-per-512-entries rule.
inline int num_splits_total(int k, int k2) {
  const int a = num_splits_for_k(k);
  const int b = (k + k2 + 767) / 768;
  return a > b ? a : b;
}

struct AttnArgs {
  const void* q;             // bf16 [R, H, 576]
  const void* kv;            // pool base
  int kv_dtype;              // 0 bf16, 1 fp8
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_bt_rows;       // rows of block_table
  const int32_t* row_req;    // nullptr: row r reads block-table row r
  const int32_t* idx;        // [R, k]
  const int32_t* lens;       // [R]
  int64_t R;
  int H;
  int k;
  float scale;
  void* out;                 // bf16 [R, H, 512]
  float* lse;                // [R, H]
  void* workspace;
  int32_t* err_flag;         // may be nullptr
  // Optional second entry list into a second pool (a sliding window), with
  // its own block table: k2 entries per row, 0 = none.
  const void* kv2 = nullptr;
  int64_t num_pages2 = 0;
  const int32_t* block_table2 = nullptr;
  int64_t bt_stride2 = 0;
  const int32_t* idx2 = nullptr;   // [R, k2]
  const int32_t* lens2 = nullptr;  // [R]
  int k2 = 0;
  const float* sink = nullptr;     // [H] per-head sink logits (natural log), may be nullptr
};

// Workspace layout of the attention path: partial O, m and l per split.
struct AttnWorkspace {
  uint16_t* part_o;  // [S, R, H, 512] bf16 bits
  float* part_m;  // [S, R, H]  (log2 domain, scale folded in)
  float* part_l;  // [S, R, H]
};

size_t attn_workspace_bytes(int64_t R, int H, int k, int k2 = 0);
AttnWorkspace attn_workspace_carve(void* base, int64_t R, int H, int k, int k2 = 0);

// Workspace bytes of the grid top-k for this shape (0: the shape takes a
// kernel that needs none). With a workspace of at least this size the grid
// kernel runs; without one, another kernel computes the same output.
size_t topk_workspace_bytes(int64_t rows, int64_t stride);
cudaError_t launch_topk(const float* scores, int64_t stride, int64_t rows, const int32_t* starts,
                        const int32_t* ends, int k, int32_t* out, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream);

cudaError_t launch_sparse_mla(const AttnArgs& a, cudaStream_t stream);

// The indexer scores of ds_indexer_logits.
struct IndexerArgs {
  const void* q;              // bf16 [R, H, 128]
  const float* w;             // [R, H]
  const void* k_pages;        // bf16 [num_pages, 64, 128]
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_bt_rows;
  const int32_t* row_req;     // nullptr: row r reads block-table row r
  const int32_t* lens;        // [R]
  int64_t R;
  int H;
  float* logits;              // [R, logits_stride]
  int64_t logits_stride;
  int32_t* err_flag;          // may be nullptr
};

cudaError_t launch_indexer_logits(const IndexerArgs& a, cudaStream_t stream);
int64_t indexer_chunks(int64_t bt_stride);   // CTAs per row of one call

cudaError_t launch_kv_cache_write(const void* latent, int64_t n, const int64_t* slots,
                                  int kv_dtype, void* pool, int64_t num_pages, int32_t* err,
                                  cudaStream_t stream);

// ---- programmatic dependent launch. Every kernel of this library is
// launched with the programmatic-stream-serialization attribute, so it may
// become resident while the previous kernel of the stream is still running.
// It calls pdl_wait() before its first global-memory access (that returns
// once the previous grid has finished and its writes are visible) and
// pdl_trigger() to let the next kernel of the stream start the same way.
// Neither changes what any kernel computes.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// cudaLaunchKernelEx with programmatic stream serialization and, when
// cluster_x > 1, a (cluster_x, 1, 1) thread-block cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

// Records a printf-style message for ds_last_error() on this host thread and
// returns `status`.
int report_error(int status, const char* fmt, ...);

// The device a launch on `stream` runs on. The runtime launches only into a
// stream of the current device (a stream of another device is refused), so
// this is the current device; the stream is not queried, since querying a
// stream is not allowed while it is being captured into a CUDA graph.
inline cudaError_t stream_device(cudaStream_t /*stream*/, int* dev) {
  return cudaGetDevice(dev);
}

// A kernel attribute (the dynamic shared memory limit) is a per-device
// setting: it is set once for each device the library launches on, the flag
// of device d recording that it was. Devices beyond the table are set on
// every launch.
struct PerDeviceOnce {
  static constexpr int kMaxDevices = 64;
  std::atomic<bool> done[kMaxDevices] = {};
};

template <typename Kernel>
cudaError_t set_max_dynamic_smem(PerDeviceOnce& once, int dev, Kernel kernel, int bytes) {
  const bool tracked = dev >= 0 && dev < PerDeviceOnce::kMaxDevices;
  if (tracked && once.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  int prev = 0;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return e;
  if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (prev != dev) {
    const cudaError_t e2 = cudaSetDevice(prev);
    if (e == cudaSuccess) e = e2;
  }
  if (e == cudaSuccess && tracked) once.done[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace dsmla
