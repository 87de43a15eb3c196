// Indexer scores (the "MQA logits" the top-k selects from) over a paged key
// cache: for query row r and context position s,
//
//   I[r, s] = sum_j w[r, j] * max(0, q[r, j, :] . k[s, :])
//
// with one shared key per position (MQA). "[SM120] Sync DS4 with upstream
// main + validated perf backports" routes these logits through their own
// kernel and sizes a paged-MQA warm-up; "[Bugfix] Make DSV4 sparse MLA work
// end-to-end ...", section "What is fixed", gives the indexer one signed
// context length per query token. The formula is the lightning indexer of
// the DeepSeek-V3.2-Exp technical report (the pages give none).
//
// One CTA scores 2048 positions of one row. Keys are read a page at a time
// (64 positions x 256 bytes, contiguous) by TMA tile copies into a 128-byte
// swizzled K-major tile of 128 positions; one tcgen05.mma chain per tile
// computes S^T = K Q^T (M = 128 positions, N = heads, K = 128 dims) into a
// TMEM accumulator, double buffered; four epilogue warps read one position
// each per lane, apply the clamp and the head weights in a fixed head order,
// and store the fp32 score. A score depends only on its row's q and w and on
// its key, so it is the same whatever else the batch holds.
//
// Warps 0-3: epilogue (and the Q copy); warp 4: TMA producer; warp 5: MMA
// issuer (and TMEM owner). Every wait is bounded; a timeout sets
// DS_DEVERR_TIMEOUT and the CTA winds down.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace dsmla {

namespace {

constexpr int kDim = 128;             // indexer head dimension
constexpr int kTilePos = 128;         // positions per tile (two pages)
constexpr int kChunkTiles = 16;       // tiles per CTA
constexpr int kChunk = kTilePos * kChunkTiles;
constexpr int kStages = 2;   // and two CTAs per SM
constexpr int kTileBytes = kTilePos * kDim * 2;     // 32 KB: two 64-dim column blocks
constexpr int kAtomBytes = kTilePos * 128;          // 16 KB: one column block of a tile
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kErrPage = 2, kErrRowReq = 4, kErrTimeout = 8;   // DS_DEVERR_* bits

template <int NH>
struct IxLayout {
  static constexpr int kQ = 0;                                   // 2 column blocks of NH rows
  static constexpr int kQBytes = 2 * NH * 128;
  static constexpr int kK = (kQBytes + 1023) / 1024 * 1024;       // kStages tiles
  static constexpr int kW = kK + kStages * kTileBytes;           // NH floats
  static constexpr int kBars = kW + 64 * 4;                      // 11 x u64
  static constexpr int kTmemSlot = kBars + 16 * 8;
  static constexpr int kEnd = kTmemSlot + 16;
  static constexpr int kSmemBytes = kEnd + 1024;                 // + alignment slack
  static constexpr uint32_t kTmemCols = 2 * NH < 32 ? 32u : (uint32_t)(2 * NH);
};

enum IxBar {
  kFull = 0,      // kStages: producer's expected bytes -> MMA issuer (tile landed)
  kEmpty = 2,     // kStages: MMA commit -> producer (stage free)
  kDFull = 4,     // 2: MMA commit -> epilogue (accumulator ready)
  kDEmpty = 6,    // 2: epilogue threads -> MMA issuer (accumulator read)
  kMmaDone = 8,   // MMA issuer's final drain
  kNumIxBars = 9
};
static_assert(kStages == 2, "barrier slots assume two stages");

struct IxParams {
  const __nv_bfloat16_raw* q;   // [R, NH, 128]
  const float* w;               // [R, NH]
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_bt_rows;
  const int32_t* row_req;       // nullptr: row r reads block-table row r
  const int32_t* lens;
  int64_t R;
  int chunks;                   // CTAs per row
  float* logits;
  int64_t logits_stride;
  int32_t* err;
};

// The key cache is read as a 2D tensor map [num_pages * 64, 128] bf16: box
// (0 or 64, page * 64) is 64 rows x 64 columns, 8 KB of 128-byte swizzled
// shared memory.
template <int NH>
__global__ void __launch_bounds__(kThreads) indexer_kernel(const __grid_constant__ CUtensorMap kmap,
                                                          const IxParams p) {
  using LY = IxLayout<NH>;
  extern __shared__ uint8_t ix_smem_raw[];
  // 1024-byte aligned base derived by pointer arithmetic on the shared
  // array, so accesses through it stay shared-memory accesses.
  uint8_t* smem = ix_smem_raw + ((1024u - (smem_u32(ix_smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::kBars);
  float* w_s = reinterpret_cast<float*>(smem + LY::kW);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::kTmemSlot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row = blockIdx.x / p.chunks;
  const int chunk = (int)(blockIdx.x % p.chunks);

  pdl_wait();
  pdl_trigger();

  // The row's scored length, clamped signed to the block table's reach.
  int64_t L = p.lens[row];
  if (L < 0) L = 0;
  if (L > 64 * p.bt_stride) L = 64 * p.bt_stride;
  int64_t req = row;
  if (p.row_req != nullptr) {
    req = p.row_req[row];
    if (req < 0 || req >= p.num_bt_rows) {
      if (tid == 0 && chunk == 0 && L > 0 && p.err != nullptr) atomicOr(p.err, kErrRowReq);
      L = 0;   // nothing of this row is scored
    }
  }
  const int64_t start = (int64_t)chunk * kChunk;
  if (start >= L) return;   // the same for every thread: nothing set up yet
  const int n = (int)((L - start < kChunk ? L - start : kChunk));
  const int ntiles = (n + kTilePos - 1) / kTilePos;
  const int32_t* bt_row = p.block_table + req * p.bt_stride;

  if (tid == 0) {
    for (int i = 0; i < kNumIxBars; ++i) {
      uint32_t count = 1u;
      if (i == kDEmpty || i == kDEmpty + 1) count = 128u;   // every epilogue thread read it
      mbar_init(&bars[i], count);
    }
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, LY::kTmemCols);
    tmem_relinquish();
  }
  if (tid < 128) {
    // Q of the row into two 128-byte swizzled K-major column blocks, and w.
    const uint8_t* qg = reinterpret_cast<const uint8_t*>(p.q + row * (int64_t)NH * kDim);
    for (int c = tid; c < NH * 16; c += 128) {
      const int h = c >> 4, ch = c & 15;   // 16-byte chunk ch of head h's 256 bytes
      const uint32_t dst = sbase + LY::kQ + (ch >> 3) * (NH * 128) + (h >> 3) * 1024 +
                           (h & 7) * 128 + (((ch & 7) ^ (h & 7)) << 4);
      cp_async_16(dst, qg + h * 256 + ch * 16, 16);
    }
    cp_async_commit();
    if (tid < NH) w_s[tid] = p.w[row * NH + tid];
    cp_async_wait_all();
    fence_proxy_async_smem();   // Q is read by the tensor core (async proxy)
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool failed = false;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kStages;
        if (t >= kStages && !mbar_wait(&bars[kEmpty + st], ((t / kStages) - 1) & 1)) {
          failed = true;
          break;
        }
        // The tile's two pages; a page outside the pool (or past the row) is
        // not copied, and the epilogue scores its positions -inf.
        const int64_t pos0 = start + (int64_t)t * kTilePos;
        int64_t pg[2];
        uint32_t tx = 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          pg[h] = -1;
          const int64_t pos = pos0 + 64 * h;
          if (pos < L) {
            const int64_t v = bt_row[pos >> 6];
            if (v >= 0 && v < p.num_pages) {
              pg[h] = v;
              tx += 2u * 8192u;
            }
          }
        }
        mbar_arrive_expect_tx(&bars[kFull + st], tx);
        const uint32_t dst = sbase + LY::kK + st * kTileBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (pg[h] < 0) continue;
          const int y = (int)(pg[h] * 64);
          tma_load_box(dst + h * 8192, &kmap, 0, y, &bars[kFull + st]);
          tma_load_box(dst + kAtomBytes + h * 8192, &kmap, 64, y, &bars[kFull + st]);
        }
        issued = t + 1;
      }
      // Every copy this thread started has landed before the CTA can exit.
      for (int t = issued - kStages > 0 ? issued - kStages : 0; t < issued; ++t)
        if (!mbar_wait(&bars[kFull + t % kStages], (t / kStages) & 1)) failed = true;
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kTilePos, NH, 0, 0);
      const uint64_t a_desc0 = make_sw128_desc(sbase + LY::kK, 16, 1024);
      const uint64_t b_desc0 = make_sw128_desc(sbase + LY::kQ, 16, 1024);
      for (int t = 0; t < ntiles && !failed; ++t) {
        const int st = t % kStages, db = t & 1;
        if (!mbar_wait(&bars[kFull + st], (t / kStages) & 1) ||
            (t >= 2 && !mbar_wait(&bars[kDEmpty + db], ((t >> 1) - 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint64_t a0 = a_desc0 + (uint64_t)((st * kTileBytes) >> 4);
        const uint32_t d = tmem + (uint32_t)(db * NH);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            mma_bf16_ss(d, a0 + ((a * kAtomBytes + k4 * 32) >> 4),
                        b_desc0 + ((a * NH * 128 + k4 * 32) >> 4), idesc, (a | k4) ? 1u : 0u);
          }
        }
        mma_commit(&bars[kEmpty + st]);
        mma_commit(&bars[kDFull + db]);
      }
      // Every MMA issued here has completed before TMEM is freed.
      mma_commit(&bars[kMmaDone]);
      if (!mbar_wait(&bars[kMmaDone], 0)) failed = true;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // TMEM lane 32 warp + lane is position m of the tile: this thread's
    // score reads NH columns of it.
    float* out_row = p.logits + row * p.logits_stride;
    int err_bits = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int db = t & 1;
      const bool ok = mbar_wait(&bars[kDFull + db], (t >> 1) & 1);
      if (named_bar_or(1, 128, !ok)) {
        failed = true;
        break;
      }
      tc_fence_after();
      float s[NH];
      const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(db * NH);
      if constexpr (NH == 64)
        tmem_ld64_sync(taddr, s);
      else if constexpr (NH == 32)
        tmem_ld32_sync(taddr, s);
      else
        tmem_ld16_sync(taddr, s);
      tc_fence_before();
      mbar_arrive(&bars[kDEmpty + db]);
      const int64_t pos = start + (int64_t)t * kTilePos + warp * 32 + lane;
      if (pos < L) {
        const int64_t v = bt_row[pos >> 6];
        float score;
        if (v >= 0 && v < p.num_pages) {
          score = 0.0f;
#pragma unroll
          for (int j = 0; j < NH; ++j) score = __fmaf_rn(w_s[j], fmaxf(s[j], 0.0f), score);
        } else {
          score = -INFINITY;
          err_bits |= kErrPage;
        }
        out_row[pos] = score;
      }
    }
    if (err_bits && p.err != nullptr) atomicOr(p.err, err_bits);
  }
  if (failed && p.err != nullptr) atomicOr(p.err, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, LY::kTmemCols);
}

template <int NH>
cudaError_t launch_indexer_nh(const CUtensorMap& map, const IxParams& ip, cudaStream_t stream) {
  using LY = IxLayout<NH>;
  static PerDeviceOnce attr_once;
  auto kern = indexer_kernel<NH>;
  int dev = 0;
  cudaError_t e = stream_device(stream, &dev);
  if (e == cudaSuccess) e = set_max_dynamic_smem(attr_once, dev, kern, LY::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)(ip.R * ip.chunks)), dim3(kThreads), LY::kSmemBytes,
                    stream, 1u, map, ip);
}

}  // namespace

cudaError_t launch_indexer_logits(const IndexerArgs& a, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)kDim, (cuuint64_t)(a.num_pages * 64)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kDim * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.k_pages), gdim, gstride,
          box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  IxParams ip;
  ip.q = reinterpret_cast<const __nv_bfloat16_raw*>(a.q);
  ip.w = a.w;
  ip.num_pages = a.num_pages;
  ip.block_table = a.block_table;
  ip.bt_stride = a.bt_stride;
  ip.num_bt_rows = a.num_bt_rows;
  ip.row_req = a.row_req;
  ip.lens = a.lens;
  ip.R = a.R;
  ip.chunks = (int)((64 * a.bt_stride + kChunk - 1) / kChunk);
  ip.logits = a.logits;
  ip.logits_stride = a.logits_stride;
  ip.err = a.err_flag;
  if (a.H == 64) return launch_indexer_nh<64>(map, ip, stream);
  if (a.H == 32) return launch_indexer_nh<32>(map, ip, stream);
  return launch_indexer_nh<16>(map, ip, stream);
}

int64_t indexer_chunks(int64_t bt_stride) { return (64 * bt_stride + kChunk - 1) / kChunk; }

}  // namespace dsmla
