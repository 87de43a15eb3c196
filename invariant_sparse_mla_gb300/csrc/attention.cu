// Sparse MLA attention over a paged latent KV cache, for decode and prefill.
//
// Computes, per query row and head, out = softmax(scale * q K^T) V over the
// row's selected entries, V being the first 512 of the 576 latent dims of the
// same rows ("[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for
// 0-diff RL", section "Sparse MLA and FlashMLA": decode gathers the selected
// KV and runs sparse attention; prefill handles each token on its own). The
// page lookup of a context position is page = block_table[row][pos / 64],
// slot = pos % 64 ("[Bugfix] Make DSV4 sparse MLA work end-to-end ...",
// section "What is fixed").
//
// Work decomposition (fixed by k alone, never by the batch): a CTA owns one
// (query row, split of 512 entries, group of <= 64 heads). A fixed-order
// combine kernel merges the splits. Within a CTA:
//
//   loader warps        gather 64-entry tiles of 1152-byte bf16 rows into a
//                       128-byte-swizzled shared-memory tile (FP8 rows are
//                       dequantised to bf16 on the way), double buffered:
//                       warps 4-11; bf16 copies arrive on the tile's
//                       barrier by themselves when they land;
//   MMA warps           the next three warps; one thread each issues tcgen05
//                       MMAs (a single thread can issue one MMA per ~54
//                       cycles, so three issuers keep the tensor pipe fed):
//                         QK issuers: S = Q K^T M=64 (heads), N=64, over
//                                     dims 0-319 and 320-575 into two TMEM
//                                     accumulators summed by the softmax
//                         PV issuer:  O^T += V^T P^T M=128 (dv block), N=heads, K=64
//                       The same swizzled tile is the K-major B operand of
//                       the first and the MN-major A operand of the second.
//   softmax warps 0-3   copy Q in the prologue, then read S from TMEM (one
//                       head per TMEM lane), keep a running max m and sum l
//                       per head, write P (bf16) over the rope block of the
//                       tile's own stage, and rescale O^T in TMEM only when
//                       a head's max grows by more than 2^8 (exact: p <= 256
//                       is kept relative to the stored max).
//
// The QK MMA has M = 64: for head groups smaller than 64, the A descriptor
// simply continues into the following smem, and those D rows are never read
// (a D row depends only on its own A row). Every wait is bounded; a timeout
// sets DS_DEVERR_TIMEOUT and the CTA winds down, frees its TMEM and exits.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace dsmla {

namespace {

constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kRowBytesBf16 = kD * 2;                 // 1152
constexpr int kRowBytesFp8 = 656;
constexpr int kChunks = kRowBytesBf16 / 16;           // 72 16-byte chunks per bf16 row
constexpr int kTile = kTileEntries;                   // 64 entries per tile
constexpr int kStages = 2;                            // KV tile ring
constexpr int kStageBytes = kTile * kRowBytesBf16;    // 73728
constexpr int kAtomStride = kTile * 128;              // bytes between 64-dim column blocks
constexpr int kSCols = kTile;                         // TMEM columns of one S buffer
constexpr int kSbCol = 2 * kSCols;                    // second QK accumulator (2 buffers)
constexpr int kOCol = 4 * kSCols;                     // first TMEM column of O^T
constexpr int kMaxSplitTiles = 12;                    // tiles one split may hold
// Largest split count: top-k 2048 (4 splits of 512), or 2048 + 512 window
// entries at most 768 per split (4).
constexpr int kMaxSplits = 4;
static_assert((2048 + kSplitEntries - 1) / kSplitEntries <= kMaxSplits &&
                  (2048 + 512 + 767) / 768 <= kMaxSplits,
              "every split of the largest call is merged");
constexpr int kQkSplitAtom = 5;                       // QK column blocks [0,5) -> S_a, [5,9) -> S_b
constexpr float kRescaleThreshold = 8.0f;             // log2 units
// P(t) is written over the rope column block of tile t's own stage: QK(t) is
// its only reader and has completed once S(t) is ready, PV(t) never reads it,
// and the stage is refilled only after PV(t). So P is double-buffered with
// the stages at no cost in shared memory.
constexpr int kPAtom = 8 * kAtomStride;

// Warp roles. Warps 0-3 run the softmax (warp w reads the TMEM lane
// quadrant w, i.e. heads 16 w .. 16 w + 15); the next kLoaderWarps warps
// load; then come one QK issuer, the PV issuer and the second QK issuer.
// Loader warp pw fills rows kRowsPerWarp * pw .. + kRowsPerWarp - 1 of every
// tile; for the page lookups, lane l owns row kRowsPerWarp * pw +
// (l % kRowsPerWarp) of tiles l / kRowsPerWarp + kTileGroups * i,
// i = 0 .. kSlots - 1. (Eight softmax warps, or four loader warps, were
// measured no faster.)
template <bool FP8>
struct Roles {
  static constexpr int kSoftmaxWarps = 4;
  static constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
  static constexpr int kLoaderWarps = 8;
  static constexpr int kLoaderThreads = 32 * kLoaderWarps;
  static constexpr int kRowsPerWarp = 64 / kLoaderWarps;
  static constexpr int kTileGroups = 32 / kRowsPerWarp;
  static constexpr int kSlots = kMaxSplitTiles / kTileGroups;
  static constexpr int kQkA = kSoftmaxWarps + kLoaderWarps;       // also allocates TMEM
  static constexpr int kPv = kQkA + 1;
  static constexpr int kQkB = kQkA + 2;
  static constexpr int kThreads = 32 * (kQkA + 3);
  static_assert(kLoaderWarps == 4 || kLoaderWarps == 8, "loader warps");
};

// The loader lane's KV row of slot `sel` (select chain: no local memory).
template <int N>
__device__ __forceinline__ int slot_row(const int (&grow)[N], int sel) {
  int r = grow[0];
#pragma unroll
  for (int i = 1; i < N; ++i) r = sel == i ? grow[i] : r;
  return r;
}

// Error bits (match DS_DEVERR_* in the public header).
constexpr int kErrIdx = 1, kErrPage = 2, kErrRowReq = 4, kErrTimeout = 8;

template <int HG>
struct Layout {
  static constexpr int kQBytes = HG * kRowBytesBf16;
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kQBytes;                    // kStages x kStageBytes
  static constexpr int kBars = kKV + kStages * kStageBytes;   // 16 x u64
  static constexpr int kMask = kBars + 16 * 8;                // kMaxSplitTiles x u64
  static constexpr int kAlpha = kMask + kMaxSplitTiles * 8;   // 2 x 64 floats
  static constexpr int kTmemSlot = kAlpha + 2 * 64 * 4;       // u32
  static constexpr int kNeff = kTmemSlot + 4;                 // int
  static constexpr int kEnd = kNeff + 12;
  static constexpr int kSmemBytes = kEnd + 1024;              // + alignment slack
  static constexpr uint32_t kTmemCols = 512u;   // S_a, S_b (2 buffers each) + O^T
};

// Barrier slots. Every barrier waited on by parity is only ever waited on
// for a phase that cannot be overtaken by the next one, so the parity test
// is unambiguous.
enum Bar {
  kQFull = 0,      // Q landed -> QK issuers (bf16: one expect-tx arrival; FP8: one per softmax thread)
  kKvFull = 1,     // 2: loader threads -> QK issuers (tile landed)
  kKvEmpty = 3,    // 2: PV issuer commit -> loaders (stage free), softmax (O^T holds the tile)
  kSFull = 5,      // 2: both QK issuers' commits -> softmax (S ready)
  kPFull = 7,      // 2: softmax threads -> PV issuer, QK issuers (P written, S read)
  kMmaDone = 9,    // 3: each issuer's final drain
  kNumBars = 12
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- The fixed-order merge of one (row, head)'s splits (A9), in log2 units
// (the sink logit s enters as s log2 e):
// M = max(m_s, sink), L = sum 2^(m_s - M) l_s + 2^(sink - M),
// out = sum 2^(m_s - M) O_s / L, lse = (M + log2 L) ln 2, splits in order
// s = 0, 1, ...; a split with m = -inf is empty and skipped (its O is never
// read); a NaN m (a split that gave up on a wait) makes the result NaN.
struct MergeWeights {
  float w[kMaxSplits];   // 2^(m_s - M); 0 for skipped splits
  float inv;             // 1 / L
  float lse;             // natural log
  uint32_t skip;         // bit s: split s is empty
  int state;             // 0: merged; 1: no entry (out 0, lse -inf); 2: gave up (NaN)
};

__device__ __forceinline__ MergeWeights merge_weights(const float (&ms)[kMaxSplits],
                                                      const float (&ls)[kMaxSplits], float sl) {
  MergeWeights r;
  float M = sl;
  bool gave_up = false;
  r.skip = 0u;
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    M = fmaxf(M, ms[s]);
    gave_up |= ms[s] != ms[s];
    r.w[s] = 0.0f;
    if (ms[s] == -INFINITY) r.skip |= 1u << s;
  }
  r.inv = 0.0f;
  r.lse = -INFINITY;
  r.state = gave_up ? 2 : (M == -INFINITY ? 1 : 0);
  if (r.state != 0) return r;
  float L = 0.0f;
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    if ((r.skip >> s) & 1u) continue;
    r.w[s] = ex2(ms[s] - M);
    L = __fmaf_rn(r.w[s], ls[s], L);
  }
  if (sl != -INFINITY) L = __fadd_rn(L, ex2(sl - M));
  r.inv = __fdiv_rn(1.0f, L);
  r.lse = __fmul_rn(__fadd_rn(M, log2f(L)), 0.69314718055994530942f);
  return r;
}

// One output element from the splits' unnormalised partial values o[s].
__device__ __forceinline__ float merge_value(const MergeWeights& mw, const float (&o)[kMaxSplits]) {
  float acc = 0.0f;
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s)
    if (!((mw.skip >> s) & 1u)) acc = __fmaf_rn(mw.w[s], o[s], acc);
  return __fmul_rn(acc, mw.inv);
}

// Byte offset of 16-byte chunk `c` (of 72) of tile row `r` in a 128-byte
// swizzled K-major tile whose 64-dim column blocks are `atom_stride` apart.
__device__ __forceinline__ uint32_t swz_off(int r, int c, int atom_stride) {
  return (uint32_t)((c >> 3) * atom_stride + (r >> 3) * 1024 + (r & 7) * 128 +
                    (((c & 7) ^ (r & 7)) << 4));
}

// N (16, 32 or 64) consecutive TMEM columns of this warp's lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v) {
  if constexpr (N == 64)
    tmem_ld64_sync(taddr, v);
  else if constexpr (N == 32)
    tmem_ld32_sync(taddr, v);
  else
    tmem_ld16_sync(taddr, v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 8 E4M3 codes (little-endian in `lo`, `hi`) times `scale` -> 8 bf16 (uint4).
__device__ __forceinline__ uint4 dequant8(uint32_t lo, uint32_t hi, float scale) {
  float f[8];
  const uint32_t w[2] = {lo, hi};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i] >> (16 * j)) & 0xFFFFu);
      const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const __half2 hh = *reinterpret_cast<const __half2*>(&h);
      const float2 ff = __half22float2(hh);
      f[i * 4 + j * 2 + 0] = ff.x * scale;
      f[i * 4 + j * 2 + 1] = ff.y * scale;
    }
  }
  uint4 r;
  r.x = pack_bf16x2(f[0], f[1]);
  r.y = pack_bf16x2(f[2], f[3]);
  r.z = pack_bf16x2(f[4], f[5]);
  r.w = pack_bf16x2(f[6], f[7]);
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Requests every 128-byte line of [base, base + bytes) into L2 (or into this
// SM's L1), thread `first` of `step` threads taking every step-th line. A
// line that holds a byte of the range lies in a mapped page, so no request
// leaves the range's pages.
template <bool kL1>
__device__ __forceinline__ void prefetch_lines(const void* base, int64_t bytes, int first,
                                               int step) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  const uintptr_t end = b + (uintptr_t)bytes;
  for (uintptr_t a = (b & ~uintptr_t(127)) + (uintptr_t)first * 128u; a < end;
       a += (uintptr_t)step * 128u) {
    if constexpr (kL1)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a) : "memory");
    else
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a) : "memory");
  }
}

struct KParams {
  const __nv_bfloat16* q;
  const uint8_t* kv;
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_bt_rows;
  const int32_t* row_req;
  const int32_t* idx;
  const int32_t* lens;
  int64_t R;
  int H;
  int k;
  int num_splits;
  int num_hg;
  float scale_log2;
  // Second entry list (sliding window), read through its own pool and block
  // table; its tiles follow the top-k tiles in the concatenated list.
  const uint8_t* kv2;
  int64_t num_pages2;
  const int32_t* block_table2;
  int64_t bt_stride2;
  const int32_t* idx2;
  const int32_t* lens2;
  int k2;
  uint16_t* part_o;   // bf16 bits
  float* part_m;
  float* part_l;
  int32_t* err;
};

// `qmap` (bf16 pools only): q as a 2D tensor map [R * H rows, 576 bf16],
// boxes of 64 columns x HG rows in the 128-byte swizzle (one box is one
// K-major atom of the CTA's Q tile).
template <int HG, bool FP8>
__global__ void __launch_bounds__(Roles<FP8>::kThreads, 1) sparse_mla_split_kernel(
    const __grid_constant__ CUtensorMap qmap, const KParams p) {
  using LY = Layout<HG>;
  using RL = Roles<FP8>;
  constexpr int RW = RL::kRowsPerWarp, TG = RL::kTileGroups;
  constexpr int SWT = RL::kSoftmaxThreads;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled tiles, derived from the shared
  // array by pointer arithmetic (not through an integer), so every access
  // below stays a shared-memory access rather than a generic one.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::kBars);
  uint32_t* vmask = reinterpret_cast<uint32_t*>(smem + LY::kMask);   // 2 words per tile
  float* alpha_s = reinterpret_cast<float*>(smem + LY::kAlpha);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::kTmemSlot);
  int* neff_s = reinterpret_cast<int*>(smem + LY::kNeff);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // The loader warps load every KV tile together (see Roles); the softmax
  // warps copy Q.
  const bool producer = warp >= RL::kSoftmaxWarps && warp < RL::kSoftmaxWarps + RL::kLoaderWarps;
  const int pw = warp - RL::kSoftmaxWarps;
  const int lgroup = lane / RW, lrow = lane % RW;   // tile group and row of this lane

  int64_t bid = blockIdx.x;
  const int hg = (int)(bid % p.num_hg);
  bid /= p.num_hg;
  const int split = (int)(bid % p.num_splits);
  const int64_t row = bid / p.num_splits;

  // ---- set-up that reads no global memory, done while the previous kernel
  // of the stream may still run: thread 0 sets up the barriers, one warp
  // allocates TMEM, and the loaders ask L2 for this CTA's Q tile, (for
  // decode) its block-table row, its row length and its top-k entries. L2 is
  // where every write lands, so a line requested before the previous kernel
  // wrote it is never seen stale.
  if (tid == 0) {
    *neff_s = 0;
    for (int i = 0; i < kNumBars; ++i) {
      // q_full and p_full: one arrival per softmax thread; kv_full: one per
      // loader thread; s_full: one tcgen05.commit from each QK issuer; the
      // rest: one tcgen05.commit.
      uint32_t count = 1u;
      if (i == kPFull || i == kPFull + 1) count = (uint32_t)SWT;
      if (i == kQFull && FP8) count = (uint32_t)SWT;
      if (i >= kKvFull && i < kKvFull + kStages) count = RL::kLoaderThreads;
      if (i == kSFull || i == kSFull + 1) count = 2u;
      mbar_init(&bars[i], count);
    }
    mbar_fence_init();
  }
  if (warp == RL::kQkA) {
    tmem_alloc(tmem_slot, LY::kTmemCols);
    tmem_relinquish();
  }
  // The concatenated entry list [top-k list || second list] in 64-entry
  // tiles: tile u < T1 holds top-k entries 64u .. 64u + 63 (main pool), tile
  // u >= T1 entries 64(u - T1) .. of the second list (its own pool). Split s
  // owns tiles [floor(s T / S), floor((s + 1) T / S)): a function of k and
  // the second list's width alone, never of the batch.
  const int T1 = p.k / kTile;
  const int T = T1 + p.k2 / kTile;
  const int u0 = (int)((int64_t)split * T / p.num_splits);
  const int ntiles = (int)((int64_t)(split + 1) * T / p.num_splits) - u0;
  if (producer) {
    prefetch_lines<false>(p.q + ((int64_t)row * p.H + (int64_t)hg * HG) * kD,
                          HG * kRowBytesBf16, tid - SWT, RL::kLoaderThreads);
    if (p.row_req == nullptr)
      prefetch_lines<false>(p.block_table + row * p.bt_stride, p.bt_stride * 4, tid - SWT,
                            RL::kLoaderThreads);
    // The split's top-k entries, usually written by the kernel still running
    // ahead of this one: the request warms L2 and this SM's address
    // translation for the first reads after the wait.
    const int u_end = min(u0 + ntiles, T1);
    if (u_end > u0)
      prefetch_lines<false>(p.idx + row * (int64_t)p.k + u0 * kTile,
                            (int64_t)(u_end - u0) * kTile * 4, tid - SWT, RL::kLoaderThreads);
    prefetch_lines<false>(p.lens + row, 4, tid - SWT, RL::kLoaderThreads);
  }
  pdl_wait();
  pdl_trigger();

  int64_t bt_row = row;
  bool row_ok = true;
  if (p.row_req != nullptr) {
    bt_row = p.row_req[row];
    row_ok = bt_row >= 0 && bt_row < p.num_bt_rows;
  }
  int64_t len1 = p.lens[row], len2 = p.k2 > 0 ? p.lens2[row] : 0;
  if (len1 < 0) len1 = 0;
  if (len2 < 0) len2 = 0;
  const int32_t* idx_row1 = p.idx + row * (int64_t)p.k;
  const int32_t* idx_row2 = p.k2 > 0 ? p.idx2 + row * (int64_t)p.k2 : nullptr;
  // Pool of local tile t (tiles never straddle the two lists).
  auto tile_kv = [&](int t) { return u0 + t >= T1 ? p.kv2 : p.kv; };
  const int64_t part_base = ((int64_t)split * p.R + row) * p.H + (int64_t)hg * HG;

  // ---- prologue (one block-wide barrier): producers read their idx
  // entries, resolve pages and start the tile 0 and 1 copies; the softmax
  // warps copy Q.
  __syncthreads();   // barriers, TMEM and neff_s = 0 are visible before use
  if constexpr (!FP8) {
    if (tid == 0) {
      // Q by nine box copies (one per 64 columns), laid out by the copy
      // engine in the swizzle the tensor cores read, through its own path:
      // the loader warps' 16-byte copies of tiles 0 and 1 never queue behind
      // Q's.
      mbar_arrive_expect_tx(&bars[kQFull], (uint32_t)(HG * kRowBytesBf16));
      const int y = (int)(row * p.H + (int64_t)hg * HG);
#pragma unroll 1
      for (int j = 0; j < kChunks / 8; ++j)
        tma_load_box(sbase + LY::kQ + j * (HG * 128), &qmap, 64 * j, y, &bars[kQFull]);
    }
  } else if (tid < SWT) {
    // FP8: the loaders fill tiles through registers, so nothing queues
    // behind Q's 16-byte copies; the softmax warps, idle until the first S,
    // copy it (measured faster here than the box copies).
    const __nv_bfloat16* qg = p.q + ((int64_t)row * p.H + (int64_t)hg * HG) * kD;
    for (int c = tid; c < HG * kChunks; c += SWT) {
      const int h = c / kChunks, ch = c - h * kChunks;
      cp_async_16(sbase + LY::kQ + swz_off(h, ch, HG * 128), qg + (int64_t)h * kD + ch * 8, 16);
    }
    cp_async_commit();
    cp_async_mbar_arrive_noinc(&bars[kQFull]);
  }
  // KV row (page * 64 + slot) of each owned entry, -1 = skip: slot i is
  // tile lgroup + TG i, row RW pw + lrow.
  int grow[RL::kSlots];
#pragma unroll
  for (int i = 0; i < RL::kSlots; ++i) grow[i] = -1;
  // bf16 pools: loader warp pw copies rows RW pw .. RW pw + RW - 1 of tile t
  // into the stage at stage_base, 16-byte cp.async into the 128-byte
  // swizzled layout; entries that are not valid copy zeros.
  auto copy_tile_bf16 = [&](int t, uint32_t stage_base) {
    const int gi = slot_row(grow, t / TG);
    const int src_lane0 = (t % TG) * RW;
#pragma unroll 4
    for (int rr = 0; rr < RW; ++rr) {
      const int64_t g = __shfl_sync(0xffffffffu, gi, src_lane0 + rr);
      const uint8_t* src = tile_kv(t) + (g >= 0 ? g : 0) * (int64_t)kRowBytesBf16;
      const uint32_t nbytes = g >= 0 ? 16u : 0u;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const int c = lane + 32 * j;
        if (c < kChunks)
          cp_async_16(stage_base + swz_off(RW * pw + rr, c, kAtomStride), src + c * 16, nbytes);
      }
    }
    cp_async_commit();
  };
  if (producer) {
    int pos[RL::kSlots];
    bool sec[RL::kSlots];   // slot's tile is in the second list
#pragma unroll
    for (int i = 0; i < RL::kSlots; ++i) {
      pos[i] = -1;
      sec[i] = false;
    }
    int last = 0;
#pragma unroll
    for (int i = 0; i < RL::kSlots; ++i) {
      const int t = lgroup + TG * i;
      if (t < ntiles) {
        const int u = u0 + t;
        sec[i] = u >= T1;
        pos[i] = sec[i] ? idx_row2[(u - T1) * kTile + RW * pw + lrow]
                        : idx_row1[u * kTile + RW * pw + lrow];
      }
    }
    // While the entries are in flight, bring the block-table row(s) into
    // this SM's L1 (after the wait on the previous kernel, so nothing stale
    // is cached): the page lookups below then hit L1 instead of making a
    // second round trip to L2.
    if (row_ok) {
      prefetch_lines<true>(p.block_table + bt_row * p.bt_stride, p.bt_stride * 4, tid - SWT,
                           RL::kLoaderThreads);
      if (p.k2 > 0)
        prefetch_lines<true>(p.block_table2 + bt_row * p.bt_stride2, p.bt_stride2 * 4,
                             tid - SWT, RL::kLoaderThreads);
    }
#pragma unroll
    for (int i = 0; i < RL::kSlots; ++i)
      if (pos[i] != -1) last = lgroup + TG * i + 1;
    // All block-table reads go out before any is used: one round trip.
    int64_t page[RL::kSlots];
#pragma unroll
    for (int i = 0; i < RL::kSlots; ++i) {
      const int ps = pos[i];
      const int64_t len = sec[i] ? len2 : len1;
      const int64_t bts = sec[i] ? p.bt_stride2 : p.bt_stride;
      page[i] = -2;   // no lookup
      if (ps >= 0 && (int64_t)ps < len && row_ok && (int64_t)(ps >> 6) < bts)
        page[i] = (sec[i] ? p.block_table2 : p.block_table)[bt_row * bts + (ps >> 6)];
    }
    int err_bits = 0;
#pragma unroll
    for (int i = 0; i < RL::kSlots; ++i) {
      const int ps = pos[i];
      const int64_t len = sec[i] ? len2 : len1;
      bool valid = false;
      if (ps >= 0 && (int64_t)ps < len && row_ok) {
        if (page[i] >= 0 && page[i] < (sec[i] ? p.num_pages2 : p.num_pages)) {
          grow[i] = (int)(page[i] * 64 + (ps & 63));
          valid = true;
        } else {
          err_bits |= kErrPage;   // outside the pool, or beyond the block table
        }
      } else if (ps != -1 && row_ok) {
        err_bits |= kErrIdx;
      }
      const uint32_t ballot = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) {
        // Lanes RW g .. RW g + RW - 1 hold rows RW pw .. of tile g + TG i:
        // bits RW pw .. RW pw + RW - 1 of that tile's 64-bit row mask.
#pragma unroll
        for (int g = 0; g < TG; ++g) {
          const uint32_t piece = (ballot >> (RW * g)) & ((1u << RW) - 1u);
          if constexpr (RW == 16)
            reinterpret_cast<uint16_t*>(vmask + 2 * (g + TG * i))[pw] = (uint16_t)piece;
          else
            reinterpret_cast<uint8_t*>(vmask + 2 * (g + TG * i))[pw] = (uint8_t)piece;
        }
      }
    }
    // Start tile 0 (stage 0) and tile 1 (stage 1) right away, before the
    // block-wide barrier. Entries that are not valid copy zeros, so this is
    // harmless when the split turns out to be short. Each arrival tracks
    // every earlier copy of the thread, so tile 0 signals its barrier before
    // tile 1 is issued.
    if constexpr (!FP8) {
      copy_tile_bf16(0, sbase + LY::kKV);
      cp_async_mbar_arrive_noinc(&bars[kKvFull]);
      if (ntiles > 1) {   // a one-tile split has no tile 1 (nor its pool)
        copy_tile_bf16(1, sbase + LY::kKV + kStageBytes);
        cp_async_mbar_arrive_noinc(&bars[kKvFull + 1]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (lane == 0 && last > 0) atomicMax(neff_s, last);
    if (err_bits && p.err != nullptr) atomicOr(p.err, err_bits);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_eff = row_ok ? *neff_s : 0;
  if (!row_ok && tid == 0 && p.err != nullptr) atomicOr(p.err, kErrRowReq);

  bool failed = false;
  if (n_eff == 0) {
    // Nothing to attend to in this split: an empty partial.
    if (producer || (FP8 && tid < SWT)) cp_async_wait_all();  // copies land before the CTA exits
    if (tid < HG) {
      p.part_m[part_base + tid] = -INFINITY;
      p.part_l[part_base + tid] = 0.0f;
    }
  } else if (producer) {
    // ------------------------------------------------------------ producers
    // All loader warps fill each tile in turn (RW rows each) into stage t & 1.
    // bf16: the copies arrive on the tile's barrier by themselves when they
    // land (cp.async.mbarrier.arrive), so a loader moves on to the next stage
    // as soon as it is free and up to two tiles are in flight; the tensor-core
    // issuers fence the landed tiles for the async proxy. FP8: the loaders
    // dequantise through registers, store, fence and arrive. Nothing is
    // requested into L2 ahead of the copies: measured on this gather
    // pattern, bulk or per-line L2 prefetches of later tiles slowed the
    // tile fills down rather than hiding their latency.
    // Rows of tile u are held by lanes with lgroup == u % TG, slot u / TG.
#pragma unroll 1
    for (int t = 0; t < n_eff; ++t) {
      const int stage = t & 1;
      const uint32_t stage_base = sbase + LY::kKV + stage * kStageBytes;
      const bool ok = t < 2 || mbar_wait(&bars[kKvEmpty + stage], ((t >> 1) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
      if constexpr (!FP8) {
        if (t >= 2) {   // tiles 0 and 1 went out in the prologue
          copy_tile_bf16(t, stage_base);
          cp_async_mbar_arrive_noinc(&bars[kKvFull + stage]);
        }
      } else {
        const int gi = slot_row(grow, t / TG);
        const int src_lane0 = (t % TG) * RW;
#pragma unroll 1
        for (int r0 = 0; r0 < RW; r0 += 8) {
          uint2 codes[8][2];
          float scl[8][2];
          uint4 rope[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int64_t g = __shfl_sync(0xffffffffu, gi, src_lane0 + r0 + u);
            const uint8_t* src = tile_kv(t) + (g >= 0 ? g : 0) * (int64_t)kRowBytesFp8;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int c = lane + 32 * j;  // latent output chunk 0..63
              codes[u][j] = make_uint2(0u, 0u);
              scl[u][j] = 0.0f;
              if (g >= 0) {
                codes[u][j] = *reinterpret_cast<const uint2*>(src + c * 8);
                scl[u][j] = *reinterpret_cast<const float*>(src + 512 + (c >> 4) * 4);
              }
            }
            rope[u] = make_uint4(0u, 0u, 0u, 0u);
            if (lane < 8 && g >= 0)
              rope[u] = *reinterpret_cast<const uint4*>(src + 528 + lane * 16);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int tr = RW * pw + r0 + u;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int c = lane + 32 * j;
              st_shared_v4(stage_base + swz_off(tr, c, kAtomStride),
                           dequant8(codes[u][j].x, codes[u][j].y, scl[u][j]));
            }
            if (lane < 8) st_shared_v4(stage_base + swz_off(tr, 64 + lane, kAtomStride), rope[u]);
          }
        }
      }
      if constexpr (FP8) {
        fence_proxy_async_smem();
        mbar_arrive(&bars[kKvFull + stage]);
      }
    }
    cp_async_wait_all();
  } else if (warp == RL::kQkA || warp == RL::kQkB) {
    // ------------------------------------------------------------ QK issuers
    // The first issuer accumulates column blocks [0, 5) of QK(t) into S_a,
    // the second blocks [5, 9) into S_b. QK(t) needs tile t landed and its S buffers
    // free: P(t-2) written means softmax(t-2) has read S(t-2). Descriptors
    // are precomputed; each issuer's MMAs of a tile go back to back.
    if (lane == 0) {
      const int a_lo = warp == RL::kQkA ? 0 : kQkSplitAtom;
      const int a_hi = warp == RL::kQkA ? kQkSplitAtom : kD / 64;
      const uint32_t s_col = warp == RL::kQkA ? 0u : (uint32_t)kSbCol;
      constexpr uint32_t idesc_qk = make_idesc_bf16(64, kTile, 0, 0);
      const uint64_t q_desc = make_sw128_desc(sbase + LY::kQ, 16, 1024);
      const uint64_t kv_desc0 = make_sw128_desc(sbase + LY::kKV, 16, 1024);
      if (!mbar_wait(&bars[kQFull], 0)) failed = true;
      for (int t = 0; t < n_eff && !failed; ++t) {
        const int sb = t & 1;
        if (!mbar_wait(&bars[kKvFull + sb], (t >> 1) & 1) ||
            (t >= 2 && !mbar_wait(&bars[kPFull + sb], ((t >> 1) - 1) & 1))) {
          failed = true;
          break;
        }
        // The tile (and, for FP8, Q) landed through generic-proxy writes:
        // order them before the tensor core's async-proxy reads (bf16 Q came
        // by the copy engine, itself an async-proxy write).
        fence_proxy_async_smem();
        tc_fence_after();
        const uint64_t b0 = kv_desc0 + (uint64_t)((sb * kStageBytes) >> 4);
        const uint32_t d = tmem + s_col + sb * kSCols;
#pragma unroll 1
        for (int ka = a_lo; ka < a_hi; ++ka) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t off = k4 * 32;
            mma_bf16_ss(d, q_desc + ((ka * (HG * 128) + off) >> 4),
                        b0 + ((ka * kAtomStride + off) >> 4), idesc_qk,
                        (ka > a_lo || k4 > 0) ? 1u : 0u);
          }
        }
        mma_commit(&bars[kSFull + sb]);
      }
      const int done_bar = kMmaDone + (warp == RL::kQkA ? 0 : 2);
      mma_commit(&bars[done_bar]);
      mbar_wait(&bars[done_bar], 0);
    }
    __syncwarp();
  } else if (warp == RL::kPv) {
    // ------------------------------------------------------------ PV issuer
    // PV(t) needs P(t); its completion frees the KV stage and lets softmax
    // overwrite P and rescale O^T.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, HG, 1, 0);
      const uint64_t p_desc0 = make_sw128_desc(sbase + LY::kKV + kPAtom, 16, 1024);
      const uint64_t v_desc0 = make_sw128_desc(sbase + LY::kKV, kAtomStride, 1024);
      for (int t = 0; t < n_eff && !failed; ++t) {
        const int sb = t & 1;
        if (!mbar_wait(&bars[kPFull + sb], (t >> 1) & 1)) {
          failed = true;
          break;
        }
        fence_proxy_async_smem();   // V landed through cp.async
        tc_fence_after();
        const uint64_t a0 = v_desc0 + (uint64_t)((sb * kStageBytes) >> 4);
        const uint64_t p0 = p_desc0 + (uint64_t)((sb * kStageBytes) >> 4);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_bf16_ss(tmem + kOCol + b * HG, a0 + (((2 * b * kAtomStride) + kk * 2048) >> 4),
                        p0 + ((kk * 32) >> 4), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&bars[kKvEmpty + sb]);
      }
      mma_commit(&bars[kMmaDone + 1]);
      mbar_wait(&bars[kMmaDone + 1], 0);
    }
    __syncwarp();
  } else if (warp < RL::kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    // S was computed with M = 64: head h sits in TMEM lane 32*(h/16) + h%16,
    // so warp qd holds heads 16 qd .. 16 qd + 15 (its lanes 0-15). With the
    // 16x32bx2 load, lane l and lane l + 16 both read head 16 qd + l % 16:
    // entries 0-31 and 32-63 of the tile. A head's max and sum are combined
    // between the two halves with one shuffle.
    constexpr int NE = kTile / 2;   // entries per thread
    const int qd = warp;
    const int hl = lane & 15;
    const int half = lane >> 4;
    const int h = qd * 16 + hl;
    const bool active = h < HG;
    const bool warp_has_heads = qd * 16 < HG;
    const int e0 = half * NE;   // first entry of this thread
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t prow = sbase + LY::kKV + kPAtom + (h >> 3) * 1024 + (h & 7) * 128;
    float m = -INFINITY, l = 0.0f;   // l: this thread's share of the row sum
    float s[NE];
    // The softmax warps meet at named barriers (ids 1-2), so every timeout
    // decision is made jointly: either all leave the loop or none.
    for (int t = 0; t < n_eff; ++t) {
      const int sb = t & 1;
      bool ok = mbar_wait(&bars[kSFull + sb], (t >> 1) & 1);
      bool need = false;
      float mt = -INFINITY;
      if (ok) {
        tc_fence_after();
        if (warp_has_heads) {
          float s2[NE];
          const uint32_t col = (uint32_t)(sb * kSCols);
          tmem_ld16x32bx2_x32_pair_sync(tmem + lane_base + col, tmem + lane_base + kSbCol + col, s,
                                        s2);
#pragma unroll
          for (int j = 0; j < NE; ++j) s[j] += s2[j];
          const uint32_t mask = vmask[2 * t + (e0 >> 5)] >> (e0 & 31);
#pragma unroll
          for (int j = 0; j < NE; ++j) {
            s[j] = ((mask >> j) & 1u) ? s[j] * p.scale_log2 : -INFINITY;
            mt = fmaxf(mt, s[j]);
          }
          mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        }
      }
      if (named_bar_or(1, SWT, !ok)) {
        failed = true;
        break;
      }
      if (warp_has_heads) {
        float a = 1.0f;
        if (mt > m + kRescaleThreshold) {
          a = (m == -INFINITY) ? 0.0f : ex2(m - mt);
          need = t > 0;
          l *= a;
          m = mt;
        }
        if (active && half == 0) alpha_s[sb * 64 + h] = a;
      }
      const bool any = named_bar_or(2, SWT, need && active);
      tc_fence_after();
      if (active) {
        float lsum = 0.0f;
#pragma unroll
        for (int c4 = 0; c4 < NE / 8; ++c4) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = (m == -INFINITY) ? 0.0f : ex2(s[8 * c4 + 2 * i] - m);
            const float p1 = (m == -INFINITY) ? 0.0f : ex2(s[8 * c4 + 2 * i + 1] - m);
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            const float2 pr = __bfloat1622float2(pb);
            lsum += pr.x;
            lsum += pr.y;
            w[i] = *reinterpret_cast<const uint32_t*>(&pb);
          }
          const int c8 = (e0 >> 3) + c4;   // 16-byte chunk of the 128-byte P row
          st_shared_v4(prow + sb * kStageBytes + ((c8 ^ (h & 7)) << 4),
                       make_uint4(w[0], w[1], w[2], w[3]));
        }
        l += lsum;
      }
      if (any) {
        // O^T must hold PV(t-1) before it is rescaled. Tile t was loaded after
        // PV(t-2) completed, so the stage barrier of PV(t-1) is at most one
        // phase from it and its parity test is exact.
        const bool pv_ok = mbar_wait(&bars[kKvEmpty + ((t - 1) & 1)], ((t - 1) >> 1) & 1);
        if (named_bar_or(1, SWT, !pv_ok)) {
          failed = true;
          break;
        }
        tc_fence_after();
        // O^T lanes are dv rows; columns are heads. Scale column h by alpha[h].
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
#pragma unroll 1
          for (int c = 0; c < HG / 16; ++c) {
            float v[16];
            const uint32_t addr = tmem + lane_base + kOCol + b * HG + 16 * c;
            tmem_ld16_sync(addr, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha_s[sb * 64 + 16 * c + i];
            tmem_st16(addr, v);
          }
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kPFull + sb]);
    }
    if (!failed) {
      const bool pv_ok =
          mbar_wait(&bars[kKvEmpty + ((n_eff - 1) & 1)], ((n_eff - 1) >> 1) & 1);
      failed = named_bar_or(1, SWT, !pv_ok);   // a joint decision
    }
    if (!failed) {
      tc_fence_after();
      // Epilogue: partial O (unnormalised, relative to m) rounded to bf16,
      // m and l in fp32.
      const int dv_lane = qd * 32 + lane;
      __nv_bfloat16* po = reinterpret_cast<__nv_bfloat16*>(p.part_o) + part_base * kDv;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        float v[HG];
        tmem_ld_cols<HG>(tmem + lane_base + kOCol + b * HG, v);
#pragma unroll
        for (int i = 0; i < HG; ++i)
          po[(int64_t)i * kDv + 128 * b + dv_lane] = __float2bfloat16_rn(v[i]);
      }
      const float lw = l + __shfl_xor_sync(0xffffffffu, l, 16);
      if (active && half == 0) {
        p.part_m[part_base + h] = m;
        p.part_l[part_base + h] = lw;
      }
    }
  }

  // Q's copies land before the CTA exits, on every path (bf16: a bounded
  // wait on the box copies).
  if constexpr (FP8) {
    if (tid < SWT) cp_async_wait_all();
  } else {
    if (tid == 0) (void)mbar_wait(&bars[kQFull], 0);
  }
  if (failed && p.err != nullptr) atomicOr(p.err, kErrTimeout);
  tc_fence_before();
  const bool cta_failed = __syncthreads_or(failed);
  tc_fence_after();
  // A split that gave up leaves a NaN m and l, so its row's output is NaN
  // (never a plausible value built from a previous call's partials).
  if (cta_failed && tid < HG) {
    p.part_m[part_base + tid] = __int_as_float(0x7fc00000);
    p.part_l[part_base + tid] = __int_as_float(0x7fc00000);
  }
  if (warp == RL::kQkA) tmem_dealloc(tmem, LY::kTmemCols);
}

// The combine: one warp merges the splits of one (row, head) pair in split
// order (merge_weights once per pair, merge_value per output element). Lane l
// takes output columns [16 l, 16 l + 16): two 16-byte loads of bf16 partials
// per split, all of them (128 bytes per lane) issued before any arithmetic.
// W warps (pairs) per CTA; which warp takes a pair never changes its
// arithmetic.
template <int W>
__global__ void __launch_bounds__(32 * W) combine_warp_kernel(const uint16_t* __restrict__ part_o,
                                                              const float* __restrict__ part_m,
                                                              const float* __restrict__ part_l,
                                                              int64_t R, int H, int S,
                                                              const float* __restrict__ sink,
                                                              __nv_bfloat16* __restrict__ out,
                                                              float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t RH = R * H;
  const int64_t rh = (int64_t)blockIdx.x * W + (threadIdx.x >> 5);   // row * H + h
  if (rh >= RH) return;
  float ms[kMaxSplits], ls[kMaxSplits];
  uint4 raw[kMaxSplits][2];
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    ms[s] = -INFINITY;
    ls[s] = 0.0f;
    raw[s][0] = raw[s][1] = make_uint4(0u, 0u, 0u, 0u);
    if (s < S) {
      ms[s] = part_m[s * RH + rh];
      ls[s] = part_l[s * RH + rh];
      const uint4* p = reinterpret_cast<const uint4*>(part_o + (s * RH + rh) * kDv + 16 * lane);
      raw[s][0] = p[0];
      raw[s][1] = p[1];
    }
  }
  const float sl = sink != nullptr ? sink[rh % H] * 1.4426950408889634f : -INFINITY;
  const MergeWeights mw = merge_weights(ms, ls, sl);
  uint4* o = reinterpret_cast<uint4*>(out + rh * kDv + 16 * lane);
  if (mw.state != 0) {   // 2: a split gave up (NaN); 1: no entry (0, lse -inf)
    const uint32_t f = mw.state == 2 ? 0x7fc07fc0u : 0u;
    o[0] = o[1] = make_uint4(f, f, f, f);
    if (lane == 0) lse[rh] = mw.state == 2 ? __int_as_float(0x7fc00000) : -INFINITY;
    return;
  }
  uint32_t packed[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {   // word j holds elements 2j (low half) and 2j + 1
    float lo[kMaxSplits], hi[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      const uint4& q = raw[s][j >> 2];
      const uint32_t w = (j & 3) == 0 ? q.x : (j & 3) == 1 ? q.y : (j & 3) == 2 ? q.z : q.w;
      lo[s] = __uint_as_float(w << 16);
      hi[s] = __uint_as_float(w & 0xffff0000u);
    }
    packed[j] = pack_bf16x2(merge_value(mw, lo), merge_value(mw, hi));
  }
  o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  if (lane == 0) lse[rh] = mw.lse;
}

template <int HG, bool FP8>
cudaError_t launch_split(const KParams& kp, int64_t blocks, cudaStream_t stream) {
  using LY = Layout<HG>;
  static PerDeviceOnce attr_once;
  auto kern = sparse_mla_split_kernel<HG, FP8>;
  int dev = 0;
  cudaError_t e = stream_device(stream, &dev);
  if (e == cudaSuccess) e = set_max_dynamic_smem(attr_once, dev, kern, LY::kSmemBytes);
  if (e != cudaSuccess) return e;
  // q viewed as [R * H rows, 576 columns] of bf16 (rows 1152 bytes apart);
  // the FP8 kernel copies Q itself and never reads the map.
  CUtensorMap qmap{};
  if (FP8)
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(Roles<FP8>::kThreads), LY::kSmemBytes,
                      stream, 1u, qmap, kp);
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)(kp.R * kp.H)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kRowBytesBf16};
  const cuuint32_t box[2] = {64, (cuuint32_t)HG};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(kp.q), gdim,
          gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return launch_pdl(kern, dim3((unsigned)blocks), dim3(Roles<FP8>::kThreads), LY::kSmemBytes, stream,
                    1u, qmap, kp);
}

}  // namespace

size_t attn_workspace_bytes(int64_t R, int H, int k, int k2) {
  const int64_t S = num_splits_total(k, k2);
  const int64_t n = S * R * H;
  const size_t o = (size_t)n * kDv * sizeof(uint16_t);
  const size_t ml = ((size_t)n * sizeof(float) + 255) & ~size_t(255);
  return o + 2 * ml;
}

AttnWorkspace attn_workspace_carve(void* base, int64_t R, int H, int k, int k2) {
  const int64_t S = num_splits_total(k, k2);
  const int64_t n = S * R * H;
  const size_t o = (size_t)n * kDv * sizeof(uint16_t);
  const size_t ml = ((size_t)n * sizeof(float) + 255) & ~size_t(255);
  AttnWorkspace w;
  w.part_o = reinterpret_cast<uint16_t*>(base);
  w.part_m = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(base) + o);
  w.part_l = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(base) + o + ml);
  return w;
}

cudaError_t launch_sparse_mla(const AttnArgs& a, cudaStream_t stream) {
  if (a.R == 0) return cudaSuccess;
  const int HG = a.H < 64 ? a.H : 64;
  KParams kp;
  kp.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  kp.kv = reinterpret_cast<const uint8_t*>(a.kv);
  kp.num_pages = a.num_pages;
  kp.block_table = a.block_table;
  kp.bt_stride = a.bt_stride;
  kp.num_bt_rows = a.num_bt_rows;
  kp.row_req = a.row_req;
  kp.idx = a.idx;
  kp.lens = a.lens;
  kp.R = a.R;
  kp.H = a.H;
  kp.k = a.k;
  kp.num_splits = num_splits_total(a.k, a.k2);
  kp.kv2 = reinterpret_cast<const uint8_t*>(a.kv2);
  kp.num_pages2 = a.num_pages2;
  kp.block_table2 = a.block_table2;
  kp.bt_stride2 = a.bt_stride2;
  kp.idx2 = a.idx2;
  kp.lens2 = a.lens2;
  kp.k2 = a.k2;
  kp.num_hg = a.H / HG;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  AttnWorkspace ws = attn_workspace_carve(a.workspace, a.R, a.H, a.k, a.k2);
  kp.part_o = ws.part_o;
  kp.part_m = ws.part_m;
  kp.part_l = ws.part_l;
  kp.err = a.err_flag;
  const int64_t blocks = a.R * kp.num_splits * kp.num_hg;
  const bool fp8 = a.kv_dtype == 1;
  cudaError_t e;
  if (HG == 64)
    e = fp8 ? launch_split<64, true>(kp, blocks, stream) : launch_split<64, false>(kp, blocks, stream);
  else if (HG == 32)
    e = fp8 ? launch_split<32, true>(kp, blocks, stream) : launch_split<32, false>(kp, blocks, stream);
  else
    e = fp8 ? launch_split<16, true>(kp, blocks, stream) : launch_split<16, false>(kp, blocks, stream);
  if (e != cudaSuccess) return e;
  const int64_t RH = a.R * a.H;
  return launch_pdl(combine_warp_kernel<8>, dim3((unsigned)((RH + 7) / 8)), dim3(256), 0, stream, 1u,
                    (const uint16_t*)ws.part_o, (const float*)ws.part_m, (const float*)ws.part_l, a.R,
                    a.H, kp.num_splits, a.sink, reinterpret_cast<__nv_bfloat16*>(a.out), a.lse);
}

}  // namespace dsmla
