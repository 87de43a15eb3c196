// Deterministic per-row top-k: radix select of the k-th largest key, then an
// ordered compaction that writes the selected positions in ascending order.
//
// Follows "[DeepSeek-V4][Preview][DO NOT MERGE] Batch-invariant kernels for
// 0-diff RL", section "Deterministic sparse top-k": positions are ranked by a
// composite (score, position) key with a stable tie-break and the selected
// positions are put in canonical ascending order. The signed length clamp and
// the -1 padding follow "[Bugfix] Make DSV4 sparse MLA work end-to-end for
// plain decode, MTP, and DSpark", section "What is fixed".
//
// Five kernels, chosen by the shape of the call (and, for the grid kernel,
// by whether a workspace is given and the scores start 16-byte aligned):
//   topk_smem_kernel     one CTA per row, the whole row in shared memory;
//   topk_stream_kernel   a persistent grid, each CTA streaming whole rows;
//   topk_grid_kernel     every row spread over the whole GPU: one cooperative
//                        launch whose phases are separated by two grid
//                        barriers (bounded waits on a workspace counter);
//   topk_cluster_kernel  one thread-block cluster of up to 8 CTAs per row,
//                        which exchange histograms and counts through
//                        distributed shared memory between hardware cluster
//                        barriers;
//   topk_rows_kernel     one CTA per row, histogram passes over global memory.
// Only the grid kernel waits on a value written by another CTA, and it is
// launched cooperatively (every CTA resident). The selected set is unique
// (the order is total), so every kernel gives the same bit-exact output, and
// a row's output never depends on the rest of the batch.
//
// Key: the float's bits mapped to an unsigned integer whose order is the
// float order (sign flipped for non-negatives, all bits flipped for
// negatives), with -0.0 first canonicalised to +0.0 and every NaN mapped to
// 0 (below -inf, whose key is 0x007FFFFF).
//
// Select: histograms of 11, 11 and 10-bit digits from the top find the
// threshold prefix P (at `shift` resolved bits) and `take`, the number of
// positions whose prefix equals P that are selected (the lowest-position
// ones). A digit pass stops early once the threshold bucket is taken whole.
// Compact: one ordered pass; a position with prefix > P is selected, one with
// prefix == P is selected iff fewer than `take` such positions precede it.
// Its output slot is (#greater before it) + min(#equal before it, take).

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace dsmla {

namespace {

constexpr int kThreads = 512;
constexpr int kChunk = kThreads * 4;  // elements per block-wide step
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;

__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of one uint32 per thread (NT threads);
// `total` gets the block sum. Ends with a barrier so `buf` may be reused.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan_nt(uint32_t v, uint32_t* buf,
                                                            uint32_t& total) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? buf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) buf[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? buf[warp - 1] : 0u;
  total = buf[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* buf,
                                                         uint32_t& total) {
  return block_exclusive_scan_nt<kThreads>(v, buf, total);
}

// Loads elements [i0, i0 + 4) of the row (those below L) as keys; `valid`
// gets one bit per loaded element. Uses one 16-byte load when the row
// pointer is 16-byte aligned and the four elements are in range.
__device__ __forceinline__ void load4_keys(const float* __restrict__ p, int64_t i0, int64_t L,
                                           bool aligned, uint32_t key[4], uint32_t& valid) {
  if (aligned && i0 + 3 < L) {
    const float4 v = *reinterpret_cast<const float4*>(p + i0);
    key[0] = score_key(v.x);
    key[1] = score_key(v.y);
    key[2] = score_key(v.z);
    key[3] = score_key(v.w);
    valid = 0xFu;
    return;
  }
  valid = 0u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    key[q] = 0u;
    if (i0 + q < L) {
      key[q] = score_key(p[i0 + q]);
      valid |= 1u << q;
    }
  }
}

__global__ void __launch_bounds__(kThreads) topk_rows_kernel(
    const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ ends, int k, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t scan_buf[32];
  __shared__ uint32_t pick[3];

  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int64_t s = starts[row];
  const int64_t e = ends[row];
  int64_t L = 0;
  if (s >= 0 && s <= stride) {
    L = e - s;
    if (L < 0) L = 0;
    if (L > stride - s) L = stride - s;
  }
  int32_t* __restrict__ orow = out + row * (int64_t)k;

  if (L <= (int64_t)k) {  // every position is selected; no score is read
    for (int j = tid; j < k; j += kThreads) orow[j] = (int64_t)j < L ? j : -1;
    return;
  }

  const float* __restrict__ p = scores + row * stride + s;
  const bool aligned = (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;

  uint32_t prefix = 0u;  // resolved high bits of the threshold key
  int shift = 32;        // number of unresolved low bits
  uint32_t take = (uint32_t)k;

  for (int pass = 0; pass < 3; ++pass) {
    const int width = pass < 2 ? 11 : 10;
    const int nshift = shift - width;
    const uint32_t nbins = 1u << width;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0u;
    __syncthreads();

    for (int64_t base = 0; base < L; base += kChunk) {
      uint32_t key[4], valid;
      load4_keys(p, base + 4 * tid, L, aligned, key, valid);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool match = (valid >> q) & 1u && (pass == 0 || (key[q] >> shift) == prefix);
        if (match) atomicAdd(&hist[(key[q] >> nshift) & (nbins - 1u)], 1u);
      }
    }
    __syncthreads();

    // Bins in descending order: thread t owns kBinsPerThread consecutive ones.
    uint32_t c[kBinsPerThread];
    uint32_t mine = 0u;
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) {
      const int b = (int)nbins - 1 - (tid * kBinsPerThread + q);
      c[q] = b >= 0 ? hist[b] : 0u;
      mine += c[q];
    }
    uint32_t total;
    uint32_t above = block_exclusive_scan(mine, scan_buf, total);
#pragma unroll
    for (int q = 0; q < kBinsPerThread; ++q) {
      const int b = (int)nbins - 1 - (tid * kBinsPerThread + q);
      if (b >= 0 && above < take && take <= above + c[q]) {
        pick[0] = (uint32_t)b;
        pick[1] = take - above;
        pick[2] = c[q];
      }
      above += c[q];
    }
    __syncthreads();
    const uint32_t b = pick[0];
    const uint32_t cnt = pick[2];
    take = pick[1];
    prefix = (pass == 0 ? 0u : (prefix << width)) | b;
    shift = nshift;
    if (cnt == take) break;  // the whole bucket is selected: no tie left to order
  }

  // Ordered compaction.
  uint32_t carry_gt = 0u, carry_eq = 0u;
  for (int64_t base = 0; base < L; base += kChunk) {
    const int64_t i0 = base + 4 * tid;
    uint32_t key[4], valid;
    load4_keys(p, i0, L, aligned, key, valid);
    uint32_t gt = 0u, eq = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if ((valid >> q) & 1u) {
        const uint32_t hi = shift >= 32 ? 0u : (key[q] >> shift);
        gt |= (uint32_t)(hi > prefix) << q;
        eq |= (uint32_t)(hi == prefix) << q;
      }
    }
    const uint32_t packed = ((uint32_t)__popc(gt) << 16) | (uint32_t)__popc(eq);
    uint32_t total;
    const uint32_t ex = block_exclusive_scan(packed, scan_buf, total);
    uint32_t g = carry_gt + (ex >> 16);
    uint32_t q_eq = carry_eq + (ex & 0xFFFFu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if ((gt >> q) & 1u) {
        orow[g + min(q_eq, take)] = (int32_t)(i0 + q);
        ++g;
      } else if ((eq >> q) & 1u) {
        if (q_eq < take) orow[g + q_eq] = (int32_t)(i0 + q);
        ++q_eq;
      }
    }
    carry_gt += total >> 16;
    carry_eq += total & 0xFFFFu;
    if (carry_gt + min(carry_eq, take) >= (uint32_t)k) break;
  }
}


// ---------------------------------------------------------------------------
// Rows of up to 32768 scores: one 1024-thread CTA per row, the whole row in
// shared memory. Every thread issues asynchronous 16-byte copies for its
// share of the row (4-byte copies when the row start is not 16-byte
// aligned) in four commit groups, and turns each group into keys and
// 12-bit histogram counts as soon as its own copies have landed.
//
// After the threshold bin is picked, one pass gives every thread the
// selection word of its own 32 positions: keys above the bin are selected,
// keys in the bin are marked as tied. The bin's low 20 bits are resolved by
// 8-, 8- and 4-bit histogram passes that visit only the tied positions, and
// each thread then settles its own tied keys. Keys equal to the threshold
// at all 32 bits go to the lowest positions by one block-wide scan of the
// tied counts, and a last scan of the selected counts gives every output
// slot in index order. Apart from the histograms, no step uses atomics.

constexpr int kRowThreads = 1024;
constexpr int kRowMaxLen = 32768;
constexpr int kRowBins = 4096;
constexpr int kRowGroups = 4;   // commit groups of the row copy
constexpr int64_t kRowMinRows = 16;   // fewer rows: a cluster per row spreads each row wider

struct RowSmem {
  uint32_t key[kRowMaxLen];
  uint32_t hist[kRowBins];
  uint32_t hsmall[3][256];   // one per refinement pass, zeroed up front
  uint32_t wsum[32];
  uint32_t pick[3];
};

__device__ __forceinline__ void cp_async_16B(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_4B(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Picks, among NBINS bins counted in `hist` (descending bin order), the bin
// holding the `take`-th largest key: every thread gets (bin, count of that
// bin, take within that bin). Two block barriers.
template <int NBINS>
__device__ __forceinline__ void row_pick(const uint32_t* hist, uint32_t take, uint32_t* wsum,
                                         uint32_t* pick, uint32_t& bin, uint32_t& cnt,
                                         uint32_t& take_in_bin) {
  constexpr int kPer = NBINS >= kRowThreads ? NBINS / kRowThreads : 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t c[kPer];
  uint32_t mine = 0u;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int b = NBINS - 1 - (tid * kPer + q);
    c[q] = b >= 0 ? hist[b] : 0u;
    mine += c[q];
  }
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  const uint32_t ws = wsum[lane];
  uint32_t wincl = ws;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += y;
  }
  uint32_t above = __shfl_sync(0xffffffffu, wincl - ws, warp) + incl - mine;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int b = NBINS - 1 - (tid * kPer + q);
    if (b >= 0 && above < take && take <= above + c[q]) {
      pick[0] = (uint32_t)b;
      pick[1] = take - above;
      pick[2] = c[q];
    }
    above += c[q];
  }
  __syncthreads();
  bin = pick[0];
  take_in_bin = pick[1];
  cnt = pick[2];
}

// Mask of the first m set bits of x.
__device__ __forceinline__ uint32_t first_set_bits(uint32_t x, uint32_t m) {
  uint32_t r = 0u;
  while (m-- > 0u && x) {
    const uint32_t low = x & (0u - x);
    r |= low;
    x ^= low;
  }
  return r;
}

__device__ __forceinline__ uint4 keys_of(uint4 w) {
  return make_uint4(score_key(__uint_as_float(w.x)), score_key(__uint_as_float(w.y)),
                    score_key(__uint_as_float(w.z)), score_key(__uint_as_float(w.w)));
}

__global__ void __launch_bounds__(kRowThreads, 1) topk_smem_kernel(
    const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ ends, int k, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char row_smem_raw[];
  RowSmem& sm = *reinterpret_cast<RowSmem*>(row_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t row = blockIdx.x;
  const int64_t s = starts[row];
  const int64_t e = ends[row];
  int L = 0;
  if (s >= 0 && s <= stride) {
    int64_t L64 = e - s;
    if (L64 < 0) L64 = 0;
    if (L64 > stride - s) L64 = stride - s;
    L = (int)L64;   // <= kRowMaxLen
  }
  int32_t* __restrict__ orow = out + row * (int64_t)k;
  if (L <= k) {   // every position is selected; no score is read
    for (int j = tid; j < k; j += kRowThreads) orow[j] = j < L ? j : -1;
    return;
  }
  const float* __restrict__ p = scores + row * stride + s;

  // Key slot i holds position i. Thread t copies granules (4 slots) t,
  // t + 1024, ...; group g holds its granules 2g and 2g + 1. Slots from L
  // up to the next multiple of 4 hold bytes of the row's last 16-byte
  // granule and are never counted or selected.
  const int n4 = (L + 3) >> 2;
  const bool aligned = (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;
#pragma unroll
  for (int g = 0; g < kRowGroups; ++g) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = (2 * g + h) * kRowThreads + tid;
      if (j < n4) {
        if (aligned) {
          cp_async_16B(&sm.key[4 * j], p + 4 * j);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (4 * j + q < L) cp_async_4B(&sm.key[4 * j + q], p + 4 * j + q);
        }
      }
    }
    cp_async_commit_group();
  }
  for (int i = tid; i < kRowBins; i += kRowThreads) sm.hist[i] = 0u;
  for (int i = tid; i < 3 * 256; i += kRowThreads) (&sm.hsmall[0][0])[i] = 0u;
  __syncthreads();   // histograms zeroed

  // Keys in place, and the histogram of their top 12 bits, group by group.
  uint4* const key4 = reinterpret_cast<uint4*>(sm.key);
  auto convert = [&](int g) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = (2 * g + h) * kRowThreads + tid;
      if (j < n4) {
        const uint4 w = keys_of(key4[j]);
        key4[j] = w;
        if (4 * j + 4 <= L) {
          atomicAdd(&sm.hist[w.x >> 20], 1u);
          atomicAdd(&sm.hist[w.y >> 20], 1u);
          atomicAdd(&sm.hist[w.z >> 20], 1u);
          atomicAdd(&sm.hist[w.w >> 20], 1u);
        } else {
          atomicAdd(&sm.hist[w.x >> 20], 1u);
          if (4 * j + 1 < L) atomicAdd(&sm.hist[w.y >> 20], 1u);
          if (4 * j + 2 < L) atomicAdd(&sm.hist[w.z >> 20], 1u);
        }
      }
    }
  };
  cp_async_wait_group<3>();
  convert(0);
  cp_async_wait_group<2>();
  convert(1);
  cp_async_wait_group<1>();
  convert(2);
  cp_async_wait_group<0>();
  convert(3);
  __syncthreads();

  // Threshold state: `P` is the threshold key's prefix with `shift` low bits
  // dropped; `take` of the `cnt` keys with that prefix (the lowest positions)
  // are selected.
  uint32_t take = (uint32_t)k, P, cnt, b;
  row_pick<kRowBins>(sm.hist, take, sm.wsum, sm.pick, P, cnt, take);

  // Thread t's positions [32t, 32t + 32): 8 granules, read in a lane-rotated
  // order so that the warp's 16-byte reads hit distinct banks. A key's 12-bit
  // prefix is above P iff the key is at least (P + 1) << 20, and equal to P
  // iff it is at least P << 20 and not above; each granule's four bits are
  // gathered first and placed with one shift.
  const int base = 32 * tid;
  uint32_t sel = 0u, eqw = 0u;
  if (base < L) {
    const uint32_t lo = P << 20;
    const bool top = P == kRowBins - 1u;   // no prefix lies above the top bin
    const uint32_t hi = top ? 0u : (P + 1u) << 20;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int cc = (c + lane) & 7;
      const uint4 w = key4[8 * tid + cc];
      uint32_t gs = (uint32_t)(w.x >= hi) | ((uint32_t)(w.y >= hi) << 1) |
                    ((uint32_t)(w.z >= hi) << 2) | ((uint32_t)(w.w >= hi) << 3);
      if (top) gs = 0u;
      const uint32_t ge = (uint32_t)(w.x >= lo) | ((uint32_t)(w.y >= lo) << 1) |
                          ((uint32_t)(w.z >= lo) << 2) | ((uint32_t)(w.w >= lo) << 3);
      sel |= gs << (4 * cc);
      eqw |= (ge & ~gs) << (4 * cc);
    }
    if (L - base < 32) {
      const uint32_t valid = (1u << (L - base)) - 1u;
      sel &= valid;
      eqw &= valid;
    }
  }

  int shift = 20;
  for (int pass = 0; pass < 3 && cnt != take; ++pass) {
    const int width = pass < 2 ? 8 : 4;
    const int nshift = shift - width;
    const uint32_t dmask = (1u << width) - 1u;
    uint32_t* const hs = sm.hsmall[pass];
    for (uint32_t m = eqw; m; m &= m - 1u) {
      const uint32_t key = sm.key[base + __ffs(m) - 1];
      if ((key >> shift) == P) atomicAdd(&hs[(key >> nshift) & dmask], 1u);
    }
    __syncthreads();
    if (width == 8) row_pick<256>(hs, take, sm.wsum, sm.pick, b, cnt, take);
    else row_pick<16>(hs, take, sm.wsum, sm.pick, b, cnt, take);
    P = (P << width) | b;
    shift = nshift;
  }

  // Settle this thread's tied keys: above the threshold, or tied with it.
  const bool all_eq = cnt == take;
  if (shift < 20) {
    uint32_t tied = 0u;
    for (uint32_t m = eqw; m; m &= m - 1u) {
      const int bit = __ffs(m) - 1;
      const uint32_t hi = sm.key[base + bit] >> shift;
      if (hi > P) sel |= 1u << bit;
      else if (hi == P) tied |= 1u << bit;
    }
    eqw = tied;
  }
  if (all_eq) {
    sel |= eqw;
  } else {
    // Keys equal at all 32 bits: the lowest `take` positions win.
    uint32_t tot;
    const uint32_t r =
        block_exclusive_scan_nt<kRowThreads>(__popc(eqw), sm.wsum, tot);
    if (r < take) sel |= first_set_bits(eqw, take - r);
  }
  uint32_t total;
  uint32_t pos = block_exclusive_scan_nt<kRowThreads>(__popc(sel), sm.wsum, total);
  while (sel) {
    const int bit = __ffs(sel) - 1;
    sel &= sel - 1u;
    if (pos < (uint32_t)k) orow[pos] = base + bit;
    ++pos;
  }
}

// ---------------------------------------------------------------------------
// Cluster variant, for batches too small to fill the GPU with one CTA per
// row: the row is cut into C <= 8 contiguous chunks of at most 16384 scores,
// one per CTA of a thread-block cluster, each held in that CTA's shared
// memory (the row is read from HBM once).
//
// Elements are ranked by a 56-bit composite: the 32-bit score key above 24
// bits of (2^24 - 1 - position), so no two elements tie and the k-th largest
// composite alone decides the selection (equal scores go to the lower
// positions first, as the order requires). Its top 12 bits come from
// per-CTA 4096-bin histograms: each CTA publishes the sums of its 128
// groups of 32 bins to every CTA of the cluster, all CTAs pick the same
// group after one cluster barrier, then read that group's 32 bins from each
// CTA. The remaining bits are resolved in 8-, 8-, 4-, 8-, 8- and 8-bit passes
// (stopping as soon as the threshold bin holds exactly the keys still
// needed), each with one cluster barrier: every CTA counts its keys of the
// current bin into a 256-bin histogram and stores it into every CTA's
// receive buffer (double buffered by pass parity), so after the barrier the
// pick reads only local memory. Each CTA then marks its selected positions
// as bitmap words, publishes its count, and after a last barrier writes its
// positions at the offset of the CTAs before it. Every CTA of the cluster
// runs the same barriers, so none can wait on one that has left.

constexpr int kClThreads = 512;
constexpr int kClMaxChunk = 16384;   // keys per CTA (64 KiB of shared memory)
constexpr int kClMaxCluster = 8;
constexpr int kClGroups = 128;       // 4096 twelve-bit bins in groups of 32
constexpr int kClCompBits = 56;      // 32-bit key, then 24 position bits

struct ClSmem {
  uint32_t hist12[4096];                          // this CTA's 12-bit histogram
  uint32_t gsum_in[kClMaxCluster][kClGroups];     // group sums, stored by each CTA
  uint32_t gbins[kClMaxCluster][32];              // the picked group's bins, per CTA
  uint32_t h8_in[2][kClMaxCluster][256];          // pass histograms, stored by each CTA
  uint32_t h8[256];                               // this CTA's pass histogram
  uint32_t cnt_in[kClMaxCluster];                 // selected counts, stored by each CTA
  uint32_t wsum[32];
  uint32_t pick[3];
  uint32_t pad;
  // followed by the chunk's keys (16-byte aligned)
};
static_assert(sizeof(ClSmem) % 16 == 0, "keys start 16-byte aligned");

// Distributed shared memory: another CTA's copy of a local shared variable.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local_ptr, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;"
      : "=r"(remote)
      : "r"((uint32_t)__cvta_generic_to_shared(local_ptr)), "r"(rank));
  return remote;
}
__device__ __forceinline__ uint32_t dsmem_ld(const uint32_t* local_ptr, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(dsmem_addr(local_ptr, rank)));
  return v;
}
__device__ __forceinline__ void dsmem_st(uint32_t* local_ptr, uint32_t rank, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dsmem_addr(local_ptr, rank)), "r"(v)
               : "memory");
}
// All threads of all CTAs of the cluster; shared-memory writes before it
// (local or remote) are visible to reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Thread t holds the count c of the t-th bin in descending order (0 past
// the last bin). Every thread gets the position of the bin holding the
// `take`-th largest element, that bin's count and the take within it.
// Two block barriers.
__device__ __forceinline__ void cl_pick(uint32_t c, uint32_t take, uint32_t* wsum, uint32_t* pick,
                                        uint32_t& pos, uint32_t& cnt, uint32_t& take_in_bin) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kClThreads / 32;
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  const uint32_t ws = lane < kWarps ? wsum[lane] : 0u;
  uint32_t wincl = ws;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += y;
  }
  const uint32_t above = __shfl_sync(0xffffffffu, wincl - ws, warp) + incl - c;
  if (above < take && take <= above + c) {
    pick[0] = (uint32_t)tid;
    pick[1] = take - above;
    pick[2] = c;
  }
  __syncthreads();
  pos = pick[0];
  take_in_bin = pick[1];
  cnt = pick[2];
}

__global__ void __launch_bounds__(kClThreads) topk_cluster_kernel(
    const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ ends, int k, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char cl_smem_raw[];
  ClSmem& sm = *reinterpret_cast<ClSmem*>(cl_smem_raw);
  uint32_t* const key = reinterpret_cast<uint32_t*>(cl_smem_raw + sizeof(ClSmem));
  const uint32_t C = cluster_size();
  const uint32_t rank = cluster_rank();
  const int tid = threadIdx.x, lane = tid & 31;

  const int64_t row = blockIdx.x / C;
  const int64_t s = starts[row];
  const int64_t e = ends[row];
  int L = 0;
  if (s >= 0 && s <= stride) {
    int64_t L64 = e - s;
    if (L64 < 0) L64 = 0;
    if (L64 > stride - s) L64 = stride - s;
    L = (int)L64;   // <= C x kClMaxChunk
  }
  int32_t* __restrict__ orow = out + row * (int64_t)k;
  if (L <= k) {   // the same in every CTA of the cluster: no cluster barrier is used
    if (rank == 0)
      for (int j = tid; j < k; j += kClThreads) orow[j] = j < L ? j : -1;
    return;
  }
  const float* __restrict__ p = scores + row * stride + s;

  // This CTA's chunk: positions [c0, c0 + n), chunks of a multiple of 128.
  const int per = (int)(((int64_t)L + C - 1) / C + 127) & ~127;
  const int c0 = min(L, (int)rank * per);
  const int n = min(L, c0 + per) - c0;
  const int n4 = (n + 3) >> 2;
  if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0u) {   // c0 is a multiple of 4
    for (int j = tid; j < n4; j += kClThreads) cp_async_16B(&key[4 * j], p + c0 + 4 * j);
  } else {
    for (int i = tid; i < n; i += kClThreads) cp_async_4B(&key[i], p + c0 + i);
  }
  cp_async_commit_group();
  for (int i = tid; i < 4096; i += kClThreads) sm.hist12[i] = 0u;
  cp_async_wait_group<0>();
  __syncthreads();

  uint4* const key4 = reinterpret_cast<uint4*>(key);
  for (int j = tid; j < n4; j += kClThreads) {
    const uint4 w = keys_of(key4[j]);
    key4[j] = w;
    const int valid = n - 4 * j;
    atomicAdd(&sm.hist12[w.x >> 20], 1u);
    if (valid > 1) atomicAdd(&sm.hist12[w.y >> 20], 1u);
    if (valid > 2) atomicAdd(&sm.hist12[w.z >> 20], 1u);
    if (valid > 3) atomicAdd(&sm.hist12[w.w >> 20], 1u);
  }
  __syncthreads();

  // Group sums (thread t sums bins 8t .. 8t + 7; four threads make a group),
  // stored into every CTA's gsum_in[rank].
  {
    const uint4 a = *reinterpret_cast<const uint4*>(&sm.hist12[8 * tid]);
    const uint4 b = *reinterpret_cast<const uint4*>(&sm.hist12[8 * tid + 4]);
    uint32_t g = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
    g += __shfl_xor_sync(0xffffffffu, g, 1);
    g += __shfl_xor_sync(0xffffffffu, g, 2);
    if ((tid & 3) == 0)
      for (uint32_t q = 0; q < C; ++q) dsmem_st(&sm.gsum_in[rank][tid >> 2], q, g);
  }
  cluster_sync_all();

  // Threshold state: the composite's top R bits are P; `take` of the `cnt`
  // elements with that prefix are still to be selected.
  uint32_t take = (uint32_t)k, cnt, bpos;
  uint32_t c = 0u;
  if (tid < kClGroups)
    for (uint32_t q = 0; q < C; ++q) c += sm.gsum_in[q][kClGroups - 1 - tid];
  cl_pick(c, take, sm.wsum, sm.pick, bpos, cnt, take);
  const int G = kClGroups - 1 - (int)bpos;
  if (tid < 32 * (int)C) sm.gbins[tid >> 5][tid & 31] = dsmem_ld(&sm.hist12[32 * G + (tid & 31)], tid >> 5);
  __syncthreads();
  c = 0u;
  if (tid < 32)
    for (uint32_t q = 0; q < C; ++q) c += sm.gbins[q][31 - tid];
  cl_pick(c, take, sm.wsum, sm.pick, bpos, cnt, take);
  uint64_t P = (uint64_t)(32 * G + 31 - (int)bpos);
  int R = 12;
  int par = 0;
  auto comp_of = [&](uint32_t kk, int local) -> uint64_t {
    return ((uint64_t)kk << 24) | (uint64_t)(0xFFFFFFu - (uint32_t)(c0 + local));
  };
  while (cnt != take) {   // at R = 56 every composite is unique, so cnt == take == 1
    const int width = (R >= 28 && R < 32) ? 4 : 8;
    const int sh = kClCompBits - R, nsh = sh - width;
    const uint32_t dmask = (1u << width) - 1u;
    if (tid < 256) sm.h8[tid] = 0u;
    __syncthreads();
    for (int j = tid; j < n4; j += kClThreads) {
      const uint4 w = key4[j];
      const uint32_t kk[4] = {w.x, w.y, w.z, w.w};
      const int valid = n - 4 * j;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t cp = comp_of(kk[q], 4 * j + q);
        if (q < valid && (cp >> sh) == P) atomicAdd(&sm.h8[(uint32_t)(cp >> nsh) & dmask], 1u);
      }
    }
    __syncthreads();
    if (tid < 256)
      for (uint32_t q = 0; q < C; ++q) dsmem_st(&sm.h8_in[par][rank][tid], q, sm.h8[tid]);
    cluster_sync_all();
    c = 0u;
    if (tid <= (int)dmask)
      for (uint32_t q = 0; q < C; ++q) c += sm.h8_in[par][q][dmask - tid];
    cl_pick(c, take, sm.wsum, sm.pick, bpos, cnt, take);
    P = (P << width) | (uint64_t)(dmask - bpos);
    R += width;
    par ^= 1;
  }

  // Selected: composite prefix >= P. Thread t owns local positions
  // [32t, 32t + 32): 8 granules read in a lane-rotated order.
  const int shf = kClCompBits - R;
  const int base = 32 * tid;
  uint32_t w = 0u;
  if (base < n) {
#pragma unroll
    for (int cc0 = 0; cc0 < 8; ++cc0) {
      const int cc = (cc0 + lane) & 7;
      const uint4 v = key4[8 * tid + cc];
      const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w |= (((comp_of(kk[q], base + 4 * cc + q) >> shf) >= P) ? 1u : 0u) << (4 * cc + q);
    }
    if (n - base < 32) w &= (1u << (n - base)) - 1u;
  }
  uint32_t tot;
  uint32_t pos = block_exclusive_scan_nt<kClThreads>(__popc(w), sm.wsum, tot);
  if (tid == 0)
    for (uint32_t q = 0; q < C; ++q) dsmem_st(&sm.cnt_in[rank], q, tot);
  cluster_sync_all();   // the last access to another CTA's shared memory is before this
  for (uint32_t q = 0; q < rank; ++q) pos += sm.cnt_in[q];
  while (w) {
    const int bit = __ffs(w) - 1;
    w &= w - 1u;
    if (pos < (uint32_t)k) orow[pos] = c0 + base + bit;
    ++pos;
  }
}

// ---------------------------------------------------------------------------
// Streaming variant for many rows of up to 65536 scores: a persistent grid of
// two 512-thread CTAs per SM walks the rows, so that one CTA's resolution
// work overlaps the other's loads.
//
// Pass A streams the row once from global memory, builds a histogram of the
// keys' top 12 bits and appends every key whose 12-bit prefix is at least a
// guess G to a candidate list (position and key). G is one bin below the
// threshold bin of the CTA's previous row, so for rows of similar score
// distributions the list holds every selected key plus a few hundred more.
// Once the threshold bin P is known, the list is valid if G <= P and it did
// not overflow; otherwise a second pass re-reads the row (now in L2) and
// collects the members of bin P alone, marking keys above it directly in the
// selection bitmap. The low 20 bits of the threshold are then resolved on the
// list in 8-, 8- and 4-bit histogram passes; a bin too large for the list is
// resolved by passes over the row in global memory instead. The guess only
// decides how much work a row takes: the selected set is always exact.
//
// The selection is a bitmap of the row's positions. Keys tied at all 32 bits
// with the threshold go to the lowest positions, ranked by a prefix count
// over a bitmap of the tied keys. Each thread owns 128 consecutive positions
// (4 words), so one block-wide scan of per-thread counts gives every output
// slot in index order.

constexpr int kStreamThreads = 512;
constexpr int kStreamCtasPerSm = 2;
constexpr int kStreamVec = 4;   // 16-byte loads per thread in flight
constexpr int kStreamMaxLen = 65536;
constexpr int kStreamBins = 4096;                      // top 12 key bits
constexpr int kStreamBinsPerThread = kStreamBins / kStreamThreads;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kStreamSeg = 512;                        // list entries per warp
constexpr int kStreamWords = kStreamMaxLen / 32;       // one bit per position
constexpr int kStreamWordsPerThread = kStreamWords / kStreamThreads;
constexpr uint32_t kStreamNoGuess = kStreamBins;       // collects nothing
constexpr int64_t kStreamMinRows = 256;   // below this the cluster kernel spreads a row wider

struct StreamSmem {
  uint32_t hist[kStreamBins];
  uint32_t cand_idx[kStreamWarps * kStreamSeg];   // warp w appends to [w * kStreamSeg, ...)
  uint32_t cand_key[kStreamWarps * kStreamSeg];
  uint32_t sel[kStreamWords];   // selected positions
  uint32_t eqb[kStreamWords];   // positions tied with the threshold key
  uint32_t hsmall[3][256];      // one per refinement pass, zeroed with the row
  uint32_t scan_buf[32];
  uint32_t pick[3];
  uint32_t nseg[kStreamWarps];   // entries in each warp's segment
  uint32_t overflow;            // some segment was full
};

// Picks, among `nbins` bins counted in `hist` (descending bin order), the bin
// holding the `take`-th largest key. Every thread returns the same (bin,
// count of that bin, take within that bin).
__device__ __forceinline__ void stream_pick(const uint32_t* hist, int nbins, uint32_t take,
                                            StreamSmem& sm, uint32_t& bin, uint32_t& cnt,
                                            uint32_t& take_in_bin) {
  const int tid = threadIdx.x;
  uint32_t c[kStreamBinsPerThread];
  uint32_t mine = 0u;
#pragma unroll
  for (int q = 0; q < kStreamBinsPerThread; ++q) {
    const int b = nbins - 1 - (tid * kStreamBinsPerThread + q);
    c[q] = b >= 0 ? hist[b] : 0u;
    mine += c[q];
  }
  uint32_t total;
  uint32_t above = block_exclusive_scan_nt<kStreamThreads>(mine, sm.scan_buf, total);
#pragma unroll
  for (int q = 0; q < kStreamBinsPerThread; ++q) {
    const int b = nbins - 1 - (tid * kStreamBinsPerThread + q);
    if (b >= 0 && above < take && take <= above + c[q]) {
      sm.pick[0] = (uint32_t)b;
      sm.pick[1] = take - above;
      sm.pick[2] = c[q];
    }
    above += c[q];
  }
  __syncthreads();
  bin = sm.pick[0];
  take_in_bin = sm.pick[1];
  cnt = sm.pick[2];
  __syncthreads();
}

// One warp picks, among NBINS (16 or 256) bins counted in `hist`
// (descending bin order), the bin holding the `take`-th largest key: lane l
// sums bins NBINS-1-8l .. NBINS-8-8l, a warp scan finds the lane where the
// count crosses `take`, and that lane walks its bins. Every warp that calls
// it on the same counts gets the same (bin, count of that bin, take within
// that bin), with no block barrier.
template <int NBINS>
__device__ __forceinline__ void warp_pick(const uint32_t* hist, uint32_t take, uint32_t& bin,
                                          uint32_t& cnt, uint32_t& take_in_bin) {
  constexpr int kPer = NBINS / 32 > 0 ? NBINS / 32 : 1;
  const int lane = threadIdx.x & 31;
  uint32_t c[kPer];
  uint32_t mine = 0u;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int b = NBINS - 1 - (lane * kPer + q);
    c[q] = b >= 0 ? hist[b] : 0u;
    mine += c[q];
  }
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t above = incl - mine;
  // The crossing lane: the first whose inclusive count reaches take.
  const uint32_t hit = __ballot_sync(0xffffffffu, incl >= take);
  const int f = __ffs(hit) - 1;   // hit != 0: the bins sum to at least take
  uint32_t rb = 0u, rc = 0u, rt = 0u;
  if (lane == f) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int b = NBINS - 1 - (lane * kPer + q);
      if (b >= 0 && above < take && take <= above + c[q]) {
        rb = (uint32_t)b;
        rc = c[q];
        rt = take - above;
      }
      above += c[q];
    }
  }
  bin = __shfl_sync(0xffffffffu, rb, f);
  cnt = __shfl_sync(0xffffffffu, rc, f);
  take_in_bin = __shfl_sync(0xffffffffu, rt, f);
}

// Clamped [start, end) of a row, as in every other kernel here: the length
// is end - start, bounded to [0, stride - start]; a start outside [0,
// stride] gives an empty row.
__device__ __forceinline__ int stream_row_len(const int32_t* starts, const int32_t* ends,
                                              int64_t row, int64_t stride, int64_t& s) {
  s = starts[row];
  const int64_t e = ends[row];
  int64_t L = 0;
  if (s >= 0 && s <= stride) {
    L = e - s;
    if (L < 0) L = 0;
    if (L > stride - s) L = stride - s;
  }
  return (int)L;
}


// First slot, in the warp's own list segment, for this thread's `n` appends;
// `used` (the same in every lane) is the segment's fill. Every lane of the
// warp must call it.
__device__ __forceinline__ uint32_t stream_reserve(uint32_t n, uint32_t& used) {
  const int lane = threadIdx.x & 31;
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t slot = used + incl - n;
  used += __shfl_sync(0xffffffffu, incl, 31);
  return slot;
}

// One streaming pass over the row's keys, kStreamVec x 16 bytes per thread in
// flight.
// kFirst: histogram of the top 12 bits; keys with prefix >= bin are listed.
// Otherwise: keys with prefix > bin are marked in `sel`, those equal listed.
template <bool kFirst>
__device__ __forceinline__ void stream_pass(const float* __restrict__ p, int L, uint32_t bin,
                                            StreamSmem& sm) {
  const int tid = threadIdx.x, warp = tid >> 5;
  uint32_t used = 0u;   // this warp's segment fill
  uint32_t* const seg_idx = sm.cand_idx + warp * kStreamSeg;
  uint32_t* const seg_key = sm.cand_key + warp * kStreamSeg;
  auto classify = [&](uint32_t key, int i) -> bool {
    const uint32_t pre = key >> 20;
    if (kFirst) {
      atomicAdd(&sm.hist[pre], 1u);
      return pre >= bin;
    }
    if (pre > bin) atomicOr(&sm.sel[i >> 5], 1u << (i & 31));
    return pre == bin;
  };
  auto append = [&](uint32_t& slot, uint32_t key, int i) {
    if (slot < (uint32_t)kStreamSeg) {
      seg_idx[slot] = (uint32_t)i;
      seg_key[slot] = key;
    }
    ++slot;
  };
  if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0u) {
    const int n4 = L >> 2;
    const uint4* p4 = reinterpret_cast<const uint4*>(p);
    for (int base = 0; base < n4; base += kStreamVec * kStreamThreads) {
      uint4 key[kStreamVec];   // raw score bits, turned into keys in place
#pragma unroll
      for (int u = 0; u < kStreamVec; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < n4) key[u] = p4[i];
      }
      uint32_t m = 0u;
#pragma unroll
      for (int u = 0; u < kStreamVec; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < n4) {
          key[u].x = score_key(__uint_as_float(key[u].x));
          key[u].y = score_key(__uint_as_float(key[u].y));
          key[u].z = score_key(__uint_as_float(key[u].z));
          key[u].w = score_key(__uint_as_float(key[u].w));
          m |= (classify(key[u].x, 4 * i) ? 1u : 0u) << (4 * u);
          m |= (classify(key[u].y, 4 * i + 1) ? 2u : 0u) << (4 * u);
          m |= (classify(key[u].z, 4 * i + 2) ? 4u : 0u) << (4 * u);
          m |= (classify(key[u].w, 4 * i + 3) ? 8u : 0u) << (4 * u);
        }
      }
      uint32_t slot = stream_reserve(__popc(m), used);
      if (m) {
#pragma unroll
        for (int u = 0; u < kStreamVec; ++u) {
          const int i = base + u * kStreamThreads + tid;
          if ((m >> (4 * u)) & 1u) append(slot, key[u].x, 4 * i);
          if ((m >> (4 * u)) & 2u) append(slot, key[u].y, 4 * i + 1);
          if ((m >> (4 * u)) & 4u) append(slot, key[u].z, 4 * i + 2);
          if ((m >> (4 * u)) & 8u) append(slot, key[u].w, 4 * i + 3);
        }
      }
    }
    // The last L % 4 keys (fewer than 4, all in warp 0).
    if (warp == 0) {
      const int i = (n4 << 2) + tid;
      uint32_t key = 0u;
      bool hit = false;
      if (i < L) {
        key = score_key(p[i]);
        hit = classify(key, i);
      }
      uint32_t slot = stream_reserve(hit ? 1u : 0u, used);
      if (hit) append(slot, key, i);
    }
  } else {
    for (int base = 0; base < L; base += kStreamVec * kStreamThreads) {
      uint32_t key[kStreamVec];   // raw score bits, turned into keys in place
      const uint32_t* pb = reinterpret_cast<const uint32_t*>(p);
#pragma unroll
      for (int u = 0; u < kStreamVec; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < L) key[u] = pb[i];
      }
      uint32_t m = 0u;
#pragma unroll
      for (int u = 0; u < kStreamVec; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < L) {
          key[u] = score_key(__uint_as_float(key[u]));
          m |= (classify(key[u], i) ? 1u : 0u) << u;
        }
      }
      uint32_t slot = stream_reserve(__popc(m), used);
      if (m) {
#pragma unroll
        for (int u = 0; u < kStreamVec; ++u)
          if ((m >> u) & 1u) append(slot, key[u], base + u * kStreamThreads + tid);
      }
    }
  }
  if ((tid & 31) == 0) {
    sm.nseg[warp] = used;
    if (used > (uint32_t)kStreamSeg) sm.overflow = 1u;
  }
}

__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm) topk_stream_kernel(
    const float* __restrict__ scores, int64_t stride, int64_t rows,
    const int32_t* __restrict__ starts, const int32_t* __restrict__ ends, int k,
    int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char stream_smem_raw[];
  StreamSmem& sm = *reinterpret_cast<StreamSmem*>(stream_smem_raw);
  const int tid = threadIdx.x;
  uint32_t guess = kStreamNoGuess;

  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    __syncthreads();   // the previous row's shared state is no longer read
    int64_t s;
    const int L = stream_row_len(starts, ends, row, stride, s);
    int32_t* __restrict__ orow = out + row * (int64_t)k;
    if (L <= k) {   // every position is selected; no score is read
      for (int j = tid; j < k; j += kStreamThreads) orow[j] = j < L ? j : -1;
      continue;
    }
    const float* __restrict__ p = scores + row * stride + s;

    for (int i = tid; i < kStreamBins; i += kStreamThreads) sm.hist[i] = 0u;
    for (int i = tid; i < kStreamWords; i += kStreamThreads) {
      sm.sel[i] = 0u;
      sm.eqb[i] = 0u;
    }
    for (int i = tid; i < 3 * 256; i += kStreamThreads) (&sm.hsmall[0][0])[i] = 0u;
    if (tid == 0) sm.overflow = 0u;
    __syncthreads();

    stream_pass<true>(p, L, guess, sm);
    __syncthreads();

    // Threshold state: `P` is the threshold key's prefix with `shift` low
    // bits dropped; `take` of the keys with that prefix (the lowest
    // positions) are selected, out of `cnt`.
    uint32_t take = (uint32_t)k, P, cnt, b;
    stream_pick(sm.hist, kStreamBins, take, sm, P, cnt, take);
    const uint32_t P12 = P;
    const bool first_list_ok = guess <= P12 && sm.overflow == 0u;
    guess = P12 > 0u ? P12 - 1u : 0u;   // for this CTA's next row
    __syncthreads();
    if (!first_list_ok) {
      if (tid == 0) sm.overflow = 0u;
      __syncthreads();
      stream_pass<false>(p, L, P12, sm);
      __syncthreads();
    }
    // Each warp walks its own list segment.
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t nc = sm.nseg[warp];
    const uint32_t* const seg_idx = sm.cand_idx + warp * kStreamSeg;
    const uint32_t* const seg_key = sm.cand_key + warp * kStreamSeg;
    const bool list_ok = sm.overflow == 0u;
    if (first_list_ok) {
      // The list also holds keys above bin P12 and some below it.
      for (uint32_t c = lane; c < nc; c += 32) {
        const uint32_t idx = seg_idx[c];
        if ((seg_key[c] >> 20) > P12) atomicOr(&sm.sel[idx >> 5], 1u << (idx & 31u));
      }
    }

    // Resolve the low 20 bits among keys of bin P12: 8, 8, then 4 bits,
    // each pass with its own zeroed histogram and one block barrier (every
    // warp picks for itself from the same counts).
    int shift = 20;
    for (int pass = 0; pass < 3 && cnt != take; ++pass) {
      const int width = pass < 2 ? 8 : 4;
      const int nshift = shift - width;
      const uint32_t dmask = (1u << width) - 1u;
      uint32_t* const hs = sm.hsmall[pass];
      if (list_ok) {
        for (uint32_t c = lane; c < nc; c += 32) {
          const uint32_t key = seg_key[c];
          if ((key >> shift) == P) atomicAdd(&hs[(key >> nshift) & dmask], 1u);
        }
      } else {
        for (int i = tid; i < L; i += kStreamThreads) {
          const uint32_t key = score_key(p[i]);
          if ((key >> shift) == P) atomicAdd(&hs[(key >> nshift) & dmask], 1u);
        }
      }
      __syncthreads();
      if (width == 8) warp_pick<256>(hs, take, b, cnt, take);
      else warp_pick<16>(hs, take, b, cnt, take);
      P = (P << width) | b;
      shift = nshift;
    }

    // Mark the selected keys of bin P12; keys tied at the threshold go to
    // `eqb` when only some of them are selected.
    auto mark = [&](uint32_t key, uint32_t idx) {
      if ((key >> 20) != P12) return;
      const uint32_t hi = key >> shift;
      if (hi > P || (hi == P && cnt == take))
        atomicOr(&sm.sel[idx >> 5], 1u << (idx & 31u));
      else if (hi == P)
        atomicOr(&sm.eqb[idx >> 5], 1u << (idx & 31u));
    };
    if (list_ok) {
      for (uint32_t c = lane; c < nc; c += 32) mark(seg_key[c], seg_idx[c]);
    } else {
      for (int i = tid; i < L; i += kStreamThreads) mark(score_key(p[i]), (uint32_t)i);
    }
    __syncthreads();

    // Thread t owns bitmap words [4t, 4t + 4): positions [128t, 128t + 128).
    uint32_t w[kStreamWordsPerThread];
    uint32_t n = 0u;
    if (cnt != take) {
      // Keys equal at all 32 bits: the lowest `take` positions win.
      uint32_t e[kStreamWordsPerThread];
#pragma unroll
      for (int q = 0; q < kStreamWordsPerThread; ++q) {
        e[q] = sm.eqb[kStreamWordsPerThread * tid + q];
        n += __popc(e[q]);
      }
      uint32_t tot;
      uint32_t r = block_exclusive_scan_nt<kStreamThreads>(n, sm.scan_buf, tot);
      n = 0u;
#pragma unroll
      for (int q = 0; q < kStreamWordsPerThread; ++q) {
        w[q] = sm.sel[kStreamWordsPerThread * tid + q];
        if (r < take) w[q] |= first_set_bits(e[q], take - r);
        r += __popc(e[q]);
        n += __popc(w[q]);
      }
    } else {
#pragma unroll
      for (int q = 0; q < kStreamWordsPerThread; ++q) {
        w[q] = sm.sel[kStreamWordsPerThread * tid + q];
        n += __popc(w[q]);
      }
    }
    uint32_t total;
    uint32_t pos = block_exclusive_scan_nt<kStreamThreads>(n, sm.scan_buf, total);
#pragma unroll
    for (int q = 0; q < kStreamWordsPerThread; ++q) {
      uint32_t bits = w[q];
      const int base = 32 * (kStreamWordsPerThread * tid + q);
      while (bits) {
        const int e = __ffs(bits) - 1;
        bits &= bits - 1u;
        if (pos < (uint32_t)k) orow[pos] = base + e;
        ++pos;
      }
    }
  }
}


// ---------------------------------------------------------------------------
// Grid variant, for up to 256 rows of up to 131072 scores (8192 to 2^24
// scores in all): every row is spread over the whole GPU and read once. One
// cooperative launch of one 1024-thread CTA per SM, all resident at once,
// runs two phases separated by one grid barrier (a counter in the
// workspace, waited on with a bounded spin):
//   1. The score matrix (16-byte aligned) is viewed as rows of 256 scores;
//      each row of the batch is cut into 8192-score segments starting at
//      the view row that holds its first score, and the segments are dealt
//      to the CTAs in contiguous runs. A CTA streams its run through a
//      6-stage shared-memory ring, one tensor-map box (32 view rows, 32 KiB)
//      per segment issued by one thread and completing on the stage's
//      mbarrier. On the first segment of each row it touches (n in-row
//      scores) it takes a bound B: the 12-bit prefix bin holding the
//      segment's (3 k n / 2L + 32)-th largest key (every key when n is
//      smaller), a generous estimate of where the row's k-th largest key
//      lies. It then lists every score of its part of the row whose key is
//      at least B << 20, with its position: segment j of a row has its own
//      8192-entry slot of the row's list, warps exchange their counts across
//      the block barrier that ends the segment and write at their offsets,
//      and the segment's count and bound go to the workspace.
//   2. One CTA per row takes M, the largest bound any segment of the row
//      used. If at least k listed keys are >= M, the row's k-th largest key
//      is >= M >= every segment's bound, so every key of the top k was
//      listed, and the top k of the listed keys >= M is the answer. Otherwise
//      (rows whose first segments misjudge the rest, such as descending
//      rows) the CTA takes the whole row from the score matrix instead. It
//      selects by 12/8/8/4-bit histograms (ties at the full key take the
//      lowest positions), marks the selected positions in a shared-memory
//      bitmap and writes them in ascending order.
// The result is the same set as every other kernel's: which scores are
// listed, and in which order, only changes the work.

constexpr int kGrThreads = 1024;
constexpr int kGrPer = 8;                    // scores per thread per segment (two 16-byte groups)
constexpr int kGrSeg = kGrThreads * kGrPer;  // 8192 scores per segment
constexpr int kGrStages = 6;                 // ring stages (segments in flight)
constexpr int kGrView = 256;                 // scores per row of the 2D view
constexpr int kGrBins = 4096;
constexpr int kGrMaxRows = 256;
constexpr int64_t kGrMaxStride = 131072;
constexpr int64_t kGrMinScores = kGrSeg;
constexpr int64_t kGrMaxScores = int64_t(1) << 24;
constexpr int kGrWords = (int)(kGrMaxStride / 32);        // bitmap words of a row
constexpr int kGrWordsPerThread = kGrWords / kGrThreads;  // 4
constexpr int kGrTileQ = 8;                                // entries per thread per tile
constexpr int kGrTile = kGrThreads * kGrTileQ;
constexpr uint32_t kGrNoPos = 0xFFFFFFFFu;
constexpr long long kGrSpinCycles = 1ll << 31;   // about one second at the top SM clock
constexpr size_t kGrRingBytes = (size_t)kGrStages * kGrSeg * sizeof(float);   // dynamic, 192 KiB
static_assert(kGrRingBytes >= 2 * kGrWords * sizeof(uint32_t), "the bitmaps alias the ring");

// Workspace: a 256-byte header (the barrier counter, then the error word;
// zeroed before each launch), the entry count and the bound of every
// segment, then the lists: per row, ns_max slots of 8192 (key, position)
// entries, ns_max = ceil((stride + 255) / 8192) being the most segments a
// row of the matrix can have.
constexpr size_t kGrHeader = 256;
constexpr int kGrMaxSegsPerRow = (int)((kGrMaxStride + kGrView - 1 + kGrSeg - 1) / kGrSeg);   // 17
__host__ __device__ constexpr size_t gr_align(size_t b) { return (b + 255) & ~size_t(255); }
__host__ __device__ constexpr int64_t gr_ns_max(int64_t stride) {
  return (stride + kGrView - 1 + kGrSeg - 1) / kGrSeg;
}
__host__ __device__ constexpr size_t gr_segcnt_off() { return kGrHeader; }
__host__ __device__ constexpr size_t gr_segbound_off(int64_t R, int64_t nsm) {
  return gr_segcnt_off() + gr_align((size_t)(R * nsm) * sizeof(uint32_t));
}
__host__ __device__ constexpr size_t gr_list_off(int64_t R, int64_t nsm) {
  return gr_segbound_off(R, nsm) + gr_align((size_t)(R * nsm) * sizeof(uint32_t));
}

struct GridArgs {
  const float* scores;
  int64_t stride;
  int32_t rows;
  int32_t k;
  const int32_t* starts;
  const int32_t* ends;
  int32_t* out;
  uint32_t* hdr;        // [0]: barrier counter; [2]: error word
  uint32_t* segcnt;     // [rows][ns_max]: entries listed from each segment
  uint32_t* segbound;   // [rows][ns_max]: the key bound each segment listed from
  uint2* list;          // [rows][ns_max][8192]: (key, position)
  int32_t ns_max;
};

struct GridSmem {
  uint32_t seg_off[kGrMaxRows + 1];   // segments before row r; rows with L <= k have none
  int32_t len[kGrMaxRows];
  int32_t g0[kGrMaxRows];             // score element of the row's position 0
  alignas(16) uint32_t hist[kGrBins];   // 12-bit prefix counts; zero between uses (read as uint4)
  uint32_t h[3][256];                 // refinement histograms, one per pass
  uint32_t wsum[32];
  uint32_t pick[3];
  uint32_t wcnt[2][32];               // each warp's entries of a segment (by parity)
  uint32_t segpre[kGrMaxSegsPerRow + 1];   // phase 2: entries before each segment of the row
  uint32_t mkey;                      // phase 2: the row's bound M
  alignas(8) uint64_t full[kGrStages];   // ring stage landed (transfer count)
};

static_assert(offsetof(GridSmem, hist) % 16 == 0, "the histogram is read 16 bytes at a time");
static_assert(offsetof(GridSmem, full) % 8 == 0, "mbarriers are 8-byte aligned");

// Every CTA arrives once; thread 0 waits until all `target` CTAs have, for at
// most kGrSpinCycles, after which it sets the error word and goes on (the
// cooperative launch makes every CTA resident, so the wait always ends).
__device__ __forceinline__ void grid_barrier(uint32_t* counter, uint32_t target, uint32_t* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1u);
    const long long t0 = clock64();
    for (;;) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > kGrSpinCycles) {
        atomicOr(err, 1u);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
}

// The row holding segment `seg`: the last r with off[r] <= seg (off[0] = 0,
// off[R] > seg), which is never an empty row.
__device__ __forceinline__ int gr_row_of(const uint32_t* off, int R, uint32_t seg) {
  int lo = 0, hi = R;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= seg) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Where a segment lies: row r, segment j of the row, the segment's first
// score element A (a multiple of 256) and the row's elements [g0, gend).
// Thread t's scores of the segment are elements A + 4t + 4096 h + i
// (h = 0, 1; i = 0..3), at the same offsets in the ring stage.
struct GrSeg {
  int r;
  uint32_t j;
  int32_t A, g0, gend;
};

__device__ __forceinline__ void gr_locate(const GridSmem& sm, const GridArgs& a, uint32_t seg,
                                          GrSeg& c) {
  if (c.r < 0 || seg >= sm.seg_off[c.r + 1]) {
    c.r = gr_row_of(sm.seg_off, a.rows, seg);
    c.g0 = sm.g0[c.r];
    c.gend = c.g0 + sm.len[c.r];
  }
  c.j = seg - sm.seg_off[c.r];
  c.A = (c.g0 & ~(kGrView - 1)) + (int32_t)c.j * kGrSeg;
}

// One bit per in-row score of this thread (bit 4h + i).
__device__ __forceinline__ uint32_t gr_valid(const GrSeg& c, int tid) {
  if (c.A >= c.g0 && c.A + kGrSeg <= c.gend) return 0xFFu;   // an interior segment
  uint32_t v = 0u;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int32_t e = c.A + 4 * tid + 4096 * h + i;
      if (e >= c.g0 && e < c.gend) v |= 1u << (4 * h + i);
    }
  return v;
}

// Issues the copy of segment `c` into ring stage `st` (one thread): one box
// of 32 view rows. View rows past the map (the matrix's last partial view
// row and beyond) arrive as zeros.
__device__ __forceinline__ void gr_issue(const CUtensorMap* smap, GridSmem& sm, float* ring,
                                         const GrSeg& c, int st) {
  uint64_t* const bar = &sm.full[st];
  mbar_arrive_expect_tx(bar, kGrSeg * (uint32_t)sizeof(float));
  tma_load_box(smem_u32(ring + st * kGrSeg), smap, 0, c.A / kGrView, bar);
}

// This thread's eight scores of the segment from its ring stage. Scores in
// the matrix's last partial view row (elements from ncov on), which the map
// does not cover, are read from global memory.
__device__ __forceinline__ void gr_scores(const float* ring_stage, const GrSeg& c, int tid,
                                          uint32_t valid, int32_t ncov,
                                          const float* __restrict__ sc, float (&x)[kGrPer]) {
  const float4 v0 = *reinterpret_cast<const float4*>(ring_stage + 4 * tid);
  const float4 v1 = *reinterpret_cast<const float4*>(ring_stage + 4096 + 4 * tid);
  x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
  x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
  if (c.A + kGrSeg > ncov) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t e = c.A + 4 * tid + 4096 * h + i;
        if (((valid >> (4 * h + i)) & 1u) && e >= ncov) x[4 * h + i] = sc[e];
      }
  }
}

// Picks, among the 4096 bins of sm.hist (descending bin order), the bin
// holding the `take`-th largest key: sm.pick = (bin, keys above the bin,
// keys in the bin). Thread t reads (and clears) bins 4095 - 4t - q,
// q = 0..3. Ends with a block barrier.
constexpr int kGrBinsPerThread = kGrBins / kGrThreads;
static_assert(kGrBinsPerThread == 4, "one 16-byte read of bins per thread");
__device__ __forceinline__ void gr_pick4096(GridSmem& sm, uint32_t take) {
  const int tid = threadIdx.x;
  uint4* const p4 = reinterpret_cast<uint4*>(sm.hist + kGrBins - 4 - 4 * tid);
  const uint4 b4 = *p4;
  *p4 = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t c[4] = {b4.w, b4.z, b4.y, b4.x};
  uint32_t tot;
  uint32_t above = block_exclusive_scan_nt<kGrThreads>(c[0] + c[1] + c[2] + c[3], sm.wsum, tot);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (above < take && take <= above + c[q]) {
      sm.pick[0] = (uint32_t)(kGrBins - 1 - 4 * tid - q);
      sm.pick[1] = above;
      sm.pick[2] = c[q];
    }
    above += c[q];
  }
  __syncthreads();
}

// Phase 2 for row r. On entry the bitmaps, sm.hist and the refinement
// histograms are zero; they are zero again on return.
__device__ __forceinline__ void grid_resolve(const GridArgs& a, GridSmem& sm, uint32_t* sel,
                                             uint32_t* tie, int r) {
  const int tid = threadIdx.x;
  const int L = sm.len[r];
  const uint32_t k = (uint32_t)a.k;
  int32_t* __restrict__ orow = a.out + (int64_t)r * a.k;
  if (L <= a.k) {
    for (int j = tid; j < a.k; j += kGrThreads) orow[j] = j < L ? j : -1;
    return;
  }
  // The row's entries: segment j's list slot holds segcnt[r][j] of them.
  // Entry i of the row (segments in order) is entry i - segpre[j] of the
  // slot of the segment j with segpre[j] <= i < segpre[j + 1].
  const int ns = (int)(sm.seg_off[r + 1] - sm.seg_off[r]);   // <= kGrMaxSegsPerRow
  if (tid < 32) {
    const int lane = tid;
    uint32_t c = 0u, bnd = 0u;
    if (lane < ns) {
      c = __ldcg(a.segcnt + (int64_t)r * a.ns_max + lane);
      bnd = __ldcg(a.segbound + (int64_t)r * a.ns_max + lane);
    }
    if (c > (uint32_t)kGrSeg) c = (uint32_t)kGrSeg;   // only after a wait gave up
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
      bnd = max(bnd, __shfl_xor_sync(0xffffffffu, bnd, o));
    }
    if (lane <= kGrMaxSegsPerRow) sm.segpre[lane] = incl - c;
    if (lane == 0) sm.mkey = bnd;
  }
  __syncthreads();
  uint32_t n = sm.segpre[ns];
  uint32_t mkey = sm.mkey;
  if (n > (uint32_t)L) n = (uint32_t)L;   // only after a wait gave up
  const uint2* __restrict__ lr = a.list + (int64_t)r * a.ns_max * kGrSeg;
  const float* __restrict__ srow = a.scores + sm.g0[r];
  bool whole = false;   // entries from the score row itself
  uint2 e[kGrTileQ];
  // Slot q of tile t holds entry t * 8192 + q * 1024 + tid; entries below
  // the bound M are not candidates. All of a thread's addresses are worked
  // out before any load, so that its loads are in flight together.
  auto load_tile = [&](uint32_t t) {
    uint32_t off[kGrTileQ];
#pragma unroll
    for (int q = 0; q < kGrTileQ; ++q) {
      const uint32_t i = t * kGrTile + (uint32_t)(q * kGrThreads + tid);
      off[q] = i;
      if (!whole && i < n) {
        int lo = 0, hi = ns;   // segpre[lo] <= i < segpre[hi]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (sm.segpre[mid] <= i) lo = mid;
          else hi = mid;
        }
        off[q] = (uint32_t)lo * kGrSeg + (i - sm.segpre[lo]);
      }
    }
    if (whole) {
#pragma unroll
      for (int q = 0; q < kGrTileQ; ++q) {
        const uint32_t i = t * kGrTile + (uint32_t)(q * kGrThreads + tid);
        e[q] = i < n ? make_uint2(score_key(srow[i]), i) : make_uint2(0u, kGrNoPos);
      }
    } else {
#pragma unroll
      for (int q = 0; q < kGrTileQ; ++q) {
        const uint32_t i = t * kGrTile + (uint32_t)(q * kGrThreads + tid);
        e[q] = i < n ? __ldcg(lr + off[q]) : make_uint2(0u, kGrNoPos);
        if (e[q].y >= (uint32_t)L) e[q].y = kGrNoPos;
      }
    }
#pragma unroll
    for (int q = 0; q < kGrTileQ; ++q)
      if (e[q].x < mkey) e[q].y = kGrNoPos;
  };
  uint32_t ntiles = (n + kGrTile - 1) / kGrTile;
  uint32_t mine = 0u;
  for (uint32_t t = 0; t < ntiles; ++t) {
    load_tile(t);
#pragma unroll
    for (int q = 0; q < kGrTileQ; ++q) mine += e[q].y != kGrNoPos;
  }
  uint32_t cand;
  (void)block_exclusive_scan_nt<kGrThreads>(mine, sm.wsum, cand);
  if (cand < k) {
    // Fewer than k listed keys reach M: the lists may miss some of the top
    // k, so the row is taken whole.
    whole = true;
    n = (uint32_t)L;
    mkey = 0u;
    cand = n;
    ntiles = (n + kGrTile - 1) / kGrTile;
  }
  if (ntiles == 1 && whole) load_tile(0);   // (the lists' single tile is loaded already)
  const int nq = ntiles > 1 ? kGrTileQ : (int)((n + kGrThreads - 1) / kGrThreads);

  // The top 12 bits, then 8/8/4 as in the other kernels: prefix P at
  // `shift` dropped bits; `take` of the `cnt` candidates with that prefix are
  // selected.
  for (uint32_t t = 0; t < ntiles; ++t) {
    if (ntiles > 1) load_tile(t);
#pragma unroll
    for (int q = 0; q < kGrTileQ; ++q) {
      if (q >= nq) break;
      if (e[q].y != kGrNoPos) atomicAdd(&sm.hist[e[q].x >> 20], 1u);
    }
  }
  __syncthreads();
  gr_pick4096(sm, k);
  uint32_t P = sm.pick[0], take = k - sm.pick[1], cnt = sm.pick[2];
  int shift = 20;
  for (int pass = 0; pass < 3 && cnt != take; ++pass) {
    const int width = pass < 2 ? 8 : 4;
    const int nshift = shift - width;
    const uint32_t dmask = (1u << width) - 1u;
    uint32_t* const hs = sm.h[pass];
    for (uint32_t t = 0; t < ntiles; ++t) {
      if (ntiles > 1) load_tile(t);
#pragma unroll
      for (int q = 0; q < kGrTileQ; ++q) {
        if (q >= nq) break;
        if (e[q].y != kGrNoPos && (e[q].x >> shift) == P)
          atomicAdd(&hs[(e[q].x >> nshift) & dmask], 1u);
      }
    }
    __syncthreads();
    uint32_t b;
    if (width == 8) warp_pick<256>(hs, take, b, cnt, take);
    else warp_pick<16>(hs, take, b, cnt, take);
    P = (P << width) | b;
    shift = nshift;
  }
  const bool all_eq = cnt == take;
  for (uint32_t t = 0; t < ntiles; ++t) {
    if (ntiles > 1) load_tile(t);
#pragma unroll
    for (int q = 0; q < kGrTileQ; ++q) {
      if (q >= nq) break;
      if (e[q].y == kGrNoPos) continue;
      const uint32_t hi = e[q].x >> shift;
      const uint32_t bit = 1u << (e[q].y & 31u);
      if (hi > P || (hi == P && all_eq)) atomicOr(&sel[e[q].y >> 5], bit);
      else if (hi == P) atomicOr(&tie[e[q].y >> 5], bit);
    }
  }
  __syncthreads();

  // Thread t owns bitmap words [4t, 4t + 4): positions [128t, 128t + 128).
  const int nw = (L + 31) >> 5;
  uint32_t w[kGrWordsPerThread];
#pragma unroll
  for (int i = 0; i < kGrWordsPerThread; ++i) {
    const int wi = kGrWordsPerThread * tid + i;
    w[i] = wi < nw ? sel[wi] : 0u;
  }
  if (!all_eq) {
    uint32_t tw[kGrWordsPerThread], c = 0u;
#pragma unroll
    for (int i = 0; i < kGrWordsPerThread; ++i) {
      const int wi = kGrWordsPerThread * tid + i;
      tw[i] = wi < nw ? tie[wi] : 0u;
      c += __popc(tw[i]);
    }
    uint32_t tot;
    const uint32_t before = block_exclusive_scan_nt<kGrThreads>(c, sm.wsum, tot);
    if (before < take) {
      uint32_t rem = take - before;
#pragma unroll
      for (int i = 0; i < kGrWordsPerThread; ++i) {
        const uint32_t m = first_set_bits(tw[i], rem);
        w[i] |= m;
        rem -= __popc(m);
      }
    }
  }
  uint32_t c = 0u;
#pragma unroll
  for (int i = 0; i < kGrWordsPerThread; ++i) c += __popc(w[i]);
  uint32_t total;
  uint32_t pos = block_exclusive_scan_nt<kGrThreads>(c, sm.wsum, total);
  // Clear this thread's words and the histograms for the next row.
#pragma unroll
  for (int i = 0; i < kGrWordsPerThread; ++i) {
    const int wi = kGrWordsPerThread * tid + i;
    if (wi < nw) {
      sel[wi] = 0u;
      tie[wi] = 0u;
    }
  }
  for (int i = tid; i < 3 * 256; i += kGrThreads) (&sm.h[0][0])[i] = 0u;
  // Each thread stores its positions at its own slots. (Staging them in
  // shared memory for contiguous stores measured 0.8 µs slower on TP1.)
#pragma unroll
  for (int i = 0; i < kGrWordsPerThread; ++i) {
    const int base = 32 * (kGrWordsPerThread * tid + i);
    for (uint32_t m = w[i]; m; m &= m - 1u) {
      if (pos < k) orow[pos] = base + __ffs(m) - 1;
      ++pos;
    }
  }
}

__global__ void __launch_bounds__(kGrThreads, 1)
    topk_grid_kernel(const __grid_constant__ CUtensorMap smap, const GridArgs a) {
  __shared__ GridSmem sm;
  extern __shared__ __align__(128) float gr_ring[];   // [kGrStages][kGrSeg]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.rows;
  const uint32_t G = gridDim.x;
  const uint32_t k = (uint32_t)a.k;

  if (tid == 0) {
    for (int s = 0; s < kGrStages; ++s) mbar_init(&sm.full[s], 1);
    mbar_fence_init();
  }
  // Row table: clamped length, start and segment offsets of every row.
  uint32_t ns = 0u;
  if (tid < R) {
    const int64_t s = a.starts[tid];
    const int64_t e = a.ends[tid];
    int L = 0;
    if (s >= 0 && s <= a.stride) {
      int64_t L64 = e - s;
      if (L64 < 0) L64 = 0;
      if (L64 > a.stride - s) L64 = a.stride - s;
      L = (int)L64;
    }
    const int32_t g0 = (int32_t)(tid * a.stride + (s >= 0 && s <= a.stride ? s : 0));
    sm.len[tid] = L;
    sm.g0[tid] = g0;
    if (L > a.k) ns = (uint32_t)(((g0 & (kGrView - 1)) + L + kGrSeg - 1) / kGrSeg);
  }
  for (int i = tid; i < kGrBins; i += kGrThreads) sm.hist[i] = 0u;
  uint32_t S;
  const uint32_t ex = block_exclusive_scan_nt<kGrThreads>(ns, sm.wsum, S);
  if (tid <= R) sm.seg_off[tid] = ex;   // thread R's exclusive sum is the total
  __syncthreads();
  const uint32_t sb = (uint32_t)((uint64_t)S * blockIdx.x / G);
  const uint32_t se = (uint32_t)((uint64_t)S * (blockIdx.x + 1) / G);
  const int32_t ncov = (int32_t)(((int64_t)R * a.stride) & ~int64_t(kGrView - 1));

  // The ring: segment sb + i goes to stage i % kGrStages. Thread 0 fills the
  // stages; every thread waits for a stage's copies and reads its scores,
  // and after the block barrier that ends each segment thread 0 refills the
  // stage with the segment kGrStages further on. `par` holds the parity of
  // each stage's next phase.
  GrSeg ic, pc;
  uint32_t par = 0u;
  bool late = false;   // a ring wait gave up
  if (tid == 0) {
    ic.r = -1;
    for (int s = 0; s < kGrStages && sb + s < se; ++s) {
      gr_locate(sm, a, sb + s, ic);
      gr_issue(&smap, sm, gr_ring, ic, s);
    }
  }

  // Phase 1.
  pc.r = -1;
  int cur = -1;
  // A key is listed iff key >= lo_key. For 8 <= B <= 0xFF8 (0xFF8 is the
  // bin of +inf, the highest a key reaches) that is the float comparison
  // x >= lo_x, lo_x being the float whose key is lo_key: keys are monotone
  // in the float order, -0 and +0 compare equal as they should, and NaN (key
  // 0) compares false. Outside that range lo_x would be a NaN pattern; such
  // bounds compare keys.
  uint32_t lo_key = 0u;
  float lo_x = 0.f;
  bool by_float = false;
  uint32_t wpar = 0u;
  for (uint32_t seg = sb; seg < se; ++seg) {
    gr_locate(sm, a, seg, pc);
    const bool first = pc.r != cur;
    cur = pc.r;
    const uint32_t valid = gr_valid(pc, tid);
    float x[kGrPer];
    {
      const int st = (int)((seg - sb) % kGrStages);
      if (!mbar_wait(&sm.full[st], (par >> st) & 1u)) late = true;
      par ^= 1u << st;
      gr_scores(gr_ring + st * kGrSeg, pc, tid, valid, ncov, a.scores, x);
    }
    if (first) {
      // The bound from this segment's n in-row scores: the bin of its
      // (3 k n / 2L + 32)-th largest key.
#pragma unroll
      for (int q = 0; q < kGrPer; ++q)
        if ((valid >> q) & 1u) atomicAdd(&sm.hist[score_key(x[q]) >> 20], 1u);
      __syncthreads();
      const int32_t lo_e = pc.A > pc.g0 ? pc.A : pc.g0;
      const int32_t hi_e = pc.A + kGrSeg < pc.gend ? pc.A + kGrSeg : pc.gend;
      const uint32_t nseg = (uint32_t)(hi_e - lo_e);
      uint64_t t1 = 3ull * k * nseg / (2ull * (uint64_t)(pc.gend - pc.g0)) + 32u;
      if (t1 > nseg) t1 = nseg;
      gr_pick4096(sm, (uint32_t)t1);
      const uint32_t B = sm.pick[0];
      lo_key = B << 20;
      by_float = B >= 8u && B <= 0xFF8u;
      lo_x = __uint_as_float((lo_key & 0x80000000u) ? (lo_key & 0x7FFFFFFFu) : ~lo_key);
    }
    uint32_t m = 0u;
    if (by_float) {
#pragma unroll
      for (int q = 0; q < kGrPer; ++q)
        if (x[q] >= lo_x) m |= 1u << q;
    } else {
#pragma unroll
      for (int q = 0; q < kGrPer; ++q)
        if (score_key(x[q]) >= lo_key) m |= 1u << q;
    }
    m &= valid;
    const uint32_t cm = __popc(m);
    uint32_t incl = cm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sm.wcnt[wpar][warp] = incl;
    __syncthreads();   // every thread has read the stage; the warp counts are out
    {
      const uint32_t nx = seg + kGrStages;
      if (tid == 0 && nx < se) {
        gr_locate(sm, a, nx, ic);
        gr_issue(&smap, sm, gr_ring, ic, (int)((nx - sb) % kGrStages));
      }
    }
    // This warp's offset in the segment's slot: the counts of the warps
    // before it.
    const uint32_t wc = sm.wcnt[wpar][lane];
    uint32_t winc = wc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += y;
    }
    const uint32_t woff = __shfl_sync(0xffffffffu, winc - wc, warp);
    if (tid == 31) {   // the segment's total and bound
      a.segcnt[(int64_t)cur * a.ns_max + pc.j] = winc;
      a.segbound[(int64_t)cur * a.ns_max + pc.j] = lo_key;
    }
    if (m) {
      uint2* const ls = a.list + ((int64_t)cur * a.ns_max + pc.j) * kGrSeg;
      const uint32_t p0 = (uint32_t)(pc.A + 4 * tid - pc.g0);   // position of score q = 0
      uint32_t o = woff + incl - cm;
#pragma unroll
      for (int q = 0; q < kGrPer; ++q)
        if ((m >> q) & 1u)
          ls[o++] = make_uint2(score_key(x[q]), p0 + (uint32_t)(4096 * (q >> 2) + (q & 3)));
    }
    wpar ^= 1u;
  }
  if (late && tid == 0) atomicOr(a.hdr + 2, 4u);

  // Every copy issued has been waited for: the ring's space becomes the two
  // bitmaps of phase 2.
  uint32_t* const sel = reinterpret_cast<uint32_t*>(gr_ring);
  uint32_t* const tie = sel + kGrWords;
  for (int i = tid; i < 2 * kGrWords; i += kGrThreads) sel[i] = 0u;
  for (int i = tid; i < 3 * 256; i += kGrThreads) (&sm.h[0][0])[i] = 0u;
  grid_barrier(a.hdr, G, a.hdr + 2);
  pdl_trigger();

  // Phase 2: one CTA per row.
  for (int r = blockIdx.x; r < R; r += (int)G) {
    grid_resolve(a, sm, sel, tie, r);
    __syncthreads();
  }
}

}  // namespace

bool topk_grid_shape(int64_t rows, int64_t stride) {
  if (rows < 1 || rows > kGrMaxRows || stride > kGrMaxStride || rows * stride > kGrMaxScores ||
      rows * stride < kGrMinScores)
    return false;
  if (stride <= kRowMaxLen && rows >= kRowMinRows) return false;      // whole rows in shared memory
  if (stride <= kStreamMaxLen && rows >= kStreamMinRows) return false;  // the streaming grid
  return true;
}

size_t topk_workspace_bytes(int64_t rows, int64_t stride) {
  if (!topk_grid_shape(rows, stride)) return 0;
  const int64_t nsm = gr_ns_max(stride);
  return gr_list_off(rows, nsm) + (size_t)(rows * nsm) * kGrSeg * sizeof(uint2);
}

namespace {

// CTAs of one grid top-k launch on device `dev`: every CTA resident at once.
struct PerDeviceCount {
  std::atomic<int> v[PerDeviceOnce::kMaxDevices] = {};
};

cudaError_t grid_ctas(int dev, int* ctas) {
  static PerDeviceCount cache;
  const bool tracked = dev >= 0 && dev < PerDeviceOnce::kMaxDevices;
  if (tracked && (*ctas = cache.v[dev].load(std::memory_order_acquire)) > 0) return cudaSuccess;
  int sms = 0, occ = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, topk_grid_kernel, kGrThreads,
                                                    kGrRingBytes);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorCooperativeLaunchTooLarge;
  *ctas = sms * occ;
  if (tracked) cache.v[dev].store(*ctas, std::memory_order_release);
  return cudaSuccess;
}

cudaError_t launch_topk_grid(const float* scores, int64_t stride, int64_t rows,
                             const int32_t* starts, const int32_t* ends, int k, int32_t* out,
                             void* workspace, int dev, cudaStream_t stream) {
  static PerDeviceOnce grid_attr;
  cudaError_t e = set_max_dynamic_smem(grid_attr, dev, topk_grid_kernel, (int)kGrRingBytes);
  if (e != cudaSuccess) return e;
  int G = 0;
  e = grid_ctas(dev, &G);
  if (e != cudaSuccess) return e;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  e = cudaMemsetAsync(ws, 0, kGrHeader, stream);
  if (e != cudaSuccess) return e;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  // The score matrix as whole rows of 256 scores (a partial last view row is
  // left out of the map and read with plain loads).
  CUtensorMap smap;
  const cuuint64_t gdim[2] = {(cuuint64_t)kGrView, (cuuint64_t)(rows * stride / kGrView)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kGrView * sizeof(float)};
  const cuuint32_t box[2] = {(cuuint32_t)kGrView, (cuuint32_t)(kGrSeg / kGrView)};
  const cuuint32_t estride[2] = {1, 1};
  if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(scores), gdim, gstride, box,
          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  GridArgs a;
  a.scores = scores;
  a.stride = stride;
  a.rows = (int32_t)rows;
  a.k = k;
  a.starts = starts;
  a.ends = ends;
  a.out = out;
  a.hdr = reinterpret_cast<uint32_t*>(ws);
  const int64_t nsm = gr_ns_max(stride);
  a.segcnt = reinterpret_cast<uint32_t*>(ws + gr_segcnt_off());
  a.segbound = reinterpret_cast<uint32_t*>(ws + gr_segbound_off(rows, nsm));
  a.list = reinterpret_cast<uint2*>(ws + gr_list_off(rows, nsm));
  a.ns_max = (int32_t)nsm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kGrThreads);
  cfg.dynamicSmemBytes = kGrRingBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_grid_kernel, smap, a);
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t stride, int64_t rows, const int32_t* starts,
                        const int32_t* ends, int k, int32_t* out, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  // The kernel depends on the shapes alone, and the selected set is unique,
  // so the choice never changes the output:
  //  - 16 or more rows of up to 32K: one CTA per row, the whole row in
  //    shared memory (this leaves most SMs free, so the next kernel's CTAs
  //    become resident while it runs);
  //  - at least 256 rows of up to 64K: the streaming grid;
  //  - otherwise a cluster of up to 8 CTAs per row (rows of up to 128K);
  //  - longer rows: one CTA per row with passes over global memory.
  int dev = 0;
  cudaError_t e = stream_device(stream, &dev);
  if (e != cudaSuccess) return e;
  // The grid kernel reads the scores with tensor-map copies: their start must
  // be 16-byte aligned (other pointers take the kernels below).
  const size_t grid_ws = topk_workspace_bytes(rows, stride);
  if (grid_ws != 0 && workspace != nullptr && workspace_bytes >= grid_ws &&
      (reinterpret_cast<uintptr_t>(scores) & 15u) == 0u)
    return launch_topk_grid(scores, stride, rows, starts, ends, k, out, workspace, dev, stream);
  if (stride <= kRowMaxLen && rows >= kRowMinRows) {
    static PerDeviceOnce row_attr;
    e = set_max_dynamic_smem(row_attr, dev, topk_smem_kernel, (int)sizeof(RowSmem));
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_smem_kernel, dim3((unsigned)rows), dim3(kRowThreads), sizeof(RowSmem),
                      stream, 1u, scores, stride, starts, ends, k, out);
  }
  if (stride <= kStreamMaxLen && rows >= kStreamMinRows) {
    static PerDeviceOnce stream_attr;
    e = set_max_dynamic_smem(stream_attr, dev, topk_stream_kernel, (int)sizeof(StreamSmem));
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)sms * kStreamCtasPerSm;
    const int64_t grid = rows < slots ? rows : slots;
    return launch_pdl(topk_stream_kernel, dim3((unsigned)grid), dim3(kStreamThreads),
                      sizeof(StreamSmem), stream, 1u, scores, stride, rows, starts, ends, k, out);
  }
  // Cluster size from the row stride alone: about 8K keys per CTA, at most 8
  // CTAs; chunks are multiples of 128 keys.
  int64_t C = (stride + 8191) / 8192;
  if (C > kClMaxCluster) C = kClMaxCluster;
  const int64_t per = ((stride + C - 1) / C + 127) & ~int64_t(127);
  if (per > kClMaxChunk || rows * C > (int64_t)INT32_MAX) {
    return launch_pdl(topk_rows_kernel, dim3((unsigned)rows), dim3(kThreads), 0, stream, 1u, scores,
                      stride, starts, ends, k, out);
  }
  const size_t smem = sizeof(ClSmem) + (size_t)per * sizeof(uint32_t);
  static PerDeviceOnce cl_attr;
  e = set_max_dynamic_smem(cl_attr, dev, topk_cluster_kernel,
                           (int)(sizeof(ClSmem) + kClMaxChunk * sizeof(uint32_t)));
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_cluster_kernel, dim3((unsigned)(rows * C)), dim3(kClThreads), smem, stream,
                    (unsigned)C, scores, stride, starts, ends, k, out);
}

}  // namespace dsmla
