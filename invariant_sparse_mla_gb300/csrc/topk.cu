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
// One CTA owns one row; there is no inter-CTA communication and no spin on
// another CTA. The selected set is unique (the order is total), so the
// output is bit-exact and batch-independent by construction.
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
#include <stdint.h>

#include "internal.h"

namespace dsmla {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = kThreads * 4;  // elements per block-wide step
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;

__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of one uint32 per thread; `total` gets the
// block sum. Ends with a barrier so `buf` may be reused right away.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* buf,
                                                         uint32_t& total) {
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

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t stride, int64_t rows, const int32_t* starts,
                        const int32_t* ends, int k, int32_t* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  topk_rows_kernel<<<(unsigned)rows, kThreads, 0, stream>>>(scores, stride, starts, ends, k, out);
  return cudaGetLastError();
}

}  // namespace dsmla
