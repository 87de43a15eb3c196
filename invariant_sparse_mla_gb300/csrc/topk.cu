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

#include <atomic>

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
// Cluster variant: the row is cut into C contiguous chunks, one per CTA of a
// thread-block cluster (C <= 8). Each CTA keeps its chunk's keys in shared
// memory, so the row is read from HBM exactly once. The per-CTA digit
// histograms are summed through distributed shared memory after a hardware
// cluster barrier (every CTA of a cluster is co-scheduled, so the barrier
// cannot wait on a CTA that never runs); every CTA then derives the same
// threshold. Histograms are double buffered, so one cluster barrier per digit
// pass suffices. The compaction counts (greater, equal) per warp with
// ballots, exchanges the per-CTA totals through distributed shared memory to
// get each chunk's carry-in, and writes the output in ascending order.

constexpr int kMaxChunk = 16384;       // keys per CTA (64 KiB of shared memory)
constexpr int kMaxCluster = 8;

// Reads of another CTA's shared memory. They are only issued after a cluster
// barrier that orders the writes, so they need no memory clobber and may be
// overlapped freely.
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

__device__ __forceinline__ uint4 dsmem_ld4(const uint32_t* local_ptr, uint32_t rank) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(dsmem_addr(local_ptr, rank)));
  return v;
}

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

__global__ void __launch_bounds__(kThreads) topk_cluster_kernel(
    const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ ends, int k, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint32_t keys[];  // this CTA's chunk
  __shared__ __align__(16) uint32_t hist[2][kBins];
  __shared__ uint32_t scan_buf[32];
  __shared__ uint32_t pick[3];
  __shared__ uint32_t wcount[kWarps][2];        // per-warp (greater, equal) counts
  __shared__ uint32_t cta_tot[2];               // this CTA's totals, read by later ranks

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_size();
  const uint32_t crank = cluster_rank();
  const int64_t row = blockIdx.x / C;
  const int64_t s = starts[row];
  const int64_t e = ends[row];
  int64_t L = 0;
  if (s >= 0 && s <= stride) {
    L = e - s;
    if (L < 0) L = 0;
    if (L > stride - s) L = stride - s;
  }
  int32_t* __restrict__ orow = out + row * (int64_t)k;
  if (L <= (int64_t)k) {  // uniform over the cluster: no cluster barrier is used
    if (crank == 0)
      for (int j = tid; j < k; j += kThreads) orow[j] = (int64_t)j < L ? j : -1;
    return;
  }

  // Chunk of this CTA: [c0, c0 + n), chunks a multiple of 4 elements long.
  const int64_t per = ((L + C - 1) / C + 3) & ~int64_t(3);
  const int64_t c0 = per * crank;
  const int n = (int)(c0 >= L ? 0 : (L - c0 < per ? L - c0 : per));
  const float* __restrict__ p = scores + row * stride + s + c0;
  const bool aligned = (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;

  for (int i = tid; i < kBins; i += kThreads) {
    hist[0][i] = 0u;
    hist[1][i] = 0u;
  }
  __syncthreads();

  // Load the chunk (8 x 16 B per thread in flight), store keys, histogram
  // of the top 11 bits.
  if (aligned) {
    const int n4 = n >> 2;
    const float4* p4 = reinterpret_cast<const float4*>(p);
    for (int base = 0; base < n4; base += 8 * kThreads) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kThreads + tid;
        if (i < n4) v[u] = p4[i];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kThreads + tid;
        if (i < n4) {
          uint4 kk;
          kk.x = score_key(v[u].x);
          kk.y = score_key(v[u].y);
          kk.z = score_key(v[u].z);
          kk.w = score_key(v[u].w);
          reinterpret_cast<uint4*>(keys)[i] = kk;
          atomicAdd(&hist[0][kk.x >> 21], 1u);
          atomicAdd(&hist[0][kk.y >> 21], 1u);
          atomicAdd(&hist[0][kk.z >> 21], 1u);
          atomicAdd(&hist[0][kk.w >> 21], 1u);
        }
      }
    }
    for (int i = (n4 << 2) + tid; i < n; i += kThreads) {
      const uint32_t kk = score_key(p[i]);
      keys[i] = kk;
      atomicAdd(&hist[0][kk >> 21], 1u);
    }
  } else {
    for (int base = 0; base < n; base += 8 * kThreads) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kThreads + tid;
        if (i < n) v[u] = p[i];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kThreads + tid;
        if (i < n) {
          const uint32_t kk = score_key(v[u]);
          keys[i] = kk;
          atomicAdd(&hist[0][kk >> 21], 1u);
        }
      }
    }
  }

  uint32_t prefix = 0u;
  int shift = 32;
  uint32_t take = (uint32_t)k;
  for (int pass = 0; pass < 3; ++pass) {
    const int width = pass < 2 ? 11 : 10;
    const int nshift = shift - width;
    const uint32_t nbins = 1u << width;
    const int buf = pass & 1;
    if (pass > 0) {
      if (pass == 2) {
        // hist[0] was last read by the other CTAs in pass 0, before the
        // cluster barrier of pass 1. (hist[1] starts out zeroed.)
        for (int i = tid; i < kBins; i += kThreads) hist[0][i] = 0u;
        __syncthreads();
      }
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t kk = keys[i];
        if ((kk >> shift) == prefix) atomicAdd(&hist[buf][(kk >> nshift) & (nbins - 1u)], 1u);
      }
    }
    __syncthreads();
    cluster_sync_all();

    // Cluster-wide counts of this thread's bins (descending bin order): the
    // thread's four bins are contiguous, so one 16-byte remote load per rank.
    uint32_t c[kBinsPerThread];
    uint32_t mine = 0u;
    const int bhi = (int)nbins - 1 - tid * kBinsPerThread;   // highest of the four
    {
      uint4 acc = make_uint4(0u, 0u, 0u, 0u);
      if (bhi >= kBinsPerThread - 1) {
        uint4 part[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < (int)C) part[r] = dsmem_ld4(&hist[buf][bhi - 3], (uint32_t)r);
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
          if (r < (int)C) {
            acc.x += part[r].x;
            acc.y += part[r].y;
            acc.z += part[r].z;
            acc.w += part[r].w;
          }
      }
      c[0] = acc.w;  // bin bhi
      c[1] = acc.z;
      c[2] = acc.y;
      c[3] = acc.x;  // bin bhi - 3
      mine = acc.x + acc.y + acc.z + acc.w;
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
    if (cnt == take) break;  // same decision in every CTA of the cluster
  }

  // Ordered compaction. Warp w owns the contiguous segment [w*seg, w*seg+seg)
  // of the chunk, read 32 keys at a time.
  const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int w0 = warp * seg;
  const int w1 = min(n, w0 + seg);
  uint32_t ngt = 0u, neq = 0u;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    uint32_t hi = 0u;
    const bool in = i < w1;
    if (in) hi = keys[i] >> shift;
    ngt += __popc(__ballot_sync(0xffffffffu, in && hi > prefix));
    neq += __popc(__ballot_sync(0xffffffffu, in && hi == prefix));
  }
  if (lane == 0) {
    wcount[warp][0] = ngt;
    wcount[warp][1] = neq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t g = 0u, q = 0u;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t a = wcount[w][0], b2 = wcount[w][1];
      wcount[w][0] = g;
      wcount[w][1] = q;
      g += a;
      q += b2;
    }
    cta_tot[0] = g;
    cta_tot[1] = q;
  }
  __syncthreads();
  cluster_sync_all();
  // Carry-in of this chunk: the totals of the lower-ranked CTAs, read in
  // parallel by warp 0 and shared through shared memory.
  __shared__ uint32_t carry[2];
  if (warp == 0) {
    uint32_t cg = 0u, ce = 0u;
    if ((uint32_t)lane < crank) {
      cg = dsmem_ld(&cta_tot[0], (uint32_t)lane);
      ce = dsmem_ld(&cta_tot[1], (uint32_t)lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cg += __shfl_xor_sync(0xffffffffu, cg, o);
      ce += __shfl_xor_sync(0xffffffffu, ce, o);
    }
    if (lane == 0) {
      carry[0] = cg;
      carry[1] = ce;
    }
  }
  __syncthreads();
  uint32_t g = carry[0] + wcount[warp][0];
  uint32_t qe = carry[1] + wcount[warp][1];
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    uint32_t hi = 0u;
    const bool in = i < w1;
    if (in) hi = keys[i] >> shift;
    const bool is_gt = in && hi > prefix;
    const bool is_eq = in && hi == prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t my_g = g + __popc(bg & lt_mask);
    const uint32_t my_e = qe + __popc(be & lt_mask);
    if (is_gt) orow[my_g + min(my_e, take)] = (int32_t)(c0 + i);
    else if (is_eq && my_e < take) orow[my_g + my_e] = (int32_t)(c0 + i);
    g += __popc(bg);
    qe += __popc(be);
  }
  // No CTA may exit while another can still read its shared memory.
  cluster_sync_all();
}


// ---------------------------------------------------------------------------
// Streaming variant for many rows of up to 65536 scores: one CTA per row, no
// cluster. The row is read from global memory once; while it streams in,
// each key's top 16 bits go to shared memory (2 bytes per score, 128 KB for
// the longest row) and a histogram of its top 12 bits is built. A second
// pass over shared memory refines the threshold to 16 bits. Only if the
// threshold bucket still holds more keys than needed are the low 16 bits
// read back from global memory (L2-resident by then), for the keys of that
// bucket alone, in two 8-bit passes. The ordered compaction reads the
// prefixes from shared memory and re-reads full keys only for that bucket.

constexpr int kStreamThreads = 1024;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kStreamMaxLen = 65536;
constexpr int kStreamBins = 4096;   // top 12 key bits
constexpr int kStreamBinsPerThread = kStreamBins / kStreamThreads;
constexpr int64_t kStreamMinRows = 256;   // below this the cluster kernel spreads a row wider

// Picks, among `nbins` bins counted in `hist` (descending bin order), the bin
// holding the `take`-th largest key. Every thread returns the same (bin,
// count of that bin, take within that bin).
__device__ __forceinline__ void stream_pick(const uint32_t* hist, int nbins, uint32_t take,
                                            uint32_t* scan_buf, uint32_t* pick, uint32_t& bin,
                                            uint32_t& cnt, uint32_t& take_in_bin) {
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
  uint32_t above = block_exclusive_scan_nt<kStreamThreads>(mine, scan_buf, total);
#pragma unroll
  for (int q = 0; q < kStreamBinsPerThread; ++q) {
    const int b = nbins - 1 - (tid * kStreamBinsPerThread + q);
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
  __syncthreads();
}

__global__ void __launch_bounds__(kStreamThreads, 1) topk_stream_kernel(
    const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ starts,
    const int32_t* __restrict__ ends, int k, int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint16_t pre[];   // top 16 key bits of each score
  __shared__ uint32_t hist[kStreamBins];
  __shared__ uint32_t scan_buf[32];
  __shared__ uint32_t pick[3];
  __shared__ uint32_t wcount[kStreamWarps][2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int64_t s = starts[row];
  const int64_t e = ends[row];
  int64_t L64 = 0;
  if (s >= 0 && s <= stride) {
    L64 = e - s;
    if (L64 < 0) L64 = 0;
    if (L64 > stride - s) L64 = stride - s;
  }
  int32_t* __restrict__ orow = out + row * (int64_t)k;
  if (L64 <= (int64_t)k) {
    for (int j = tid; j < k; j += kStreamThreads) orow[j] = (int64_t)j < L64 ? j : -1;
    return;
  }
  const int L = (int)L64;   // <= kStreamMaxLen
  const float* __restrict__ p = scores + row * stride + s;
  const bool aligned = (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;

  for (int i = tid; i < kStreamBins; i += kStreamThreads) hist[i] = 0u;
  __syncthreads();

  // Pass A: stream the row (8 x 16 bytes per thread in flight), keep the top
  // 16 key bits, histogram the top 12.
  if (aligned) {
    const int n4 = L >> 2;
    const float4* p4 = reinterpret_cast<const float4*>(p);
    for (int base = 0; base < n4; base += 8 * kStreamThreads) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < n4) v[u] = p4[i];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < n4) {
          const uint32_t k0 = score_key(v[u].x), k1 = score_key(v[u].y);
          const uint32_t k2 = score_key(v[u].z), k3 = score_key(v[u].w);
          reinterpret_cast<uint2*>(pre)[i] =
              make_uint2((k0 >> 16) | (k1 & 0xFFFF0000u), (k2 >> 16) | (k3 & 0xFFFF0000u));
          atomicAdd(&hist[k0 >> 20], 1u);
          atomicAdd(&hist[k1 >> 20], 1u);
          atomicAdd(&hist[k2 >> 20], 1u);
          atomicAdd(&hist[k3 >> 20], 1u);
        }
      }
    }
    for (int i = (n4 << 2) + tid; i < L; i += kStreamThreads) {
      const uint32_t kk = score_key(p[i]);
      pre[i] = (uint16_t)(kk >> 16);
      atomicAdd(&hist[kk >> 20], 1u);
    }
  } else {
    for (int base = 0; base < L; base += 8 * kStreamThreads) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < L) v[u] = p[i];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kStreamThreads + tid;
        if (i < L) {
          const uint32_t kk = score_key(v[u]);
          pre[i] = (uint16_t)(kk >> 16);
          atomicAdd(&hist[kk >> 20], 1u);
        }
      }
    }
  }
  __syncthreads();

  // Threshold: prefix P of the key at `shift` resolved bits, `take` of the
  // keys equal to it are selected (the lowest positions).
  uint32_t take = (uint32_t)k, P, cnt, b;
  int shift = 20;
  stream_pick(hist, kStreamBins, take, scan_buf, pick, P, cnt, take);
  if (cnt != take) {
    // Pass B (shared memory only): next 4 bits among keys with prefix P.
    if (tid < 16) hist[tid] = 0u;
    __syncthreads();
    for (int i = tid; i < L; i += kStreamThreads) {
      const uint32_t v = pre[i];
      if ((v >> 4) == P) atomicAdd(&hist[v & 15u], 1u);
    }
    __syncthreads();
    stream_pick(hist, 16, take, scan_buf, pick, b, cnt, take);
    P = (P << 4) | b;
    shift = 16;
    // Passes C and D: low 16 bits, read back for the keys of bucket P only.
    for (int pass = 0; pass < 2 && cnt != take; ++pass) {
      const int nshift = shift - 8;
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
      for (int i = tid; i < L; i += kStreamThreads) {
        if ((uint32_t)pre[i] == (P >> (16 - shift))) {
          const uint32_t kk = score_key(p[i]);
          if ((kk >> shift) == P) atomicAdd(&hist[(kk >> nshift) & 255u], 1u);
        }
      }
      __syncthreads();
      stream_pick(hist, 256, take, scan_buf, pick, b, cnt, take);
      P = (P << 8) | b;
      shift = nshift;
    }
  }

  // Ordered compaction: warp w owns the contiguous segment [w*seg, w*seg+seg).
  const uint32_t p16 = P >> (shift >= 16 ? 0 : 16 - shift);   // bucket at 16 bits
  auto classify = [&](int i, bool& gt, bool& eq) {
    const uint32_t v = pre[i];
    if (shift >= 16) {
      const uint32_t hi = v >> (shift - 16);
      gt = hi > P;
      eq = hi == P;
    } else if (v != p16) {
      gt = v > p16;
      eq = false;
    } else {
      const uint32_t hi = score_key(p[i]) >> shift;
      gt = hi > P;
      eq = hi == P;
    }
  };
  const int seg = ((L + kStreamWarps - 1) / kStreamWarps + 31) & ~31;
  const int w0 = warp * seg;
  const int w1 = min(L, w0 + seg);
  uint32_t ngt = 0u, neq = 0u;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    bool gt = false, eq = false;
    if (i < w1) classify(i, gt, eq);
    ngt += __popc(__ballot_sync(0xffffffffu, gt));
    neq += __popc(__ballot_sync(0xffffffffu, eq));
  }
  if (lane == 0) {
    wcount[warp][0] = ngt;
    wcount[warp][1] = neq;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t cg = wcount[lane][0], ce = wcount[lane][1];
    const uint32_t og = cg, oe = ce;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t yg = __shfl_up_sync(0xffffffffu, cg, o);
      const uint32_t ye = __shfl_up_sync(0xffffffffu, ce, o);
      if (lane >= o) {
        cg += yg;
        ce += ye;
      }
    }
    wcount[lane][0] = cg - og;   // exclusive
    wcount[lane][1] = ce - oe;
  }
  __syncthreads();
  uint32_t g = wcount[warp][0];
  uint32_t qe = wcount[warp][1];
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    bool gt = false, eq = false;
    if (i < w1) classify(i, gt, eq);
    const uint32_t bg = __ballot_sync(0xffffffffu, gt);
    const uint32_t be = __ballot_sync(0xffffffffu, eq);
    const uint32_t my_g = g + __popc(bg & lt_mask);
    const uint32_t my_e = qe + __popc(be & lt_mask);
    if (gt) orow[my_g + min(my_e, take)] = i;
    else if (eq && my_e < take) orow[my_g + my_e] = i;
    g += __popc(bg);
    qe += __popc(be);
  }
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t stride, int64_t rows, const int32_t* starts,
                        const int32_t* ends, int k, int32_t* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  // Many rows of up to 64K scores: one streaming CTA per row. Fewer rows
  // (or longer ones): a cluster per row, so that one row's work is spread
  // over several SMs. The selected set is unique, so the kernel choice never
  // changes the output.
  if (stride <= kStreamMaxLen && rows >= kStreamMinRows) {
    const size_t smem = ((size_t)stride * sizeof(uint16_t) + 15) & ~size_t(15);
    static std::atomic<bool> stream_attr{false};
    if (!stream_attr.load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(topk_stream_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(kStreamMaxLen * sizeof(uint16_t)));
      if (e != cudaSuccess) return e;
      stream_attr.store(true, std::memory_order_release);
    }
    topk_stream_kernel<<<(unsigned)rows, kStreamThreads, smem, stream>>>(scores, stride, starts,
                                                                         ends, k, out);
    return cudaGetLastError();
  }
  // Cluster size from the row stride alone: about 8K keys per CTA, at most 8
  // CTAs. Rows longer than 8 x 16K keys take the single-CTA kernel.
  int64_t C = (stride + 8191) / 8192;
  if (C > kMaxCluster) C = kMaxCluster;
  const int64_t per = ((stride + C - 1) / C + 3) & ~int64_t(3);
  if (per > kMaxChunk || rows * C > (int64_t)INT32_MAX) {
    topk_rows_kernel<<<(unsigned)rows, kThreads, 0, stream>>>(scores, stride, starts, ends, k, out);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)per * sizeof(uint32_t);
  static std::atomic<bool> attr_set{false};
  if (!attr_set.load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kMaxChunk * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_set.store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, scores, stride, starts, ends, k, out);
}

}  // namespace dsmla
