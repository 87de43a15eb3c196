// KV cache write: new latent rows into the paged cache.
//
// Row i goes to slot slots[i] = page * 64 + offset ("[Bugfix] Make DSV4
// sparse MLA work end-to-end for plain decode, MTP, and DSpark", section
// "What is fixed": slot = block_id * block_size + offset, with a guard so that
// padding rows never write into a real block). A negative slot is a padding
// row and writes nothing; a slot past the pool writes nothing and sets
// DS_DEVERR_PAGE.
//
// FP8 KV (MooreThreads/vllm-musa PR 178, optimisation table: the FP8 cache
// write, with each row's fp32 scale groups kept contiguous): per group of 128
// latent dims, scale = amax / 448 (1 for an all-zero group) and code =
// E4M3(x / scale), rounded to nearest with ties to even and saturating at
// +-448; the 64 bf16 rope dims are copied. The row layout is [0, 512) codes,
// [512, 528) the four fp32 scales, [528, 656) the rope. amax, the scale and
// x / scale are float32 values with correctly rounded float32 division, so
// every code is decided exactly as a float32 reference decides it.
//
// One warp per row: lane l holds latent chunks l and l + 32 (8 dims each), so
// the two 16-lane halves of the warp hold groups (0, 2) and (1, 3), and each
// group's amax is a 16-lane reduction. Loads and stores are 16 or 8 bytes
// per lane, coalesced. The kernel is HBM-bound: 1152 bytes read and 656
// written per row.

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dsmla {

namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kLatentChunks = 64;   // 16-byte chunks of the 512 latent dims
constexpr int kRowChunks = 72;      // 16-byte chunks of a 1152-byte bf16 row
constexpr int64_t kFp8RowBytes = 656;
constexpr int kErrPage = 2;         // DS_DEVERR_PAGE

__device__ __forceinline__ void bf16x8_to_float(uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Eight values divided by `scale` and rounded to E4M3 (nearest, ties to even,
// saturating), little-endian in a uint2.
__device__ __forceinline__ uint2 e4m3x8(const float* x, float scale) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 pair = make_float2(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale));
    const uint32_t b = (uint32_t)__nv_cvt_float2_to_fp8x2(pair, __NV_SATFINITE, __NV_E4M3);
    w[i >> 1] |= (b & 0xFFFFu) << (16 * (i & 1));
  }
  return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ float group_amax(const float* x) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;   // the same in the 16 lanes of a half-warp
}

__global__ void __launch_bounds__(32 * kWarpsPerCta) kv_write_fp8_kernel(
    const uint4* __restrict__ latent, int64_t n, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ pool, int64_t num_slots, int32_t* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + warp;
  if (row >= n) return;
  // The row's loads go out together with its slot's (a padding row's latent
  // is read and dropped), so a row costs one memory round trip, not two.
  const int64_t slot = slots[row];
  const uint4* src = latent + row * kRowChunks;
  const uint4 c0 = src[lane], c1 = src[lane + 32];
  uint4 rope = make_uint4(0u, 0u, 0u, 0u);
  if (lane < 8) rope = src[kLatentChunks + lane];
  if (slot < 0) return;   // padding row
  if (slot >= num_slots) {
    if (lane == 0 && err != nullptr) atomicOr(err, kErrPage);
    return;
  }
  float x0[8], x1[8];
  bf16x8_to_float(c0, x0);
  bf16x8_to_float(c1, x1);
  const float a0 = group_amax(x0), a1 = group_amax(x1);   // groups lane/16 and 2 + lane/16
  const float s0 = a0 > 0.0f ? __fdiv_rn(a0, 448.0f) : 1.0f;
  const float s1 = a1 > 0.0f ? __fdiv_rn(a1, 448.0f) : 1.0f;
  uint8_t* dst = pool + slot * kFp8RowBytes;
  *reinterpret_cast<uint2*>(dst + 8 * lane) = e4m3x8(x0, s0);
  *reinterpret_cast<uint2*>(dst + 256 + 8 * lane) = e4m3x8(x1, s1);
  if ((lane & 15) == 0) {
    const int g = lane >> 4;
    reinterpret_cast<float*>(dst + 512)[g] = s0;
    reinterpret_cast<float*>(dst + 512)[2 + g] = s1;
  }
  if (lane < 8) reinterpret_cast<uint4*>(dst + 528)[lane] = rope;
}

__global__ void __launch_bounds__(32 * kWarpsPerCta) kv_write_bf16_kernel(
    const uint4* __restrict__ latent, int64_t n, const int64_t* __restrict__ slots,
    uint4* __restrict__ pool, int64_t num_slots, int32_t* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + warp;
  if (row >= n) return;
  const int64_t slot = slots[row];
  const uint4* src = latent + row * kRowChunks;
  const uint4 c0 = src[lane], c1 = src[lane + 32];   // chunks lane, lane + 32
  uint4 c2 = make_uint4(0u, 0u, 0u, 0u);             // chunk lane + 64 (lanes 0-7)
  if (lane < kRowChunks - 64) c2 = src[lane + 64];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0 && err != nullptr) atomicOr(err, kErrPage);
    return;
  }
  uint4* dst = pool + slot * kRowChunks;
  dst[lane] = c0;
  dst[lane + 32] = c1;
  if (lane < kRowChunks - 64) dst[lane + 64] = c2;
}

}  // namespace

cudaError_t launch_kv_cache_write(const void* latent, int64_t n, const int64_t* slots,
                                  int kv_dtype, void* pool, int64_t num_pages, int32_t* err,
                                  cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const dim3 grid((unsigned)((n + kWarpsPerCta - 1) / kWarpsPerCta));
  const int64_t num_slots = num_pages * 64;
  if (kv_dtype == 1)
    return launch_pdl(kv_write_fp8_kernel, grid, dim3(32 * kWarpsPerCta), 0, stream, 1u,
                      reinterpret_cast<const uint4*>(latent), n, slots,
                      reinterpret_cast<uint8_t*>(pool), num_slots, err);
  return launch_pdl(kv_write_bf16_kernel, grid, dim3(32 * kWarpsPerCta), 0, stream, 1u,
                    reinterpret_cast<const uint4*>(latent), n, slots,
                    reinterpret_cast<uint4*>(pool), num_slots, err);
}

}  // namespace dsmla
