// kernel_common.cuh -- parameters, tile rasterisation and store helpers shared
// by the GEMM kernels (device side of the library only).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace dgb {

// status codes written to the device status word (first writer wins); the
// low byte says which wait gave up
enum : uint32_t {
  DEV_TIMEOUT_BASE = 0x7100u,
  WAIT_PRODUCER_EMPTY = 0x7101u,
  WAIT_MMA_FULL = 0x7102u,
  WAIT_MMA_ACC_EMPTY = 0x7103u,
  WAIT_EPI_ACC_FULL = 0x7104u,
  WAIT_RING_FULL = 0x7105u,
  WAIT_RING_EMPTY = 0x7106u,
  WAIT_CLC = 0x7107u,
  WAIT_LADDER_MMA = 0x7108u,
  WAIT_LADDER_TMA = 0x7109u,
  WAIT_DRAIN = 0x710Au,
};

// test hook: the producer leaves out one TMA load of the first stage while
// still expecting its bytes, so the consumer's bounded wait must give up
constexpr uint32_t DEBUG_SKIP_ONE_LOAD = 1u;

struct KParams {
  int32_t M, N, K;
  uint32_t idesc;        // tcgen05 instruction descriptor
  int32_t tiles_m;       // tiles (cluster tiles for the pair kernels) along M
  int32_t tiles_n;
  int32_t raster_group;  // tile rows per raster group
  int32_t stages;        // SMEM ring depth
  uint32_t* status;      // [0] status word, [1] tile counter, [2] finished-cluster counter
  int32_t* visits;       // optional per-tile visit counts (tests), may be null
  uint64_t timeout_ns;   // bound on every wait
  uint32_t debug_flags;
  int32_t out_ld;        // leading dimension of C (= N)
  const uint16_t* A;     // raw operands for the kernels that copy with threads
  const uint16_t* B;
  void* C;
};

// Grouped (L2-aware) raster order: consecutive tile ids walk down a group of
// `group` tile rows before moving one tile column to the right, so the CTAs
// running at the same time share A row panels and B column panels in L2.
__device__ __forceinline__ void raster_tile(int32_t tile, int32_t tiles_m, int32_t tiles_n,
                                            int32_t group, int32_t& tm, int32_t& tn) {
  const int32_t per_group = group * tiles_n;
  const int32_t g = tile / per_group;
  const int32_t first_m = g * group;
  const int32_t rows = min(group, tiles_m - first_m);
  const int32_t r = tile - g * per_group;
  tm = first_m + r % rows;
  tn = r / rows;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

// Store one row segment of 32 fp32 accumulator values (columns col0..col0+31)
// with bounds checks; vector stores when the whole segment is inside and aligned.
template <typename OutT>
__device__ __forceinline__ void store_row32(OutT* C, int64_t ld, int32_t row, int32_t col0,
                                            int32_t N, const uint32_t (&v)[32]) {
  OutT* dst = C + (int64_t)row * ld + col0;
  if constexpr (sizeof(OutT) == 4) {
    if (col0 + 32 <= N && (((uintptr_t)dst) & 15u) == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 q = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        reinterpret_cast<uint4*>(dst)[j] = q;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < N) reinterpret_cast<uint32_t*>(dst)[j] = v[j];
    }
  } else {
    if (col0 + 32 <= N && (((uintptr_t)dst) & 15u) == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 q = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                             pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        reinterpret_cast<uint4*>(dst)[j] = q;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < N) dst[j] = __float2bfloat16_rn(__uint_as_float(v[j]));
    }
  }
}

// first address at or after `p` whose shared-window offset is 1024-byte aligned
// (the 128-byte swizzle pattern is anchored to 1024-byte boundaries)
__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  const uint32_t s = smem_u32(p);
  return p + (((s + 1023u) & ~1023u) - s);
}

}  // namespace dgb
