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
  WAIT_SK_PARTIAL = 0x710Bu,
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
  // fused writeback epilogue (steps 7-9): C = act(acc + bias[col]) + residual[row][col]
  const float* bias;     // N fp32 values, or null
  const void* residual;  // M x N in C's type, row-major (ld = out_ld), or null
  int32_t act;           // EPI_ACT_*
  // operand layouts (steps 7-9): bit 0 = A stored K x M (M-major), bit 1 = B stored K x N (N-major)
  uint32_t layout;
  // element kind of A and B (steps 7-9): 0 = fp16 / bf16 (kind::f16), 1 = 8-bit float
  // (kind::f8f6f4), 2 = 8-bit float with MX block scales (kind::mxf8f6f4)
  int32_t mma_kind;
  int32_t bk;            // K elements per 128-byte stage row: 64 (16-bit) or 128 (8-bit)
  // fused-epilogue dequantisation: acc * scale_a[row] * scale_b[col] before the bias
  const float* scale_a;  // M fp32 values, or null
  const float* scale_b;  // N fp32 values, or null
  // stream-K (steps 7-9): fp32 workspace of one slot per cluster and one flag per
  // writeback warp of each slot (zero between launches)
  float* sk_ws;
  uint32_t* sk_flags;
};

constexpr uint32_t LAYOUT_A_MN = 1u;
constexpr uint32_t LAYOUT_B_MN = 2u;

// activations of the fused epilogue
enum : int32_t {
  EPI_ACT_NONE = 0,
  EPI_ACT_RELU = 1,
  EPI_ACT_SILU = 2,       // x * sigmoid(x)
  EPI_ACT_GELU_TANH = 3,  // 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
  EPI_ACT_GELU_ERF = 4,   // 0.5 x (1 + erf(x / sqrt(2)))
};

// the activation is a compile-time choice: each fused kernel carries the code
// of one activation only (the writeback code shares the SM's instruction cache
// with the producer and MMA warps)
template <int ACT>
__device__ __forceinline__ float epi_activation(float x) {
  if constexpr (ACT == EPI_ACT_RELU) {
    return fmaxf(x, 0.f);
  } else if constexpr (ACT == EPI_ACT_SILU) {
    return x * __frcp_rn(1.f + expf(-x));  // correctly rounded reciprocal
  } else if constexpr (ACT == EPI_ACT_GELU_TANH) {
    const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
    return 0.5f * x * (1.f + tanhf(k0 * (x + 0.044715f * x * x * x)));
  } else if constexpr (ACT == EPI_ACT_GELU_ERF) {
    return 0.5f * x * (1.f + erff(x * 0.7071067811865476f));
  } else {
    return x;
  }
}

// Applies the fused epilogue to n consecutive fp32 accumulator values of one row
// (columns col0 .. col0+n-1), in place.  bias is read through L1 (every lane of
// a warp reads the same columns); the residual row segment with 16-byte loads
// when it lies wholly inside C, element by element at the edges.
template <typename OutT, int n, int ACT>
__device__ __forceinline__ void apply_epilogue(uint32_t* v, const KParams& p, int32_t row, int32_t col0) {
  float x[n];
#pragma unroll
  for (int j = 0; j < n; ++j) x[j] = __uint_as_float(v[j]);
  if (p.scale_a != nullptr) {
    const float sa = (row < p.M) ? __ldg(p.scale_a + row) : 0.f;
#pragma unroll
    for (int j = 0; j < n; ++j) x[j] *= sa;
  }
  if (p.scale_b != nullptr) {
#pragma unroll
    for (int j = 0; j < n; ++j) x[j] *= (col0 + j < p.N) ? __ldg(p.scale_b + col0 + j) : 0.f;
  }
  if (p.bias != nullptr) {
#pragma unroll
    for (int j = 0; j < n; ++j) x[j] += (col0 + j < p.N) ? __ldg(p.bias + col0 + j) : 0.f;
  }
  if constexpr (ACT != EPI_ACT_NONE) {
#pragma unroll
    for (int j = 0; j < n; ++j) x[j] = epi_activation<ACT>(x[j]);
  }
  if (p.residual != nullptr && row < p.M) {
    const OutT* r = reinterpret_cast<const OutT*>(p.residual) + (int64_t)row * p.out_ld + col0;
    constexpr int per16 = 16 / (int)sizeof(OutT);
    if (col0 + n <= p.N) {
#pragma unroll
      for (int q = 0; q < n / per16; ++q) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(r) + q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        if constexpr (sizeof(OutT) == 4) {
#pragma unroll
          for (int t = 0; t < 4; ++t) x[q * 4 + t] += __uint_as_float(w[t]);
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[t]));
            x[q * 8 + 2 * t] += f.x;
            x[q * 8 + 2 * t + 1] += f.y;
          }
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < n; ++j) {
        if (col0 + j < p.N) {
          if constexpr (sizeof(OutT) == 4) {
            x[j] += r[j];
          } else {
            x[j] += __bfloat162float(r[j]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < n; ++j) v[j] = __float_as_uint(x[j]);
}

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
