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
  // step 9's 224-column tile kernel: tile columns 0 .. wide_cols-1 are wide_n wide,
  // the rest narrow_n (both multiples of 16, at most the kernel's tile width), so
  // that the CTA pairs' tiles add up to nearly the same width; narrow_n = 0: every
  // tile column is the kernel's full width
  int32_t wide_cols, wide_n, narrow_n;
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

// The logistic function 1 / (1 + e^-t) = 1 / (1 + 2^(-t log2 e)) on the special
// function unit: one ex2.approx and one rcp.approx (each within a few ulp of
// fp32; the rounding of t log2 e moves the result by at most |t| 2^-24
// relatively, where it is not already saturated at 0 or 1).  Large negative t
// gives 2^big = inf and 1 / inf = 0; large positive t gives 1 / (1 + 0) = 1.
__device__ __forceinline__ float logistic(float t) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return r;
}

// the activation is a compile-time choice: each fused kernel carries the code
// of one activation only (the writeback code shares the SM's instruction cache
// with the producer and MMA warps).  SiLU is x * logistic(x); the tanh form of
// GeLU uses 0.5 (1 + tanh(u)) = logistic(2 u), so both cost two SFU operations
// and a few FMAs per element, which matters on the path that holds an
// accumulator until its epilogue is done.
template <int ACT>
__device__ __forceinline__ float epi_activation(float x) {
  if constexpr (ACT == EPI_ACT_RELU) {
    return fmaxf(x, 0.f);
  } else if constexpr (ACT == EPI_ACT_SILU) {
    return x * logistic(x);
  } else if constexpr (ACT == EPI_ACT_GELU_TANH) {
    const float k2 = 1.5957691216057308f;  // 2 sqrt(2 / pi)
    return x * logistic(k2 * (x + 0.044715f * x * x * x));
  } else if constexpr (ACT == EPI_ACT_GELU_ERF) {
    return 0.5f * x * (1.f + erff(x * 0.7071067811865476f));
  } else {
    return x;
  }
}

// Loads 128 bytes of row `row` of the residual from column col0 on (64 bf16 or
// 32 fp32 columns) into 32 words, zero for 16-byte groups past column N (C's
// rows are 16-byte multiples, so each group lies wholly inside or outside C).
// The caller checks row < M.
// With v8 (the row segment 32-byte aligned and 32-column groups wholly inside
// or outside C, which the caller checks) the loads are 32 bytes wide.
template <typename OutT>
__device__ __forceinline__ void load_residual128(uint32_t (&r)[32], const KParams& p, int32_t row, int32_t col0,
                                                 bool v8 = false) {
  constexpr int per16 = 16 / (int)sizeof(OutT);
  const uint4* src =
      reinterpret_cast<const uint4*>(reinterpret_cast<const OutT*>(p.residual) + (int64_t)row * p.out_ld + col0);
  if (v8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t t[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (col0 + 2 * per16 * j < p.N) ld_global_v8(src + 2 * j, t);
#pragma unroll
      for (int e = 0; e < 8; ++e) r[8 * j + e] = t[e];
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 u = (col0 + per16 * j < p.N) ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
    r[4 * j] = u.x;
    r[4 * j + 1] = u.y;
    r[4 * j + 2] = u.z;
    r[4 * j + 3] = u.w;
  }
}

// Copies columns col0 .. col0+BN-1 of the per-column vector v (N fp32 values,
// 4-byte aligned) into shared memory dst (BN floats, 16-byte aligned), 0 past
// column N; the lanes of one warp share the work.
template <int BN>
__device__ __forceinline__ void stage_columns(float* dst, const float* v, int32_t col0, int32_t N, uint32_t lane) {
#pragma unroll
  for (int j = (int)lane; j < BN; j += 32) dst[j] = (col0 + j < N) ? __ldg(v + col0 + j) : 0.f;
}

// The residual of 32 columns of row `row` from column col0 (64 bytes of bf16 or 128
// of fp32) into r (16 or 32 words), 0 for 16-byte groups past column N; with v8 in
// 32-byte loads (the caller checks that rows are 32-byte aligned and N a multiple
// of 16).  The caller checks row < M.
template <typename OutT>
__device__ __forceinline__ void load_residual_cols32(uint32_t* r, const KParams& p, int32_t row, int32_t col0,
                                                     bool v8) {
  constexpr int per16 = 16 / (int)sizeof(OutT);  // columns per 16 bytes
  constexpr int NQ = 32 / per16;                 // 16-byte groups: 4 (bf16) or 8 (fp32)
  const uint4* src =
      reinterpret_cast<const uint4*>(reinterpret_cast<const OutT*>(p.residual) + (int64_t)row * p.out_ld + col0);
  if (v8) {
#pragma unroll
    for (int j = 0; j < NQ / 2; ++j) {
      uint32_t t[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (col0 + 2 * per16 * j < p.N) ld_global_v8(src + 2 * j, t);
#pragma unroll
      for (int e = 0; e < 8; ++e) r[8 * j + e] = t[e];
    }
  } else {
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      const uint4 u = (col0 + per16 * j < p.N) ? __ldg(src + j) : make_uint4(0u, 0u, 0u, 0u);
      r[4 * j] = u.x;
      r[4 * j + 1] = u.y;
      r[4 * j + 2] = u.z;
      r[4 * j + 3] = u.w;
    }
  }
}

// Applies the fused epilogue to 32 consecutive fp32 accumulator values of one
// row (columns col0 .. col0+31), in place:
//   x = act(acc * sa * scale_b[col] + bias[col]) + residual,
// each term only when present.  sa is scale_a[row] (0 past row M), read by the
// caller.  r holds the residual of these columns as load_residual128 left it
// (bf16: 16 words of column pairs; fp32: 32 words), used when has_res.  Bias
// and scale_b come from sbias / sscale_b when given (shared-memory copies of
// these 32 columns, 16-byte aligned, staged by the caller), else from global
// memory: as float4 (every lane of a warp reads the same columns) when the 32
// columns lie inside C and are 16-byte aligned, else one by one, as 0 past
// column N.
template <typename OutT, int ACT>
__device__ __forceinline__ void apply_epilogue32(uint32_t* v, const KParams& p, int32_t col0, float sa, bool has_res,
                                                 const uint32_t* r, const float* sbias = nullptr,
                                                 const float* sscale_b = nullptr) {
  float x[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
  if (p.scale_a != nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] *= sa;
  }
  const bool whole = col0 + 32 <= p.N;
  if (p.scale_b != nullptr && sscale_b != nullptr) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = reinterpret_cast<const float4*>(sscale_b)[q];
      x[4 * q] *= f.x;
      x[4 * q + 1] *= f.y;
      x[4 * q + 2] *= f.z;
      x[4 * q + 3] *= f.w;
    }
  } else if (p.scale_b != nullptr) {
    if (whole && ((reinterpret_cast<uintptr_t>(p.scale_b + col0) & 15u) == 0)) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p.scale_b + col0) + q);
        x[4 * q] *= f.x;
        x[4 * q + 1] *= f.y;
        x[4 * q + 2] *= f.z;
        x[4 * q + 3] *= f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] *= (col0 + j < p.N) ? __ldg(p.scale_b + col0 + j) : 0.f;
    }
  }
  if (p.bias != nullptr && sbias != nullptr) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 f = reinterpret_cast<const float4*>(sbias)[q];
      x[4 * q] += f.x;
      x[4 * q + 1] += f.y;
      x[4 * q + 2] += f.z;
      x[4 * q + 3] += f.w;
    }
  } else if (p.bias != nullptr) {
    if (whole && ((reinterpret_cast<uintptr_t>(p.bias + col0) & 15u) == 0)) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p.bias + col0) + q);
        x[4 * q] += f.x;
        x[4 * q + 1] += f.y;
        x[4 * q + 2] += f.z;
        x[4 * q + 3] += f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] += (col0 + j < p.N) ? __ldg(p.bias + col0 + j) : 0.f;
    }
  }
  if constexpr (ACT != EPI_ACT_NONE) {
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = epi_activation<ACT>(x[j]);
  }
  if (has_res) {
    if constexpr (sizeof(OutT) == 4) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] += __uint_as_float(r[j]);
    } else {
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[m]));
        x[2 * m] += f.x;
        x[2 * m + 1] += f.y;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(x[j]);
}

// First column and width of tile column tn: bn wide, or (balanced widths, see
// KParams) wide_n / narrow_n wide.
__device__ __forceinline__ void tile_columns(const KParams& p, int32_t tn, int32_t bn, int32_t& c0, int32_t& w) {
  if (p.narrow_n == 0) {
    c0 = tn * bn;
    w = bn;
  } else if (tn < p.wide_cols) {
    c0 = tn * p.wide_n;
    w = p.wide_n;
  } else {
    c0 = p.wide_cols * p.wide_n + (tn - p.wide_cols) * p.narrow_n;
    w = p.narrow_n;
  }
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
