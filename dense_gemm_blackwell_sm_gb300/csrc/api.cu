// api.cu -- the C ABI (include/gemm.h): argument validation, the planner that
// picks a kernel variant / tile / ring depth / raster / launch size, TMA
// descriptor encoding and caching, launches, and device-status checks.
#include <algorithm>
#include <vector>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>

#include <cudaTypedefs.h>

#include "gemm.h"
#include "idesc.h"
#include "kernel_common.cuh"
#include "launch.h"

using namespace dgb;

struct gemm_plan_s {
  int64_t M, N, K;
  int64_t ldc;  // leading dimension of C in elements (N, or wider for a block of a larger C)
  gemm_dtype_t dtype;
  bool in_bf16, out_f32;
  bool in_f8, in_e5m2;  // 8-bit float inputs (E4M3 or E5M2)
  bool in_mx;           // ... with MX block scales (gemm_plan_run_mx)
  int variant, sched, stages, raster_group;
  int wide_cols = 0, wide_n = 0, narrow_n = 0;  // two tile widths (224-column step 9), see KParams
  int device, num_sms;
  int grid_units;  // CTAs (variants 3-6) or clusters (7-9) launched
  int split_k;     // GEMV_TC: requested CTAs per 128-row block along K (0 = automatic)
  int ks_split;    // step 7: CTAs of a cluster sharing one tile's K range (0 = whole tiles)
  int cg, consumers;
  int tile_m, tile_n, tiles_m, tiles_n;
  size_t smem;
  uint64_t timeout_ns;
  uint32_t debug_flags;
  int32_t flags;      // GEMM_FLAG_*
  int32_t layout;     // GEMM_LAYOUT_*
  int32_t gemv_pf_rows;  // GEMV: weight rows prefetched into L2 before the programmatic wait
  uint32_t* scratch;  // [0] status word, [1] tile counter, [2] finished counter
  float* sk_ws;       // stream-K workspace (one slot per cluster), or null
  uint32_t* sk_flags; // stream-K flags (one per writeback warp of each slot), or null
  size_t sk_flag_bytes;
  int32_t* visits;
  dgb::LaunchSpec spec;   // kernel, launch shape and SMEM, fixed at plan time
  dgb::LaunchSpec spec_epi[5];  // the fused-epilogue kernel per activation, made on first use
  bool epi_ready[5];
  int epi_tiles_m[5], epi_tiles_n[5], epi_stages[5];  // its tiling, per activation
  dgb::KParams kbase;     // kernel parameters that do not depend on the pointers
  dgb::TgParams tgbase;   // same, for the tensor-core GEMV
  // TMA descriptors by operand role (0 = A, 1 = B, 2 = C) and pointer, least
  // recently used replaced first, so rotating between buffers re-encodes nothing
  struct MapEntry {
    const void* ptr;
    int role;
    uint64_t used;
    CUtensorMap map;
  };
  static constexpr int kMapCache = 24;
  MapEntry maps[kMapCache];
  uint64_t map_clock;
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int64_t kMaxDim = (int64_t)1 << 31;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_fn_ready() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D row-major tensor [outer][inner], tiles of box_outer x box_inner elements
// landing in SMEM with the 128-byte swizzle; out-of-range elements read as 0.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, uint64_t row_elems = 0) {
  if (!encode_fn_ready()) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(row_elems ? row_elems : inner) * (uint64_t)esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// MX scales of B seen as a 4-D byte tensor [row blocks][K blocks][4 rows][128 B]
// of 512-byte blocks; one box of 128 x 4 x 1 x `box_blocks` brings the blocks of
// that many consecutive 128-row groups for one K block (rows past the array read
// as 0).
bool encode_mx_pairs(CUtensorMap* m, const void* ptr, uint64_t k_blocks, uint64_t row_blocks, uint32_t box_blocks) {
  if (!encode_fn_ready()) return false;
  cuuint64_t dims[4] = {128, 4, k_blocks, row_blocks};
  cuuint64_t strides[3] = {128, 512, 512 * k_blocks};
  cuuint32_t box[4] = {128, 4, 1, box_blocks};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int out_bytes(gemm_dtype_t dt) {
  return (dt == GEMM_F16_F32 || dt == GEMM_BF16_F32 || dt == GEMM_E4M3_F32 || dt == GEMM_E5M2_F32 ||
          dt == GEMM_MXE4M3_F32 || dt == GEMM_MXE5M2_F32)
             ? 4
             : 2;
}

bool is_mx(gemm_dtype_t dt) { return dt >= GEMM_MXE4M3_F32 && dt <= GEMM_MXE5M2_BF16; }

bool is_f8(gemm_dtype_t dt) { return (dt >= GEMM_E4M3_F32 && dt <= GEMM_E5M2_BF16) || is_mx(dt); }

bool is_e5m2(gemm_dtype_t dt) {
  return dt == GEMM_E5M2_F32 || dt == GEMM_E5M2_BF16 || dt == GEMM_MXE5M2_F32 || dt == GEMM_MXE5M2_BF16;
}

int in_bytes(gemm_dtype_t dt) { return is_f8(dt) ? 1 : 2; }
// K blocks of one 128-byte stage row (64 16-bit or 128 8-bit elements)
int64_t k_blocks(int64_t K, gemm_dtype_t dt) { return (K + (is_f8(dt) ? 127 : 63)) / (is_f8(dt) ? 128 : 64); }

// The TMA-store writeback of variants 7-9 needs rows of C to start 16-byte aligned.
bool c_rows_tma_ok(int64_t N, gemm_dtype_t dt) { return (N * out_bytes(dt)) % 16 == 0; }

gemm_status_t validate_sizes(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype) {
  if ((int)dtype < 0 || (int)dtype > GEMM_MXE5M2_BF16) return GEMM_ERR_UNSUPPORTED_DTYPE;
  if (M < 1 || N < 1 || K < 1 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return GEMM_ERR_INVALID_ARG;
  if ((K * in_bytes(dtype)) % 16 != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;  // TMA row pitch
  return GEMM_OK;
}

gemm_status_t current_device(int* dev, int* sms) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (cudaGetDevice(dev) != cudaSuccess) return GEMM_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (major != 10 || minor != 3) return GEMM_ERR_ARCH;
  return GEMM_OK;
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Time of the warp-specialised steps, in units of one SM's MMA time per output
// element and K block: the waves of resident clusters the tiles take, times a
// tile's area over the SMs of its cluster, times (K blocks + the step's fixed
// cost per tile, in K blocks), over the step's per-SM rate relative to step 9.
// Fitted on GB300 bf16: step 8 against step 7 at equal SM counts (1024 x 4096,
// 2048 x 2048, 512 x 8192 with K = 1024 ... 8192) gives a rate ratio of 1.21 and
// fixed costs of 23 and 12 K blocks; 8192^3 (1967, 1750, 1551 TFLOP/s for steps 9,
// 8, 7) puts step 9 at 1.12 x step 8, and short K on large outputs (4096 x 14336 x
// 1024: step 9 1456, step 7 1323; 8192^2 x 1024: 1412, 1353) gives step 9 a fixed
// cost near 22 K blocks.  Stream-K (step 9 only) spreads the whole area evenly.
constexpr double kRate9 = 1.0, kRate8 = 0.89, kRate7 = 0.735;
constexpr double kFixed9 = 22.0, kFixed8 = 24.0, kFixed7 = 12.0;
double ws_tile_cost(int64_t M, int64_t N, int tile_m, int tile_n, int cluster_sms, int units, double rate,
                    int64_t kb, double fixed) {
  const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + tile_n - 1) / tile_n);
  const int64_t waves = (tiles + units - 1) / units;
  return (double)waves * tile_m * tile_n / cluster_sms * ((double)kb + fixed) / rate;
}
// Stream-K on step v's 256-column tiles: `tiles` tiles on `units` resident
// clusters, kb K blocks.  Its time in K blocks of one tile is the tiles' work spread
// evenly plus x0 + x1 * kb for the split tiles' partial sums; whole tiles take
// waves * (kb + fixed).  Fitted on GB300 bf16 with the variants timed interleaved
// (M 2048 / 4096, N 2560 - 5120, K 2048 - 8192): step 8 with stream-K on 4096 x 2560
// (160 tiles, 70 % of three waves) 1162 against 1063 TFLOP/s at K = 2048, 1429
// against 1213 at 4096; step 9 on the same shape (80 tiles, 53 % of two waves) 938
// against 1014 at 2048 and 1305 against 1198 at 4096 (a split 512 x 256 tile carries
// twice the partial sums of a step-8 tile).  Returns that time where the automatic
// plan takes stream-K: it is shorter, whole tiles fill less than max_fill of their
// waves (at 84 % step 7 lost 3-7 % and step 8 gained at most 5 %), and kb >= min_kb
// (below, the partial sums outweigh the idle clusters: 4096 x 2560 x 1024 on step 9
// 627 against 771); otherwise -1.
struct StreamKModel {
  double fixed, x0, x1, max_fill;
  int64_t min_kb;
};
StreamKModel stream_k_model(int v) {
  if (v == GEMM_VARIANT_S9_TWO_CONSUMERS) return {kFixed9, 40.0, 0.0, 0.7, 64};
  if (v == GEMM_VARIANT_S8_CTA_PAIR) return {kFixed8, 28.0, 0.16, 0.8, 32};
  return {kFixed7, 28.0, 0.16, 0.8, 32};
}
double ws_stream_k_time(int v, int64_t tiles, int64_t units, int64_t kb) {
  const StreamKModel m = stream_k_model(v);
  if (units < 1 || tiles < units || kb < m.min_kb) return -1.0;
  const int64_t waves = (tiles + units - 1) / units;
  if ((double)tiles / ((double)waves * units) >= m.max_fill) return -1.0;
  const double sk = (double)tiles / units * ((double)kb + m.fixed) + m.x0 + m.x1 * (double)kb;
  return sk < (double)waves * ((double)kb + m.fixed) ? sk : -1.0;
}
// ws_tile_cost of step v (tile_m rows per cluster tile, cluster_sms SMs, rate) with
// its whole tiles, or with stream-K where the automatic plan takes it
double ws_cost_with_stream_k(int v, int64_t M, int64_t N, int tile_m, int cluster_sms, int units, double rate,
                             int64_t kb, double whole) {
  const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + 255) / 256);
  const double sk = ws_stream_k_time(v, tiles, units, kb);
  return sk < 0 ? whole : std::min(whole, sk * tile_m * 256 / cluster_sms / rate);
}
// Step 9's automatic tiling: 0 = 512 x 256 whole tiles, 1 = 512 x 224 whole tiles
// (taken when they finish at least 3 % sooner), 2 = stream-K on 512 x 256 tiles
// (allow_stream_k); *cost receives its ws_tile_cost
int s9_tiling(int64_t M, int64_t N, int64_t kb, int units, bool allow_stream_k, double* cost) {
  const double c256 = ws_tile_cost(M, N, 512, 256, 2, units, kRate9, kb, kFixed9);
  const double c224 = ws_tile_cost(M, N, 512, 224, 2, units, kRate9, kb, kFixed9);
  int t = (c224 < 0.97 * c256) ? 1 : 0;
  double c = t ? c224 : c256;
  if (allow_stream_k) {
    const double sk = ws_cost_with_stream_k(GEMM_VARIANT_S9_TWO_CONSUMERS, M, N, 512, 2, units, kRate9, kb, c);
    if (sk < c) {
      t = 2;
      c = sk;
    }
  }
  if (cost) *cost = c;
  return t;
}

// Launch time at short K (fewer than 32 K blocks, where plans keep whole tiles and
// never default to stream-K), in microseconds: a ramp per launch plus, per wave of
// tiles, a fixed part and a part per K block.  Least-squares fits to bf16 launches
// with whole tiles on 152 SMs (M and N from 2048 to 14336, K from 256 to 2048; every
// fit within 13 %).  There the fixed costs are a large part of a tile, and
// ws_tile_cost, whose per-tile costs were set at K >= 1024, overrates step 9:
// 4096 x 4096 x 512 runs at 880 TFLOP/s on step 7 against 795 on step 9, 2048 x 4096
// x 512 at 704 against 644, 4096 x 8192 x 1024 at 1327 against 1283.
struct ShortKFit {
  double ramp, per_kb, per_wave;
};
constexpr ShortKFit kShort9{3.94, 0.592, 3.57}, kShort8{5.49, 0.333, 1.54}, kShort7{3.25, 0.369, 0.98};
double short_k_time(const ShortKFit& f, int64_t M, int64_t N, int tile_m, int tile_n, int units, int64_t kb) {
  const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + tile_n - 1) / tile_n);
  const double waves = (double)((tiles + units - 1) / units);
  return f.ramp + waves * (f.per_kb * (double)kb + f.per_wave);
}

// Automatic variant: the decode GEMV with CUDA-core FMAs for one or two rows,
// with warp-level MMAs on registers for up to 8, on the tcgen05 Tensor Core for
// up to 16 rows; the plain-store persistent kernel when C's rows are not 16-byte
// aligned for TMA stores; step 7 (with its K split over a cluster) for outputs
// whose 128 x 256 tiles fill at most half the SMs and have K blocks to split;
// otherwise the warp-specialised step whose tiles finish soonest by ws_tile_cost
// (step 9 with 512 x 256 or 512 x 224 tiles or stream-K, step 8, step 7), or, below
// 32 K blocks, by short_k_time.
// Measured against the former rule (the largest tile that gives every CTA pair a
// tile): 2048 x 4096 x 4096 step 9 1550 TFLOP/s against step 8 1364; 256 x 14336 x
// 4096 step 8 970 against step 7 862; 1024 x 8192 x 8192 step 9 1682 against 1466.
// Clusters of c one-CTA-per-SM kernels resident at once (cudaOccupancyMaxActiveClusters
// on the 152-SM GB300: its GPCs hold 15 clusters of 8 and 23 of 6), scaled to sms.
int cluster_capacity(int c, int sms) {
  static const int cap152[9] = {0, 152, 76, 46, 36, 28, 23, 15, 15};
  if (c < 1 || c > 8) return 0;
  return (int)((int64_t)cap152[c] * sms / 152);
}

// The K split (2-4 slices, 0 = none) for tiles of cg CTAs (128 x 256 per CTA: cg 1
// step 7, cg 2 step 8's pair): the most slices that keep 16 K blocks each, one CTA
// per SM, and all clusters resident at once (16 clusters of 8 do not fit: the
// 1024 x 1024 x 4096 pairs split 4 ways ran at 315 TFLOP/s, 3 ways fit).
int ks_split_for(int64_t M, int64_t N, int64_t kb, int sms, int cg) {
  const int64_t tiles = ((M + 128 * cg - 1) / (128 * cg)) * ((N + 255) / 256);
  for (int s = 4; s >= 2; --s) {
    if (s * cg > 8 || kb / s < 16 || tiles * s * cg > sms || tiles > cluster_capacity(s * cg, sms)) continue;
    return s;
  }
  return 0;
}

int auto_variant(int64_t M, int64_t N, int64_t K, gemm_dtype_t dt, int sms) {
  if (M <= 2 && gemv_smem_bytes((int)M, (int)K) <= 200 * 1024) return GEMM_VARIANT_GEMV;
  if (M >= 3 && M <= 8) return GEMM_VARIANT_GEMV;
  if (M <= 16) return GEMM_VARIANT_GEMV_TC;
  if (!c_rows_tma_ok(N, dt)) return GEMM_VARIANT_S6_PERSISTENT;
  const int pairs = std::max(1, sms / 2);
  const int64_t tiles7 = ((M + 127) / 128) * ((N + 255) / 256);
  const int64_t kb = k_blocks(K, dt);
  if (tiles7 * 2 <= sms && kb >= 32) {
    // K split over a cluster: on step 8's CTA pairs (a pair's CTA loads 32 KB per K
    // block, a step-7 CTA 48 KB) unless they would leave more SMs idle: 512 x 4096 x
    // 4096 783 -> 869 TFLOP/s, 512 x 1024 x 8192 400 -> 443, but 1024 x 1024 x 4096
    // 548 on 128 single CTAs against 511 on 96 (16 pairs x 3 slices)
    const int s7 = ks_split_for(M, N, kb, sms, 1), s8 = ks_split_for(M, N, kb, sms, 2);
    const int64_t tiles8 = ((M + 255) / 256) * ((N + 255) / 256);
    if (s8 && (!s7 || tiles8 * s8 * 2 >= tiles7 * s7)) return GEMM_VARIANT_S8_CTA_PAIR;
    return GEMM_VARIANT_S7_WARP_SPECIALIZED;
  }
  if (kb < 32) {
    const double t9 = std::min(short_k_time(kShort9, M, N, 512, 256, pairs, kb),
                               short_k_time(kShort9, M, N, 512, 224, pairs, kb));
    const double t8 = short_k_time(kShort8, M, N, 256, 256, pairs, kb);
    const double t7 = short_k_time(kShort7, M, N, 128, 256, std::max(1, sms), kb);
    if (t9 <= t8 && t9 <= t7) return GEMM_VARIANT_S9_TWO_CONSUMERS;
    return (t8 <= t7) ? GEMM_VARIANT_S8_CTA_PAIR : GEMM_VARIANT_S7_WARP_SPECIALIZED;
  }
  double c9 = 0;
  s9_tiling(M, N, kb, pairs, true, &c9);
  const double c8 = ws_cost_with_stream_k(GEMM_VARIANT_S8_CTA_PAIR, M, N, 256, 2, pairs, kRate8, kb,
                                          ws_tile_cost(M, N, 256, 256, 2, pairs, kRate8, kb, kFixed8));
  const double c7 = ws_cost_with_stream_k(GEMM_VARIANT_S7_WARP_SPECIALIZED, M, N, 128, 1, std::max(1, sms), kRate7,
                                          kb, ws_tile_cost(M, N, 128, 256, 1, std::max(1, sms), kRate7, kb, kFixed7));
  if (c9 <= c8 && c9 <= c7) return GEMM_VARIANT_S9_TWO_CONSUMERS;
  return (c8 <= c7) ? GEMM_VARIANT_S8_CTA_PAIR : GEMM_VARIANT_S7_WARP_SPECIALIZED;
}

bool is_ws(int v) { return v >= GEMM_VARIANT_S7_WARP_SPECIALIZED && v <= GEMM_VARIANT_S9_TWO_CONSUMERS; }

// The automatic variant for a dtype and operand layout: auto_variant, then the
// restrictions of the inputs.  Block-scaled inputs run on step 7 or 8 (the one
// whose tiles finish soonest, with the block-scaled kernels' rates); 8-bit inputs and MN-major operands have no GEMV or
// ladder kernel, so a shape that would take one takes step 7 or 8 instead; an
// explicit K split (split_k >= 2) runs on step 7.
int choose_variant(int64_t M, int64_t N, int64_t K, gemm_dtype_t dt, int sms, int32_t layout, int32_t split_k) {
  int v = auto_variant(M, N, K, dt, sms);
  const int pairs = std::max(1, sms / 2);
  const int64_t kb = k_blocks(K, dt);
  auto step8_or_7 = [&](double rate8, double rate7) {
    return ws_tile_cost(M, N, 256, 256, 2, pairs, rate8, kb, kFixed8) <=
                   ws_tile_cost(M, N, 128, 256, 1, std::max(1, sms), rate7, kb, kFixed7)
               ? GEMM_VARIANT_S8_CTA_PAIR
               : GEMM_VARIANT_S7_WARP_SPECIALIZED;
  };
  if (is_mx(dt)) {
    // block-scaled rates: 8192^3 3140 / 2678, 1024 x 4096 x 4096 1735 / 1686; step 9
    // (bf16 C only, 512 x 224 tiles) runs at 1935 on 8192^3 and is taken only on request
    v = step8_or_7(1.0, 0.76);
  } else if ((is_f8(dt) || layout != 0) && !is_ws(v)) {
    v = step8_or_7(kRate8, kRate7);
  }
  if (split_k >= 2 && is_ws(v) && !is_mx(dt)) v = GEMM_VARIANT_S7_WARP_SPECIALIZED;
  return v;
}

// Step 9's 224-column tiles with the static schedule: when N (a multiple of 16)
// lies between 13 and 14 sixteen-column units per tile column, give the first
// columns 224 and the rest 208 so that they add up to N exactly, if that lowers
// the widest total any cluster gets (the clusters take tiles t, t + units, ... of
// the raster order).  4096^3: 19 tile columns, 9 of 224 and 10 of 208; every CTA
// pair then runs one of each, 432 columns instead of 448.
void raster_tile_host(int32_t tile, int32_t tiles_m, int32_t tiles_n, int32_t group, int32_t& tm, int32_t& tn) {
  const int32_t per_group = group * tiles_n;
  const int32_t g = tile / per_group;
  const int32_t first_m = g * group;
  const int32_t rows = std::min(group, tiles_m - first_m);
  const int32_t r = tile - g * per_group;
  tm = first_m + r % rows;
  tn = r / rows;
}
void balance_tile_widths(gemm_plan_s* p) {
  p->wide_cols = p->wide_n = p->narrow_n = 0;
  if (p->sched != GEMM_SCHED_STATIC || p->N % 16 != 0 || p->grid_units < 1) return;
  const int64_t T = p->tiles_n, units16 = p->N / 16;
  if (units16 < 13 * T || units16 >= 14 * T) return;
  const int wide_cols = (int)(units16 - 13 * T);  // columns of 224, the others 208
  auto widest = [&](bool two_widths) {
    std::vector<int64_t> load((size_t)p->grid_units, 0);
    const int64_t tiles = (int64_t)p->tiles_m * p->tiles_n;
    for (int64_t t = 0; t < tiles; ++t) {
      int32_t tm, tn;
      raster_tile_host((int32_t)t, p->tiles_m, p->tiles_n, p->raster_group, tm, tn);
      load[(size_t)(t % p->grid_units)] += (two_widths && tn >= wide_cols) ? 208 : 224;
    }
    return *std::max_element(load.begin(), load.end());
  };
  if (widest(true) < widest(false)) {
    p->wide_cols = wide_cols;
    p->wide_n = 224;
    p->narrow_n = 208;
  }
}

// Fix the kernel, its launch shape and its pointer-independent parameters.
gemm_status_t prepare_launch(gemm_plan_s* p) {
  cudaError_t e = cudaSuccess;
  const int v = p->variant;
  if (v == GEMM_VARIANT_GEMV) {
    e = spec_gemv((int)p->M, (int)p->N, (int)p->K, p->in_bf16, p->out_f32, p->num_sms,
                  (p->flags & GEMM_FLAG_STATIC_B) != 0, &p->spec, &p->gemv_pf_rows);
    // always a programmatic dependent: its CTAs are dispatched while the previous
    // kernel drains; B is read before that kernel completes only with the flag
    p->spec.pdl = true;
  } else if (v == GEMM_VARIANT_GEMV_TC) {
    e = spec_gemv_tc((int)p->M, (int)p->N, (int)p->K, p->in_bf16, p->out_f32, p->num_sms, p->split_k, p->stages,
                     &p->spec, &p->tgbase);
    p->tgbase.timeout_ns = p->timeout_ns;
    p->spec.pdl = (p->flags & GEMM_FLAG_STATIC_B) != 0;
  } else {
    KParams& k = p->kbase;
    k.M = (int32_t)p->M;
    k.N = (int32_t)p->N;
    k.K = (int32_t)p->K;
    k.tiles_m = p->tiles_m;
    k.tiles_n = p->tiles_n;
    k.raster_group = p->raster_group;
    k.wide_cols = p->wide_cols;
    k.wide_n = p->wide_n;
    k.narrow_n = p->narrow_n;
    k.stages = p->stages;
    k.timeout_ns = p->timeout_ns;
    k.debug_flags = p->debug_flags;
    k.out_ld = (int32_t)p->ldc;
    k.idesc = is_ws(v) ? idesc_f16(p->in_bf16, 128 * p->cg, p->tile_n) : idesc_f16(p->in_bf16, 128, 128);
    k.mma_kind = 0;
    k.bk = 64;
    if (p->in_mx) {
      k.idesc = idesc_mx(p->in_e5m2, 128 * p->cg, p->tile_n);
      k.mma_kind = 2;
      k.bk = 128;
    } else if (p->in_f8) {
      k.idesc = idesc_f8(p->in_e5m2, 128 * p->cg, p->tile_n);
      k.mma_kind = 1;
      k.bk = 128;
    }
    k.layout = (uint32_t)p->layout;
    if (p->layout & GEMM_LAYOUT_A_MN) k.idesc |= IDESC_A_MN_MAJOR;
    if (p->layout & GEMM_LAYOUT_B_MN) k.idesc |= IDESC_B_MN_MAJOR;
    if (v <= GEMM_VARIANT_S3_MULTI_CTA) {
      e = spec_step123((int)p->M, (int)p->N, p->out_f32, &p->spec);
    } else if (v <= GEMM_VARIANT_S5_PIPELINE) {
      e = spec_step45((int)p->M, (int)p->N, p->stages, p->out_f32, &p->spec);
    } else if (v == GEMM_VARIANT_S6_PERSISTENT) {
      e = spec_step6(p->sched - 1, p->stages, p->out_f32, p->grid_units, &p->spec);
    } else if (p->in_mx) {
      e = spec_mx(p->cg, p->sched - 1, p->out_f32, p->stages, p->grid_units, &p->spec, -1, p->consumers);
    } else if (p->ks_split >= 2) {
      e = spec_ws_ks(p->cg, p->out_f32, p->stages, p->tiles_m * p->tiles_n, p->ks_split, &p->spec);
    } else {
      e = spec_ws(p->cg, p->consumers, p->sched - 1, p->out_f32, p->stages, p->grid_units, &p->spec, -1, p->tile_n);
    }
    // steps 7-9 launch as programmatic dependents: their set-up (barriers, TMEM,
    // cluster) overlaps the end of the previous kernel on the stream, and every
    // thread waits for that kernel to complete before touching global memory
    if (is_ws(v)) p->spec.pdl = true;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

gemm_status_t build_plan(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const gemm_opts_t* opts,
                         gemm_plan_s** out) {
  gemm_status_t st = validate_sizes(M, N, K, dtype);
  if (st != GEMM_OK) return st;
  gemm_opts_t o{};
  if (opts) o = *opts;
  if (o.variant < 0 || o.variant > GEMM_VARIANT_GEMV_TC || o.sched < 0 || o.sched > GEMM_SCHED_STREAM_K ||
      o.stages < 0 || o.stages > 12 || o.raster_group < 0 || o.max_ctas < 0 || o.timeout_ns < 0 ||
      o.split_k < 0 || o.split_k > 8 || (o.flags & ~GEMM_FLAG_STATIC_B) != 0 ||
      (o.layout & ~(GEMM_LAYOUT_A_MN | GEMM_LAYOUT_B_MN)) != 0)
    return GEMM_ERR_INVALID_ARG;

  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != GEMM_OK && !o.variant) return st;
  int variant = o.variant ? o.variant : choose_variant(M, N, K, dtype, sms, o.layout, o.split_k);
  if (is_mx(dtype)) {
    // block-scaled inputs run on step 7's one-CTA tile, step 8's CTA pair (one
    // consumer) or, for bf16 C with the static schedule, step 9's two consumers
    const bool s9_ok = variant == GEMM_VARIANT_S9_TWO_CONSUMERS && out_bytes(dtype) == 2 &&
                       (o.sched == 0 || o.sched == GEMM_SCHED_STATIC);
    if (variant != GEMM_VARIANT_S7_WARP_SPECIALIZED && variant != GEMM_VARIANT_S8_CTA_PAIR && !s9_ok)
      return GEMM_ERR_UNSUPPORTED_SHAPE;
  }
  if (is_f8(dtype)) {
    // 8-bit inputs run on the warp-specialised kernels only, K-major
    if (o.layout != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;
    if (!is_ws(variant)) return GEMM_ERR_UNSUPPORTED_SHAPE;
  }
  if (o.split_k >= 2 && is_ws(variant) && !is_mx(dtype)) {
    // a K split over a cluster exists for step 7's tile, step 8's pair tile (at
    // most 4 slices: 8 CTAs per cluster) and the tensor-core GEMV
    if (variant == GEMM_VARIANT_S8_CTA_PAIR ? o.split_k > 4 : variant != GEMM_VARIANT_S7_WARP_SPECIALIZED)
      return GEMM_ERR_UNSUPPORTED_SHAPE;
  }
  if (o.layout != 0) {
    // MN-major operands exist in the warp-specialised kernels only
    if (!is_ws(variant)) return GEMM_ERR_UNSUPPORTED_SHAPE;
    if (((o.layout & GEMM_LAYOUT_A_MN) && M % 8 != 0) || ((o.layout & GEMM_LAYOUT_B_MN) && N % 8 != 0))
      return GEMM_ERR_UNSUPPORTED_SHAPE;
  }
  // shape limits of the individual steps
  if (variant == GEMM_VARIANT_S1_SINGLE_TILE && (M > 128 || N > 128 || K > 64)) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (variant == GEMM_VARIANT_S2_KLOOP && (M > 128 || N > 128)) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (variant >= GEMM_VARIANT_S7_WARP_SPECIALIZED && variant <= GEMM_VARIANT_S9_TWO_CONSUMERS &&
      !c_rows_tma_ok(N, dtype))
    return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (variant == GEMM_VARIANT_GEMV && (M > 16 || gemv_smem_bytes((int)M, (int)K) > 200 * 1024))
    return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (variant == GEMM_VARIANT_GEMV_TC && M > 16) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (st != GEMM_OK) return st;

  gemm_plan_s* p = new (std::nothrow) gemm_plan_s();
  if (!p) return GEMM_ERR_OOM;
  p->M = M;
  p->N = N;
  p->ldc = N;
  p->K = K;
  p->dtype = dtype;
  p->in_bf16 = (dtype == GEMM_BF16_F32 || dtype == GEMM_BF16_BF16);
  p->in_f8 = is_f8(dtype);
  p->in_e5m2 = is_e5m2(dtype);
  p->in_mx = is_mx(dtype);
  p->out_f32 = (out_bytes(dtype) == 4);
  p->variant = variant;
  p->device = dev;
  p->num_sms = sms;
  p->timeout_ns = o.timeout_ns ? (uint64_t)o.timeout_ns : kDefaultTimeoutNs;
  p->debug_flags = (uint32_t)o.debug_flags;
  p->flags = o.flags;
  p->layout = o.layout;
  p->cg = 1;
  p->consumers = 1;
  p->sched = 0;
  p->stages = 1;
  p->raster_group = 1;
  p->smem = 0;
  p->tile_m = 128;
  p->tile_n = 128;

  const bool persistent = variant >= GEMM_VARIANT_S6_PERSISTENT && variant <= GEMM_VARIANT_S9_TWO_CONSUMERS;
  if (persistent) p->sched = o.sched ? o.sched : GEMM_SCHED_STATIC;
  if (o.sched == GEMM_SCHED_STREAM_K && (!is_ws(variant) || is_mx(dtype))) {
    delete p;
    return GEMM_ERR_UNSUPPORTED_SHAPE;
  }

  if (variant == GEMM_VARIANT_S5_PIPELINE || variant == GEMM_VARIANT_S6_PERSISTENT) {
    p->stages = o.stages ? o.stages : (variant == GEMM_VARIANT_S5_PIPELINE ? 2 : 4);
    if (p->stages > 6) p->stages = 6;
  }
  if (variant >= GEMM_VARIANT_S7_WARP_SPECIALIZED && variant <= GEMM_VARIANT_S9_TWO_CONSUMERS) {
    p->cg = (variant == GEMM_VARIANT_S7_WARP_SPECIALIZED) ? 1 : 2;
    p->consumers = (variant == GEMM_VARIANT_S9_TWO_CONSUMERS) ? 2 : 1;
    const WsShape sh = ws_shape(p->cg, p->consumers);
    const int maxs = ws_max_stages(p->cg, p->consumers);
    p->stages = o.stages ? std::min<int>(o.stages, maxs) : maxs;
    p->tile_m = sh.tile_m;
    p->tile_n = sh.tile_n;
    p->smem = ws_smem_bytes(p->cg, p->consumers, p->stages);
    // Step 9 with whole tiles: switch to 224-column tiles when they fill the waves of
    // resident CTA pairs clearly better (4096^3: 128 tiles of 512 x 256 on 76 pairs use
    // 84 % of two waves; 152 tiles of 512 x 224 use both, 96 % of the columns useful)
    if (variant == GEMM_VARIANT_S9_TWO_CONSUMERS && !p->in_mx && o.layout == 0 &&
        (o.sched == 0 || o.sched == GEMM_SCHED_STATIC)) {
      // (the narrower tile needs a clear margin, 3 %, by ws_tile_cost; where stream-K
      // beats both, the automatic plan keeps 256 columns and takes it below)
      if (s9_tiling(M, N, k_blocks(K, dtype), std::max(1, sms / 2), !o.sched, nullptr) == 1) {
        p->tile_n = 224;
        const int maxs224 = ws_max_stages(p->cg, p->consumers, 224);
        p->stages = o.stages ? std::min<int>(o.stages, maxs224) : maxs224;
        p->smem = ws_smem_bytes(p->cg, p->consumers, p->stages, 224);
        p->sched = GEMM_SCHED_STATIC;
      }
    }
    if (p->in_mx) {
      if (p->consumers == 2) {
        p->tile_n = 224;  // 448 TMEM columns of accumulators leave 64 for the scale slots
        p->sched = GEMM_SCHED_STATIC;
      }
      const int maxs = mx_max_stages(p->cg, p->consumers);
      p->stages = o.stages ? std::min<int>(o.stages, maxs) : maxs;
      p->smem = mx_smem_bytes(p->cg, p->stages, p->consumers);
    }
  } else if (variant == GEMM_VARIANT_S6_PERSISTENT) {
    p->smem = step6_smem_bytes(p->stages);
  }
  if (variant == GEMM_VARIANT_GEMV_TC) {
    int split = 1, kpc = 1;
    gemv_tc_config((int)N, (int)K, sms, o.split_k, o.stages, &split, &p->stages, &kpc);
    p->cg = split;
    p->split_k = o.split_k;
    p->smem = gemv_tc_smem_bytes(p->stages);
    p->tile_m = 16;
    p->tile_n = 128;
  }
  p->tiles_m = ceil_div(M, p->tile_m);
  p->tiles_n = ceil_div(N, p->tile_n);
  if (persistent) p->raster_group = o.raster_group ? o.raster_group : std::min(8, p->tiles_m);
  if (p->raster_group > p->tiles_m) p->raster_group = p->tiles_m;
  if (p->raster_group < 1) p->raster_group = 1;

  const int tiles = p->tiles_m * p->tiles_n;
  if (variant == GEMM_VARIANT_S6_PERSISTENT) {
    int units = (p->sched == GEMM_SCHED_CLC) ? tiles : std::min(tiles, sms);
    if (o.max_ctas && p->sched != GEMM_SCHED_CLC) units = std::min(units, (int)o.max_ctas);
    p->grid_units = units;
  } else if (variant >= GEMM_VARIANT_S7_WARP_SPECIALIZED && variant <= GEMM_VARIANT_S9_TWO_CONSUMERS) {
    // (the MX kernels' shared memory also allows one CTA per SM)
    int active = p->in_mx ? sms / p->cg
                          : ws_max_active_clusters(p->cg, p->consumers, p->sched - 1, p->out_f32, p->stages,
                                                   p->tile_n);
    if (active < 1) active = std::max(1, sms / p->cg);
    int units = (p->sched == GEMM_SCHED_CLC) ? tiles : std::min(tiles, active);
    if (o.max_ctas && p->sched != GEMM_SCHED_CLC) units = std::max(1, std::min(units, (int)o.max_ctas));
    p->grid_units = units;
    // stream-K by default where ws_stream_k_time takes it: whole tiles would leave
    // the clusters idle for over 20 % of the waves (30 % on step 9) and the split
    // tiles' partial sums cost less than that.  Measured on GB300: 80 tiles on 76 CTA
    // pairs (4096 x 2560 x 8192, step 9) 1115 -> 1507 TFLOP/s; at 84 % (4096^3) the
    // partial sums cost more than the idle clusters (1494 -> 1242).  Only when every
    // cluster gets at least a tile's work: with fewer tiles than clusters the shares
    // shrink below half a tile and the partial sums cost more than the extra SMs
    // bring (1024 x 1024 x 4096 on 152 SMs: 319 TFLOP/s with 32 whole tiles, 191
    // split over all SMs).  An explicit GEMM_SCHED_STREAM_K still spreads such shapes
    // over every resident cluster.
    if (!o.sched && !p->in_mx && p->tile_n == 256 &&
        ws_stream_k_time(variant, tiles, active, k_blocks(K, dtype)) >= 0)
      p->sched = GEMM_SCHED_STREAM_K;
    // Steps 7 and 8 with few tiles for the GPU: split each tile's K over a cluster
    // of CTAs (opts.split_k = 2-8 asks for it, 2-4 on step 8's pairs, 1 forbids it).
    // Automatic (ks_split_for): as many slices as the SMs hold at once, at most 4,
    // while each keeps at least 16 K blocks; with shorter shares the partial sums
    // cost more than the extra SMs bring (1024 x 1024 x 4096 on step 7: 320 TFLOP/s
    // whole, 416 split 2, 491 split 4).  Clusters of 8 single CTAs do not all fit at
    // once (512 x 1024 x 8192 on 16 tiles: 416 split 4, 250 split 8).
    if ((variant == GEMM_VARIANT_S7_WARP_SPECIALIZED || variant == GEMM_VARIANT_S8_CTA_PAIR) && !p->in_mx &&
        o.layout == 0 && (o.sched == 0 || o.sched == GEMM_SCHED_STATIC) && p->sched != GEMM_SCHED_STREAM_K &&
        o.split_k != 1) {
      const int64_t kb = (K + (p->in_f8 ? 128 : 64) - 1) / (p->in_f8 ? 128 : 64);
      int64_t split = o.split_k;
      if (!split && tiles > 0) split = ks_split_for(M, N, kb, sms, p->cg);
      if (split >= 2 && split <= kb && split * p->cg <= 8) {
        p->ks_split = (int)split;
        p->sched = GEMM_SCHED_STATIC;
        // two slices exchange their 128 KB partials through their stage rings
        if (split == 2)
          while ((size_t)p->stages * ws_shape(p->cg, 1).stage_bytes < (size_t)128 * 1024) ++p->stages;
        p->smem = ws_smem_bytes(p->cg, 1, p->stages);
        p->grid_units = tiles * (int)split * p->cg;  // CTAs
      }
    }
    if (p->sched == GEMM_SCHED_STREAM_K && !o.max_ctas) {
      const int64_t kb = (K + (p->in_f8 ? 128 : 64) - 1) / (p->in_f8 ? 128 : 64);
      p->grid_units = (int)std::max<int64_t>(1, std::min<int64_t>(active, (int64_t)tiles * kb / 4));
    }
    if (p->tile_n == 224 && !p->in_mx) balance_tile_widths(p);
  } else {
    p->grid_units = tiles;
  }

  st = prepare_launch(p);
  if (st != GEMM_OK) {
    delete p;
    return st;
  }
  if (cudaMalloc(reinterpret_cast<void**>(&p->scratch), 256) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return GEMM_ERR_OOM;
  }
  if (cudaMemset(p->scratch, 0, 256) != cudaSuccess) {
    cudaFree(p->scratch);
    delete p;
    return GEMM_ERR_CUDA;
  }
  p->kbase.status = p->scratch;
  p->tgbase.status = p->scratch;
  if (p->sched == GEMM_SCHED_STREAM_K) {
    const size_t slot = ws_sk_slot_floats(p->cg, p->consumers);
    p->sk_flag_bytes = (size_t)p->grid_units * p->cg * p->consumers * 4 * sizeof(uint32_t);
    if (cudaMalloc(reinterpret_cast<void**>(&p->sk_ws), (size_t)p->grid_units * slot * sizeof(float)) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&p->sk_flags), p->sk_flag_bytes) != cudaSuccess) {
      cudaGetLastError();
      gemm_plan_destroy(p);
      return GEMM_ERR_OOM;
    }
    if (cudaMemset(p->sk_flags, 0, p->sk_flag_bytes) != cudaSuccess) {
      gemm_plan_destroy(p);
      return GEMM_ERR_CUDA;
    }
    p->kbase.sk_ws = p->sk_ws;
    p->kbase.sk_flags = p->sk_flags;
  }
  if (p->ks_split > 2) {
    // split-K over a cluster of more than two: one fp32 partial slot (32 rows x
    // 256 columns per writeback warp, 128 KB) per CTA; an automatic split launches
    // at most one CTA per SM (19 MB on 152 SMs), and a forced split that would
    // need more than 512 MB is refused
    const size_t bytes = (size_t)p->grid_units * ws_sk_slot_floats(1, 1) * sizeof(float);
    if (bytes > ((size_t)512 << 20)) {
      gemm_plan_destroy(p);
      return GEMM_ERR_UNSUPPORTED_SHAPE;
    }
    if (cudaMalloc(reinterpret_cast<void**>(&p->sk_ws), bytes) != cudaSuccess) {
      cudaGetLastError();
      gemm_plan_destroy(p);
      return GEMM_ERR_OOM;
    }
    p->kbase.sk_ws = p->sk_ws;
  }
  *out = p;
  return GEMM_OK;
}

// The TMA descriptor of one operand, from the plan's cache or freshly encoded.
const CUtensorMap* operand_map(gemm_plan_s* p, int role, const void* ptr) {
  gemm_plan_s::MapEntry* victim = &p->maps[0];
  for (auto& m : p->maps) {
    if (m.ptr == ptr && m.role == role && m.used != 0) {
      m.used = ++p->map_clock;
      return &m.map;
    }
    if (m.used < victim->used) victim = &m;
  }
  const CUtensorMapDataType in_t = p->in_f8    ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : p->in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int ie = p->in_f8 ? 1 : 2;     // bytes per input element
  const uint32_t kbox = 128u / ie;     // one 128-byte swizzle row of K
  bool ok = false;
  if (role == 4) {
    // MX scales of A: the tiled array seen as rows of 128 bytes, one 512-byte
    // block = a box of 4 rows, copied as is
    const int64_t bytes = gemm_mx_scale_bytes(p->M, p->K);
    ok = bytes > 0 && encode_2d(&victim->map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ptr, 128, (uint64_t)(bytes / 128), 128,
                                4, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else if (role == 5 || role == 7) {
    // MX scales of B: the two 128-row blocks of a 256-row tile in one box; role 7
    // (step 9's 224-row tiles): the three blocks that hold a tile's rows
    ok = encode_mx_pairs(&victim->map, ptr, (uint64_t)((p->K + 127) / 128), (uint64_t)((p->N + 127) / 128),
                         role == 7 ? 3u : 2u);
  } else if (role == 3) {
    // activation rows of the tensor-core GEMV: 16-row boxes, rows >= M read as zero
    ok = encode_2d(&victim->map, in_t, 2, ptr, (uint64_t)p->K, (uint64_t)p->M, 64, 16);
  } else if (role == 0 && (p->layout & GEMM_LAYOUT_A_MN)) {
    // A stored K x M: 64-wide boxes along M, 64 rows of K
    ok = encode_2d(&victim->map, in_t, 2, ptr, (uint64_t)p->M, (uint64_t)p->K, 64, 64);
  } else if (role == 1 && (p->layout & GEMM_LAYOUT_B_MN)) {
    ok = encode_2d(&victim->map, in_t, 2, ptr, (uint64_t)p->N, (uint64_t)p->K, 64, 64);
  } else if (role == 0) {
    ok = encode_2d(&victim->map, in_t, ie, ptr, (uint64_t)p->K, (uint64_t)p->M, kbox, 128);
  } else if (role == 1 || role == 6) {
    // role 6: B for the fused-epilogue kernels (256-column tiles)
    const uint32_t rows = !is_ws(p->variant) ? 128u
                          : role == 6        ? (uint32_t)ws_shape(p->cg, 1).b_box_rows
                                             : (uint32_t)ws_shape(p->cg, p->consumers, p->tile_n).b_box_rows;
    ok = encode_2d(&victim->map, in_t, ie, ptr, (uint64_t)p->K, (uint64_t)p->N, kbox, rows);
  } else {
    ok = p->out_f32 ? encode_2d(&victim->map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, (uint64_t)p->N,
                                (uint64_t)p->M, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B, (uint64_t)p->ldc)
                    : encode_2d(&victim->map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, (uint64_t)p->N,
                                (uint64_t)p->M, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B, (uint64_t)p->ldc);
  }
  if (!ok) {
    victim->used = 0;
    return nullptr;
  }
  victim->ptr = ptr;
  victim->role = role;
  victim->used = ++p->map_clock;
  return &victim->map;
}

gemm_status_t launch_plan(gemm_plan_s* p, const void* A, const void* B, void* C, cudaStream_t s,
                          const gemm_epilogue_t* epi = nullptr, const void* sfa = nullptr,
                          const void* sfb = nullptr) {
  if (!A || !B || !C) return GEMM_ERR_INVALID_ARG;
  // block-scaled plans run with their scale arrays, other plans without
  if (p->in_mx != (sfa != nullptr) || p->in_mx != (sfb != nullptr)) return GEMM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_MISALIGNED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != p->device) return GEMM_ERR_INVALID_ARG;
  cudaError_t e = cudaSuccess;
  switch (p->spec.kind) {
    case ARGS_GEMV: {
      GemvParams g{A, B, C, (int32_t)p->M, (int32_t)p->N, (int32_t)p->K,
                   (p->flags & GEMM_FLAG_STATIC_B) ? 1 : 0, p->gemv_pf_rows};
      void* args[] = {&g};
      e = launch_spec(p->spec, args, s);
      break;
    }
    case ARGS_BX_TG: {
      const CUtensorMap* mb = operand_map(p, 1, B);
      const CUtensorMap* mx = operand_map(p, 3, A);
      if (!mb || !mx) return GEMM_ERR_CUDA;
      TgParams t = p->tgbase;
      t.X = static_cast<const uint16_t*>(A);
      t.Y = C;
      void* args[] = {const_cast<CUtensorMap*>(mb), const_cast<CUtensorMap*>(mx), &t};
      e = launch_spec(p->spec, args, s);
      break;
    }
    default: {
      KParams k = p->kbase;
      k.visits = p->visits;
      const LaunchSpec* spec = &p->spec;
      if (epi != nullptr) {
        k.bias = epi->bias;
        k.residual = epi->residual;
        k.act = epi->activation;
        k.scale_a = epi->scale_a;
        k.scale_b = epi->scale_b;
        k.tiles_m = p->epi_tiles_m[epi->activation];
        k.tiles_n = p->epi_tiles_n[epi->activation];
        k.stages = p->epi_stages[epi->activation];
        // the fused kernels' MMAs are 256 columns wide whatever the plan's own tile
        k.idesc = idesc_with_n(k.idesc, 256);
        spec = &p->spec_epi[epi->activation];
      }
      k.A = static_cast<const uint16_t*>(A);
      k.B = static_cast<const uint16_t*>(B);
      k.C = C;
      if (p->spec.kind == ARGS_K) {
        void* args[] = {&k};
        e = launch_spec(p->spec, args, s);
        break;
      }
      const CUtensorMap* ma = operand_map(p, 0, A);
      // (the fused kernels read B in 256-column tiles even where the plan's own are narrower)
      const CUtensorMap* mb = operand_map(p, (epi != nullptr && p->tile_n != 256) ? 6 : 1, B);
      if (!ma || !mb) return GEMM_ERR_CUDA;
      if (spec->kind == ARGS_AB_K) {
        void* args[] = {const_cast<CUtensorMap*>(ma), const_cast<CUtensorMap*>(mb), &k};
        e = launch_spec(*spec, args, s);
      } else if (spec->kind == ARGS_ABCSS_K) {
        const CUtensorMap* mc = operand_map(p, 2, C);
        const CUtensorMap* msa = operand_map(p, 4, sfa);
        const CUtensorMap* msb = operand_map(p, (epi == nullptr && p->in_mx && p->consumers == 2) ? 7 : 5, sfb);
        if (!mc || !msa || !msb) return GEMM_ERR_CUDA;
        void* args[] = {const_cast<CUtensorMap*>(ma), const_cast<CUtensorMap*>(mb), const_cast<CUtensorMap*>(mc),
                        const_cast<CUtensorMap*>(msa), const_cast<CUtensorMap*>(msb), &k};
        e = launch_spec(*spec, args, s);
      } else {
        const CUtensorMap* mc = operand_map(p, 2, C);
        if (!mc) return GEMM_ERR_CUDA;
        void* args[] = {const_cast<CUtensorMap*>(ma), const_cast<CUtensorMap*>(mb), const_cast<CUtensorMap*>(mc), &k};
        e = launch_spec(*spec, args, s);
      }
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

// Validate the fused epilogue, make its kernel's launch shape on first use,
// and launch.
gemm_status_t run_with_epilogue(gemm_plan_s* plan, const void* A, const void* B, void* C,
                                const gemm_epilogue_t* epi, cudaStream_t s, const void* sfa, const void* sfb) {
  if (!is_ws(plan->variant)) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (epi->activation < GEMM_ACT_NONE || epi->activation > GEMM_ACT_GELU_ERF) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(epi->bias) & 3u) || (reinterpret_cast<uintptr_t>(epi->residual) & 15u) ||
      (reinterpret_cast<uintptr_t>(epi->scale_a) & 3u) || (reinterpret_cast<uintptr_t>(epi->scale_b) & 3u))
    return GEMM_ERR_MISALIGNED;
  const int act = epi->activation;
  if (!plan->epi_ready[act]) {
    cudaError_t e;
    if (plan->in_mx && plan->consumers == 1) {
      // the block-scaled plan already runs one consumer on one CTA
      plan->epi_stages[act] = plan->stages;
      plan->epi_tiles_m[act] = plan->tiles_m;
      plan->epi_tiles_n[act] = plan->tiles_n;
      e = spec_mx(plan->cg, 0, plan->out_f32, plan->stages, std::min(plan->grid_units, plan->tiles_m * plan->tiles_n),
                  &plan->spec_epi[act], act);
    } else if (plan->in_mx) {
      // step 9's block-scaled kernel has no fused epilogue: step 8's (256 x 256 tiles)
      plan->epi_stages[act] = mx_max_stages(2, 1);
      plan->epi_tiles_m[act] = ceil_div(plan->M, 256);
      plan->epi_tiles_n[act] = ceil_div(plan->N, 256);
      e = spec_mx(2, 0, plan->out_f32, plan->epi_stages[act],
                  std::min(plan->grid_units, plan->epi_tiles_m[act] * plan->epi_tiles_n[act]), &plan->spec_epi[act],
                  act);
    } else {
      // The epilogue runs in the writeback warps while the MMAs of the next tile
      // proceed.  Steps 7 and 8 have a TMEM double buffer for that; step 9's two
      // consumers have one accumulator each, held while the writeback applies the
      // epilogue.  For bf16 C the residual is read before the accumulator is
      // ready and the staging and stores follow the hand-back, so step 9 keeps
      // its tile; for fp32 C (no such drain) an activation runs on step 8's 256 x
      // 256 tile (same operand boxes) and bias / residual / scales on step 9's.
      const int cons =
          (plan->cg == 2 && plan->consumers == 2 && (act == GEMM_ACT_NONE || !plan->out_f32)) ? 2 : 1;
      plan->epi_stages[act] = ws_max_stages(plan->cg, cons);
      plan->epi_tiles_m[act] = ceil_div(plan->M, 128 * plan->cg * cons);
      plan->epi_tiles_n[act] = ceil_div(plan->N, 256);  // the fused kernels use 256-column tiles
      const int tiles = plan->epi_tiles_m[act] * plan->epi_tiles_n[act];
      int active = ws_max_active_clusters(plan->cg, cons, 0, plan->out_f32, plan->epi_stages[act]);
      if (active < 1) active = std::max(1, plan->num_sms / plan->cg);
      e = spec_ws(plan->cg, cons, 0, plan->out_f32, plan->epi_stages[act], std::min(tiles, active),
                  &plan->spec_epi[act], act);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    plan->spec_epi[act].pdl = true;
    plan->epi_ready[act] = true;
  }
  return launch_plan(plan, A, B, C, s, epi, sfa, sfb);
}

gemm_status_t check_plan(gemm_plan_s* p) {
  uint32_t word = 0;
  if (cudaMemcpy(&word, p->scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (word != 0) {
    // rewind the status word, the scheduler counters and any stream-K flags left
    // set by an aborted launch
    cudaMemset(p->scratch, 0, 256);
    if (p->sk_flags) cudaMemset(p->sk_flags, 0, p->sk_flag_bytes);
    return GEMM_ERR_DEVICE_TIMEOUT;
  }
  return GEMM_OK;
}

// Copy-compute pipeline of gemm_run_host, one per device: two copy streams (one
// per direction, which run concurrently), a compute stream and their events,
// created on first use and kept; one gemm_run_host call uses them at a time.
// (8192^3 bf16 end to end: 1 panel 2.57 ms, 2 panels 1.99, 4 panels 1.74, 8 panels 1.68)
constexpr int kPipePanels = 8;
struct HostPipe {
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t b_in[2] = {}, a_in[kPipePanels] = {}, c_done[kPipePanels][2] = {};
};
std::mutex g_pipe_mu;
std::map<int, HostPipe> g_pipes;

gemm_status_t host_pipe(int dev, HostPipe** out) {
  auto it = g_pipes.find(dev);
  if (it != g_pipes.end()) {
    *out = &it->second;
    return GEMM_OK;
  }
  HostPipe h;
  bool ok = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h.comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.b_in[0], cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&h.b_in[1], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kPipePanels; ++i)
    ok = cudaEventCreateWithFlags(&h.a_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&h.c_done[i][0], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&h.c_done[i][1], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  *out = &(g_pipes[dev] = h);
  return GEMM_OK;
}

// plans made by gemm_run, keyed by shape, dtype and device
std::mutex g_cache_mu;
std::map<std::tuple<int64_t, int64_t, int64_t, int64_t, int, int>, gemm_plan_s*> g_cache;

// gemm_run's body, for a C whose rows are `ldc` elements apart (ldc = N, or a
// block of a wider C for the host pipeline; the GEMV variants need ldc = N)
gemm_status_t run_cached(int64_t M, int64_t N, int64_t K, int64_t ldc, const void* A, const void* B, void* C,
                         gemm_dtype_t dtype, cudaStream_t stream) {
  gemm_status_t st = validate_sizes(M, N, K, dtype);
  if (st != GEMM_OK) return st;
  if (is_mx(dtype)) return GEMM_ERR_INVALID_ARG;  // needs scales: gemm_plan_run_mx
  if (!A || !B || !C) return GEMM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_MISALIGNED;
  if (ldc < N || (ldc * out_bytes(dtype)) % 16 != 0) return GEMM_ERR_INVALID_ARG;
  int dev = 0;
  {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) {
      cudaGetLastError();
      return GEMM_ERR_NO_DEVICE;
    }
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  }
  gemm_plan_s* p = nullptr;
  try {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto key = std::make_tuple(M, N, K, ldc, (int)dtype, dev);
    auto it = g_cache.find(key);
    if (it != g_cache.end()) {
      p = it->second;
    } else {
      st = build_plan(M, N, K, dtype, nullptr, &p);
      if (st != GEMM_OK) return st;
      if (ldc != N) {
        if (p->variant == GEMM_VARIANT_GEMV || p->variant == GEMM_VARIANT_GEMV_TC) {
          gemm_plan_destroy(p);
          return GEMM_ERR_UNSUPPORTED_SHAPE;
        }
        p->ldc = ldc;
        p->kbase.out_ld = (int32_t)ldc;
      }
      g_cache[key] = p;
    }
  } catch (...) {
    return GEMM_ERR_OOM;
  }
  return launch_plan(p, A, B, C, stream);
}

}  // namespace

extern "C" {

gemm_status_t gemm_auto_variant(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int32_t num_sms,
                                int32_t* variant) {
  if (!variant) return GEMM_ERR_INVALID_ARG;
  *variant = 0;
  const gemm_status_t st = validate_sizes(M, N, K, dtype);
  if (st != GEMM_OK) return st;
  if (num_sms < 2) return GEMM_ERR_INVALID_ARG;
  *variant = choose_variant(M, N, K, dtype, num_sms, 0, 0);
  return GEMM_OK;
}

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const gemm_opts_t* opts,
                        gemm_plan_t* out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  try {
    return build_plan(M, N, K, dtype, opts, out);
  } catch (...) {
    return GEMM_ERR_OOM;
  }
}

gemm_status_t gemm_plan_run(gemm_plan_t plan, const void* A, const void* B, void* C, gemm_stream_t stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  return launch_plan(plan, A, B, C, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_plan_run_epilogue(gemm_plan_t plan, const void* A, const void* B, void* C,
                                     const gemm_epilogue_t* epi, gemm_stream_t stream) {
  if (!plan || !epi) return GEMM_ERR_INVALID_ARG;
  if (plan->in_mx) return GEMM_ERR_INVALID_ARG;  // needs its scales: gemm_plan_run_mx
  return run_with_epilogue(plan, A, B, C, epi, reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr);
}

gemm_status_t gemm_plan_run_mx(gemm_plan_t plan, const void* A, const void* B, void* C, const void* scale_a,
                               const void* scale_b, const gemm_epilogue_t* epi, gemm_stream_t stream) {
  if (!plan) return GEMM_ERR_INVALID_ARG;
  if (!plan->in_mx) return GEMM_ERR_UNSUPPORTED_DTYPE;
  if (!scale_a || !scale_b) return GEMM_ERR_INVALID_ARG;
  if (!aligned16(scale_a) || !aligned16(scale_b)) return GEMM_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (epi == nullptr) return launch_plan(plan, A, B, C, s, nullptr, scale_a, scale_b);
  return run_with_epilogue(plan, A, B, C, epi, s, scale_a, scale_b);
}

int64_t gemm_mx_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 1 || K < 1 || rows >= kMaxDim || K >= kMaxDim) return -1;
  return ((rows + 127) / 128) * ((K + 127) / 128) * 512;
}

gemm_status_t gemm_run(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                       gemm_dtype_t dtype, gemm_stream_t stream) {
  return run_cached(M, N, K, N, A, B, C, dtype, reinterpret_cast<cudaStream_t>(stream));
}

// Host operands, pipelined: the host-to-device stream carries the first half of
// B's rows (the first half of C's columns), the first row panel of A, the second
// half of B, then the remaining panels of A; each block of C (a row panel by a
// column half) is computed as soon as its operands have landed and returns on
// the device-to-host stream (strided copy) while later panels are copied and
// computed.  Copies in the two directions run concurrently.
gemm_status_t gemm_run_host(int64_t M, int64_t N, int64_t K, const void* A_host, const void* B_host,
                            void* C_host, gemm_dtype_t dtype, void* dA, void* dB, void* dC,
                            gemm_stream_t stream) {
  gemm_status_t st = validate_sizes(M, N, K, dtype);
  if (st != GEMM_OK) return st;
  if (is_mx(dtype)) return GEMM_ERR_INVALID_ARG;  // needs scales: gemm_plan_run_mx
  if (!A_host || !B_host || !C_host || !dA || !dB || !dC) return GEMM_ERR_INVALID_ARG;
  if (!aligned16(dA) || !aligned16(dB) || !aligned16(dC)) return GEMM_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  const int64_t ib = in_bytes(dtype), ob = out_bytes(dtype);
  // row panels: kPipePanels for problems whose operands take long enough to copy,
  // 2 for mid sizes, 1 otherwise; panel starts stay 16-byte aligned and on 128-row
  // bounds.  With more than one panel and a C at least as large as A and B
  // together, B (and C's columns) also split in two halves at a multiple of 256
  // columns.
  int64_t panels = 1;
  const int64_t in_bytes_total = (M * K + N * K) * ib;
  if ((N * ob) % 16 == 0) {
    if (M >= 128 * kPipePanels && in_bytes_total >= (int64_t)64 << 20) panels = kPipePanels;
    else if (M >= 1024 && in_bytes_total >= (int64_t)16 << 20) panels = 2;
  }
  const int64_t rows = ((M + panels - 1) / panels + 127) / 128 * 128;
  panels = (M + rows - 1) / rows;
  // (the split only pays when returning C takes at least as long as sending A and
  // B: 8192 x 14336 x 4096 bf16 482 -> 495 TFLOP/s, while 8192^3 drops 656 -> 635
  // because its half-width GEMMs then bound the pipeline)
  const bool split_b = panels > 1 && N >= 1024 && M * N * ob >= in_bytes_total;
  const int64_t split = split_b ? ((N / 2 + 255) / 256) * 256 : N;
  const int halves = split < N ? 2 : 1;
  const int64_t c0[2] = {0, split}, nc[2] = {split, N - split};

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* hp = nullptr;
  st = host_pipe(dev, &hp);
  if (st != GEMM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool ok = cudaEventRecord(hp->start, s) == cudaSuccess && cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp->comp, hp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp->d2h, hp->start, 0) == cudaSuccess;
  auto copy_b = [&](int j) {
    return cudaMemcpyAsync(static_cast<char*>(dB) + c0[j] * K * ib, static_cast<const char*>(B_host) + c0[j] * K * ib,
                           (size_t)(nc[j] * K * ib), cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess &&
           cudaEventRecord(hp->b_in[j], hp->h2d) == cudaSuccess;
  };
  auto copy_a = [&](int64_t i) {
    const int64_t r0 = i * rows, mi = std::min(rows, M - r0);
    return cudaMemcpyAsync(static_cast<char*>(dA) + r0 * K * ib, static_cast<const char*>(A_host) + r0 * K * ib,
                           (size_t)(mi * K * ib), cudaMemcpyHostToDevice, hp->h2d) == cudaSuccess &&
           cudaEventRecord(hp->a_in[i], hp->h2d) == cudaSuccess;
  };
  // copy order: B half 0, A panel 0, B half 1, A panels 1..
  ok = ok && copy_b(0) && copy_a(0) && (halves == 1 || copy_b(1));
  for (int64_t i = 1; ok && i < panels; ++i) ok = copy_a(i);
  for (int64_t i = 0; ok && i < panels && st == GEMM_OK; ++i) {
    const int64_t r0 = i * rows, mi = std::min(rows, M - r0);
    ok = cudaStreamWaitEvent(hp->comp, hp->a_in[i], 0) == cudaSuccess;
    for (int j = 0; ok && j < halves; ++j) {
      char* cd = static_cast<char*>(dC) + (r0 * N + c0[j]) * ob;
      ok = cudaStreamWaitEvent(hp->comp, hp->b_in[j], 0) == cudaSuccess;
      if (!ok) break;
      st = run_cached(mi, nc[j], K, N, static_cast<char*>(dA) + r0 * K * ib, static_cast<char*>(dB) + c0[j] * K * ib,
                      cd, dtype, hp->comp);
      if (st != GEMM_OK) break;
      ok = cudaEventRecord(hp->c_done[i][j], hp->comp) == cudaSuccess &&
           cudaStreamWaitEvent(hp->d2h, hp->c_done[i][j], 0) == cudaSuccess &&
           cudaMemcpy2DAsync(static_cast<char*>(C_host) + (r0 * N + c0[j]) * ob, (size_t)(N * ob), cd,
                             (size_t)(N * ob), (size_t)(nc[j] * ob), (size_t)mi, cudaMemcpyDeviceToHost,
                             hp->d2h) == cudaSuccess;
    }
  }
  // drain all three streams whatever happened, then report
  const bool synced = cudaStreamSynchronize(hp->h2d) == cudaSuccess && cudaStreamSynchronize(hp->comp) == cudaSuccess &&
                      cudaStreamSynchronize(hp->d2h) == cudaSuccess;
  if (st != GEMM_OK) return st;
  if (!ok || !synced) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return gemm_check(nullptr, stream);
}

gemm_status_t gemm_check(gemm_plan_t plan, gemm_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (plan) return check_plan(plan);
  std::lock_guard<std::mutex> lock(g_cache_mu);
  gemm_status_t worst = GEMM_OK;
  for (auto& kv : g_cache) {
    gemm_status_t st = check_plan(kv.second);
    if (st != GEMM_OK) worst = st;
  }
  return worst;
}

gemm_status_t gemm_plan_info(gemm_plan_t p, gemm_plan_info_t* info) {
  if (!p || !info) return GEMM_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->variant = p->variant;
  info->sched = p->sched;
  info->stages = p->stages;
  info->raster_group = p->raster_group;
  info->tile_m = p->tile_m;
  info->tile_n = p->tile_n;
  info->cluster = (p->variant == GEMM_VARIANT_GEMV) ? (int32_t)p->spec.cluster
                  : (p->ks_split >= 2)                ? p->ks_split * p->cg
                                                      : p->cg;
  info->consumers = p->consumers;
  info->grid = (int32_t)(p->spec.grid.x * p->spec.grid.y);
  info->smem_bytes = (int32_t)p->spec.smem;
  info->num_sms = p->num_sms;
  info->tiles = p->tiles_m * p->tiles_n;
  info->narrow_tile_n = p->narrow_n;
  info->wide_cols = p->wide_cols;
  return GEMM_OK;
}

gemm_status_t gemm_plan_set_visits(gemm_plan_t p, int32_t* visits) {
  if (!p) return GEMM_ERR_INVALID_ARG;
  p->visits = visits;
  return GEMM_OK;
}

void gemm_plan_destroy(gemm_plan_t p) {
  if (!p) return;
  if (p->scratch) cudaFree(p->scratch);
  if (p->sk_ws) cudaFree(p->sk_ws);
  if (p->sk_flags) cudaFree(p->sk_flags);
  delete p;
}

void gemm_clear_cache(void) {
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (auto& kv : g_cache) gemm_plan_destroy(kv.second);
  g_cache.clear();
}

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case GEMM_ERR_MISALIGNED: return "operand not 16-byte aligned";
    case GEMM_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case GEMM_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_CUDA: return "CUDA call failed";
    case GEMM_ERR_OOM: return "out of memory";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case GEMM_ERR_NO_DEVICE: return "no CUDA device";
  }
  return "unknown status";
}

const char* gemm_version(void) { return "dgb-gemm 0.1 (sm_103a)"; }

}  // extern "C"
