// kernel_gemv.cu -- the decode-shaped product Y (M x N) = X (M x K) * B^T for
// M <= 16 on CUDA cores.
//
// The reading notes of "Modern GPU Programming for MLSys" (section
// "Roofline：找到天花板") use the decode-stage 1 x 4096 x 4096 vector-matrix
// product as the bandwidth-bound example: about one FLOP per byte, far below
// the ridge point, so the Tensor Core is irrelevant and the kernel's only job
// is to stream the weight B from HBM once at full bandwidth.  Every weight
// byte is read once with 16-byte non-allocating loads by every lane straight
// into registers; X (at most 16 rows) is staged in shared memory; fp32 FMAs
// per lane, a shuffle reduction per output, one bf16/fp32 store; the grid
// covers the rows exactly once (no atomics, no scratch memory).
//
// The kernels launch as programmatic dependents of the previous kernel on the
// stream, and two cases differ in what they may do before that kernel has
// completed:
//   * B may be written by the previous kernel (the default).  Nothing of B may
//     be read before griddepcontrol.wait, so the kernel asks L2 to prefetch
//     the first 2 KB of each warp's rows while it waits (a prefetch returns no
//     data, and L2 is coherent for every SM, so a later load still sees what
//     the previous kernel wrote).  After the wait each lane keeps two groups
//     of four 16-byte loads in flight and refills a group as soon as it has
//     been consumed (k_gemv_roll, k_gemv_mma_roll), so the weight stream
//     does not stall between the halves of a row.  In a chain of dependent
//     1 x 4096 x 4096 launches this took a launch from 7.45 us (whole half
//     rows in flight, refilled after each half) to 6.5 us.
//   * B is declared static (GEMM_FLAG_STATIC_B): the first half row of every
//     warp (k_gemv, k_gemv_mma) or the first two groups of every lane (the
//     16-row cluster form of k_gemv_mma_roll) are loaded into registers before
//     the wait, so the weights stream while the previous kernel drains.
//
// For 3 <= M <= 8 the CUDA cores would need M FMAs per weight element, more
// than they can issue at HBM speed, and the tcgen05 GEMV is fed by TMA, which
// streams at most about 40 GB/s per SM from DRAM.  k_gemv_mma keeps the load
// path (16-byte loads by every lane straight into registers) and does the
// arithmetic with warp-level mma.sync m16n8k16: 8 weight rows as the A operand
// (rows 8-15 of the fragment are zero), the M <= 8 activation rows as the n8 B
// operand, fp32 accumulation.  Each lane's 16-byte weight chunk and the
// matching 16-byte activation chunk feed two MMAs; the order of K inside the
// fragments is free because A and B use the same order.  A CTA owns 8 weight
// rows; its 8 warps split K and add their 8 x 8 partial sums in shared memory.
// When the grid fits one wave, a cluster of two CTAs owns 16 rows instead (the
// fragment's rows 8-15 filled, each activation chunk feeding both rows) and
// splits K between its CTAs.
#include <algorithm>
#include <type_traits>

#include "kernel_common.cuh"
#include "launch.h"

namespace dgb {

namespace {

constexpr int GV_THREADS = 256;
constexpr int GV_U = 8;  // 16-byte chunks per lane per row in flight

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// programmatic dependent launch: let the next kernel in the stream start
// launching, and wait for the previous one's results (both no-ops when the
// launch did not ask for it)
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename InT>
__device__ __forceinline__ float2 to_f2(uint32_t w) {
  if constexpr (std::is_same<InT, __nv_bfloat16>::value) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

template <typename InT>
__device__ __forceinline__ float dot8(const uint4& x, const uint4& b, float acc) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
  const uint32_t bs[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 xf = to_f2<InT>(xs[i]);
    const float2 bf = to_f2<InT>(bs[i]);
    acc = fmaf(xf.x, bf.x, acc);
    acc = fmaf(xf.y, bf.y, acc);
  }
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Each warp owns R rows of B at a time; every lane issues its GV_U 16-byte
// loads of each row before using any of them.  The first rows' loads go out
// before the activations are staged in shared memory (and, when B is declared
// static, before the previous kernel in the stream has finished).
template <typename InT, typename OutT, int MT, int R>
__global__ void __launch_bounds__(GV_THREADS) k_gemv(GemvParams g) {
  extern __shared__ uint4 xs[];  // MT rows x K/8 chunks
  const int K8 = g.K / 8;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const uint4* X = reinterpret_cast<const uint4*>(g.X);
  const uint4* B = reinterpret_cast<const uint4*>(g.B);
  OutT* Y = reinterpret_cast<OutT*>(g.Y);
  const int lane = (int)lane_idx();
  const int warps = GV_THREADS / 32;
  const int gw = (int)blockIdx.x * warps + (int)warp_idx();
  const int nw = (int)gridDim.x * warps;

  uint4 bv[R][GV_U];
  auto load_rows = [&](int n0, int kc0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int u = 0; u < GV_U; ++u) {
        const int c = kc0 + u * 32 + lane;
        bv[r][u] = (c < K8 && n0 + r < g.N) ? ld_stream_v4(B + (int64_t)(n0 + r) * K8 + c) : zero;
      }
  };
  pdl_launch_dependents();
  if (!g.early_b) pdl_wait_prior_grids();
  if (gw * R < g.N) load_rows(gw * R, 0);
  if (g.early_b) pdl_wait_prior_grids();
  for (int i = threadIdx.x; i < MT * K8; i += GV_THREADS) {
    const int m = i / K8, c = i - m * K8;
    xs[i] = (m < g.M) ? X[(int64_t)m * K8 + c] : zero;
  }
  __syncthreads();

  bool preloaded = true;
  for (int n0 = gw * R; n0 < g.N; n0 += nw * R) {
    float acc[MT][R];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[m][r] = 0.f;
    for (int kc0 = 0; kc0 < K8; kc0 += 32 * GV_U) {
      if (!preloaded) load_rows(n0, kc0);
      preloaded = false;
#pragma unroll
      for (int u = 0; u < GV_U; ++u) {
        const int c = kc0 + u * 32 + lane;
        if (c < K8) {
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 xv = xs[m * K8 + c];
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = dot8<InT>(xv, bv[r][u], acc[m][r]);
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[m][r] = warp_sum(acc[m][r]);
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (m < g.M && n0 + r < g.N) {
            if constexpr (sizeof(OutT) == 4) {
              Y[(int64_t)m * g.N + n0 + r] = acc[m][r];
            } else {
              Y[(int64_t)m * g.N + n0 + r] = __float2bfloat16_rn(acc[m][r]);
            }
          }
        }
    }
  }
}

// B possibly written by the previous kernel, one activation row, K a multiple
// of 1024: two groups of GR_V 16-byte loads per lane in flight over the warp's
// stream of groups (a group is GR_V consecutive 512-byte segments of one row;
// the warp's rows are gw, gw + nw, ...), each group refilled as soon as it has
// been consumed.  Before the wait, L2 prefetches the first pf groups of the
// stream.  Four CTAs must fit an SM (512 CTAs give every warp of 1 x 4096 x
// 4096 one row in one wave), hence the register bound and the outer loop kept
// rolled: left to itself the compiler spent 76-112 registers on this loop,
// three CTAs per SM or fewer, and the launch took a microsecond longer.
constexpr int GR_G = 2;  // groups in flight per lane
constexpr int GR_V = 4;  // 16-byte loads per group

template <typename InT, typename OutT>
__global__ void __launch_bounds__(GV_THREADS, 4) k_gemv_roll(GemvParams g) {
  extern __shared__ uint4 xs[];  // the activation row, K/8 chunks
  const int K8 = g.K / 8;
  const int HPR = K8 / (32 * GR_V);  // groups per row
  const uint4* X = reinterpret_cast<const uint4*>(g.X);
  const uint4* B = reinterpret_cast<const uint4*>(g.B);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (GV_THREADS / 32) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (GV_THREADS / 32);
  const int nrows = gw < g.N ? (g.N - gw + nw - 1) / nw : 0;
  const int H = nrows * HPR;  // groups of this warp

  uint4 buf[GR_G][GR_V];
  auto load_grp = [&](int h, uint4 (&b)[GR_V]) {
    if (h < H) {
      const int r = h / HPR, j = h - r * HPR;
      const uint4* src = B + (int64_t)(gw + r * nw) * K8 + j * GR_V * 32 + lane;
#pragma unroll
      for (int v = 0; v < GR_V; ++v) b[v] = ld_stream_v4(src + v * 32);
    }
  };
  pdl_launch_dependents();
  if (g.pf_rows) {
    for (int h = 0; h < g.pf_rows && h < H; ++h) {
      const int r = h / HPR, j = h - r * HPR;
      const char* base = reinterpret_cast<const char*>(B + (int64_t)(gw + r * nw) * K8 + j * GR_V * 32);
      if (lane < GR_V * 4) prefetch_l2_line(base + lane * 128);  // the group's 16 lines
    }
  }
  if (!g.early_b) pdl_wait_prior_grids();
#pragma unroll
  for (int i = 0; i < GR_G; ++i) load_grp(i, buf[i]);
  if (g.early_b) pdl_wait_prior_grids();
  for (int i = threadIdx.x; i < K8; i += GV_THREADS) xs[i] = X[i];
  __syncthreads();
  float acc = 0.f;
#pragma unroll 1
  for (int h0 = 0; h0 < H; h0 += GR_G) {
#pragma unroll
    for (int i = 0; i < GR_G; ++i) {
      const int h = h0 + i;
      if (h < H) {
        const int r = h / HPR, j = h - r * HPR;
#pragma unroll
        for (int v = 0; v < GR_V; ++v) acc = dot8<InT>(xs[j * GR_V * 32 + v * 32 + lane], buf[i][v], acc);
        load_grp(h + GR_G, buf[i]);
        if (j == HPR - 1) {
          acc = warp_sum(acc);
          if (lane == 0) {
            if constexpr (sizeof(OutT) == 4) {
              reinterpret_cast<float*>(g.Y)[gw + r * nw] = acc;
            } else {
              reinterpret_cast<__nv_bfloat16*>(g.Y)[gw + r * nw] = __float2bfloat16_rn(acc);
            }
          }
          acc = 0.f;
        }
      }
    }
  }
}

template <typename InT>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  // rows 8-15 of A (a1, a3) are zero
  if constexpr (std::is_same<InT, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  }
}

constexpr int GM_ROWS = 8;  // weight rows per CTA
// 16-byte weight chunks per lane in flight: 4 keeps the kernel near 64
// registers, so several CTAs share an SM and their loads overlap (16 chunks:
// one CTA per SM, 2.87 TB/s at 8 x 4096 x 4096; 4 chunks: 4.42 TB/s)
constexpr int GM_J = 4;

template <typename InT, typename OutT>
__global__ void __launch_bounds__(GV_THREADS) k_gemv_mma(GemvParams g) {
  __shared__ float red[GV_THREADS / 32][GM_ROWS][8];
  const int K8 = g.K / 8;
  const int warps = GV_THREADS / 32;
  const int S = (K8 + warps - 1) / warps;  // chunks of each row in this warp's K slice
  const int w = (int)warp_idx(), lane = (int)lane_idx();
  const int gr = lane >> 2, c = lane & 3;  // fragment row / column group
  const int n0 = (int)blockIdx.x * GM_ROWS;
  const int row = n0 + gr;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const uint4* X = reinterpret_cast<const uint4*>(g.X);
  const uint4* B = reinterpret_cast<const uint4*>(g.B);
  // chunk j of this lane: 4 consecutive chunks (32 K-elements) per j across c
  auto chunk = [&](int j) { return w * S + 4 * j + c; };
  auto valid = [&](int j) { return 4 * j + c < S && chunk(j) < K8; };
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  uint4 bw[GM_J], xv[GM_J];
  const int JJ = (S + 3) / 4;

  pdl_launch_dependents();
  if (!g.early_b) pdl_wait_prior_grids();
  bool first = g.early_b != 0;  // the wait for the previous kernel is still to come
  for (int j0 = 0; j0 < JJ; j0 += GM_J) {
#pragma unroll
    for (int j = 0; j < GM_J; ++j)
      bw[j] = (j0 + j < JJ && row < g.N && valid(j0 + j)) ? ld_stream_v4(B + (int64_t)row * K8 + chunk(j0 + j)) : zero;
    if (first) pdl_wait_prior_grids();
    first = false;
#pragma unroll
    for (int j = 0; j < GM_J; ++j)
      xv[j] = (j0 + j < JJ && gr < g.M && valid(j0 + j)) ? X[(int64_t)gr * K8 + chunk(j0 + j)] : zero;
#pragma unroll
    for (int j = 0; j < GM_J; ++j) {
      mma_16816<InT>(d, bw[j].x, bw[j].y, xv[j].x, xv[j].y);
      mma_16816<InT>(d, bw[j].z, bw[j].w, xv[j].z, xv[j].w);
    }
  }
  if (first) pdl_wait_prior_grids();
  // d[0], d[1]: weight row gr, activation rows 2c and 2c + 1 (d[2], d[3]: zero rows)
  red[w][gr][2 * c] = d[0];
  red[w][gr][2 * c + 1] = d[1];
  __syncthreads();
  if ((int)threadIdx.x < GM_ROWS * 8) {
    const int r = (int)threadIdx.x >> 3, m = (int)threadIdx.x & 7;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < warps; ++q) v += red[q][r][m];
    if (m < g.M && n0 + r < g.N) {
      if constexpr (sizeof(OutT) == 4) {
        reinterpret_cast<float*>(g.Y)[(int64_t)m * g.N + n0 + r] = v;
      } else {
        reinterpret_cast<__nv_bfloat16*>(g.Y)[(int64_t)m * g.N + n0 + r] = __float2bfloat16_rn(v);
      }
    }
  }
}

template <typename InT>
__device__ __forceinline__ void mma_16816_full(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<InT, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// The same product with the weight chunks of each lane in two groups, each
// group refilled as soon as it has been consumed; the activation chunks are
// read when a group is consumed (they are small and stay in L1).  B possibly
// written by the previous kernel: before the wait, L2 prefetches the first pf
// groups of each row slice.  B static: the first two groups are loaded before
// the wait.
//
// RW weight rows per CTA (or cluster): with 8 the fragment's rows 8-15 are
// zero and each 16-byte activation chunk serves one 16-byte weight chunk; with
// 16 a lane also holds the chunk of row gr + 8, so the same activation chunk
// serves two weight chunks (half the activation reads and MMAs per weight
// byte).  A group holds 4 chunks of one row (RW = 8) or 2 chunks of each of two
// rows (RW = 16), so the registers in flight are the same.  With KS = 2 the
// two CTAs of a cluster take the two halves of K (16 K slices of 8 warps) and
// the second adds its sums into the first's shared memory, so 16 rows take as
// many CTAs as 8 rows do with KS = 1.
template <typename InT, typename OutT, int RW, int KS>
__global__ void __launch_bounds__(GV_THREADS, 4) k_gemv_mma_roll(GemvParams g) {
  static_assert(RW == 8 || RW == 16, "a CTA owns the 8 or 16 rows of one A fragment");
  static_assert(KS == 1 || KS == 2, "K split over one CTA or a cluster of two");
  __shared__ float peer[RW * 8];
  if constexpr (KS == 2) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const int rank = KS == 2 ? (int)cluster_ctarank() : 0;
  constexpr int RR = RW / 8;          // weight rows per lane
  constexpr int GJ = GM_J / RR;       // chunks per row in a group
  __shared__ float red[GV_THREADS / 32][RW][8];
  constexpr int MG = 2;  // groups in flight per lane
  const int K8 = g.K / 8;
  const int warps = GV_THREADS / 32;
  const int S = (K8 + warps * KS - 1) / (warps * KS);  // chunks of each row in this warp's K slice
  const int w = (int)warp_idx(), lane = (int)lane_idx();
  const int ws = rank * warps + w;         // K slice
  const int gr = lane >> 2, c = lane & 3;  // fragment row / column group
  const int n0 = (int)(blockIdx.x / KS) * RW;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const uint4* X = reinterpret_cast<const uint4*>(g.X);
  const uint4* B = reinterpret_cast<const uint4*>(g.B);
  // chunk j of this lane: 4 consecutive chunks (32 K-elements) per j across c
  auto chunk = [&](int j) { return ws * S + 4 * j + c; };
  auto valid = [&](int j) { return 4 * j + c < S && chunk(j) < K8; };
  const int JJ = (S + 3) / 4;
  const int NG = (JJ + GJ - 1) / GJ;  // groups of GJ chunks per row and lane
  uint4 bw[MG][RR][GJ];
  auto load_grp = [&](int q, uint4 (&b)[RR][GJ]) {
    if (q < NG) {
#pragma unroll
      for (int h = 0; h < RR; ++h) {
        const int row = n0 + gr + 8 * h;
#pragma unroll
        for (int v = 0; v < GJ; ++v) {
          const int j = q * GJ + v;
          b[h][v] = (j < JJ && row < g.N && valid(j)) ? ld_stream_v4(B + (int64_t)row * K8 + chunk(j)) : zero;
        }
      }
    }
  };

  // the next kernel on the stream may launch at once (8 rows per CTA: its CTAs
  // take the slots of this grid's later waves as they free up) or once this
  // CTA has issued its last loads (16-row clusters, one wave: 8 x 4096 x 4096
  // 4967-4977 -> 5045-5080 GB/s, 5020-5048 -> 5146-5166 with static weights;
  // the same for 8 rows per CTA at N = 14336: 5770 -> 5246)
  if constexpr (KS == 1) pdl_launch_dependents();
  // a group spans 4 * GJ chunks (GJ / 2 lines of 128 bytes) of each row
  for (int q = 0; q < g.pf_rows && q < NG; ++q) {
    const int k8 = ws * S + q * 4 * GJ + 8 * c;
#pragma unroll
    for (int h = 0; h < RR; ++h) {
      const int row = n0 + gr + 8 * h;
      if (c < GJ / 2 && row < g.N && q * 4 * GJ + 8 * c < S && k8 < K8) prefetch_l2_line(B + (int64_t)row * K8 + k8);
    }
  }
  if (!g.early_b) pdl_wait_prior_grids();
#pragma unroll
  for (int i = 0; i < MG; ++i) load_grp(i, bw[i]);
  if (g.early_b) pdl_wait_prior_grids();
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  for (int q0 = 0; q0 < NG; q0 += MG) {
    if constexpr (KS == 2) {
      if (q0 + MG >= NG) pdl_launch_dependents();
    }
#pragma unroll
    for (int i = 0; i < MG; ++i) {
      const int q = q0 + i;
      if (q < NG) {
        uint4 xv[GJ];
#pragma unroll
        for (int v = 0; v < GJ; ++v) {
          const int j = q * GJ + v;
          xv[v] = (j < JJ && gr < g.M && valid(j)) ? X[(int64_t)gr * K8 + chunk(j)] : zero;
        }
#pragma unroll
        for (int v = 0; v < GJ; ++v) {
          if constexpr (RR == 1) {
            mma_16816<InT>(d, bw[i][0][v].x, bw[i][0][v].y, xv[v].x, xv[v].y);
            mma_16816<InT>(d, bw[i][0][v].z, bw[i][0][v].w, xv[v].z, xv[v].w);
          } else {
            mma_16816_full<InT>(d, bw[i][0][v].x, bw[i][1][v].x, bw[i][0][v].y, bw[i][1][v].y, xv[v].x, xv[v].y);
            mma_16816_full<InT>(d, bw[i][0][v].z, bw[i][1][v].z, bw[i][0][v].w, bw[i][1][v].w, xv[v].z, xv[v].w);
          }
        }
        load_grp(q + MG, bw[i]);
      }
    }
  }
  // d[0], d[1]: weight row gr, activation rows 2c and 2c + 1; d[2], d[3]: weight
  // row gr + 8 (zero rows when RW = 8)
  red[w][gr][2 * c] = d[0];
  red[w][gr][2 * c + 1] = d[1];
  if constexpr (RR == 2) {
    red[w][gr + 8][2 * c] = d[2];
    red[w][gr + 8][2 * c + 1] = d[3];
  }
  __syncthreads();
  const int t = (int)threadIdx.x;
  const int r = t >> 3, m = t & 7;
  float v = 0.f;
  if (t < RW * 8) {
#pragma unroll
    for (int q = 0; q < warps; ++q) v += red[q][r][m];
  }
  if constexpr (KS == 2) {
    // the second CTA's sums go to the first CTA's shared memory (both CTAs
    // have started once the wait matching the arrive above returns); the
    // second barrier orders those stores before the first CTA's reads
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (rank == 1 && t < RW * 8) st_cluster_u32(mapa_shared(smem_u32(peer + t), 0), __float_as_uint(v));
    cluster_sync_all();
    if (rank == 1) return;
    if (t < RW * 8) v += peer[t];
  }
  if (t < RW * 8 && m < g.M && n0 + r < g.N) {
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float*>(g.Y)[(int64_t)m * g.N + n0 + r] = v;
    } else {
      reinterpret_cast<__nv_bfloat16*>(g.Y)[(int64_t)m * g.N + n0 + r] = __float2bfloat16_rn(v);
    }
  }
}

// L2 prefetch before the wait: one group per warp (or row slice) of the
// weight stream, two when each warp streams more than four groups.  Larger
// prefetches slowed the chain of dependent 1 x 4096 x 4096 launches: the
// prefetched lines compete with the previous kernel's own loads.
int prefetch_groups(int groups_per_warp) { return groups_per_warp > 4 ? 2 : 1; }

// 16 weight rows per cluster of two CTAs that split K when that grid is
// resident in one wave, else 8 rows per CTA.  Measured on bf16, 8 activation
// rows (GB/s, chain of dependent launches):
//   8 x 4096 x 4096:   8 rows per CTA 4645, 16 rows per CTA 3310, 16 rows per
//                      cluster of two 4950, 32 rows per cluster of four 4170
//   8 x 14336 x 4096:  5720-5770, 5390, 5519
// Half the CTAs (16 rows per CTA) leave half the loads in flight at N = 4096;
// the cluster form keeps the CTAs and halves the activation reads per weight
// byte, but loses where the rows take several waves.  With static weights the
// cluster form (its first two groups loaded before the wait) gives 5022-5056
// at N = 4096 against 4925-4944 for k_gemv_mma; over several waves the
// rolling kernel with early loads loses (5450 against 5865 at N = 14336).
// (Figures before the cluster form's late trigger of the next launch.)
template <typename InT, typename OutT>
cudaError_t spec_mma(int N, int K, int num_sms, bool static_b, LaunchSpec* out, int* pf) {
  int rw = GM_ROWS, ks = 1;
  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv_mma_roll<InT, OutT, 16, 2>, GV_THREADS, 0);
  if (e != cudaSuccess) return e;
  if ((int64_t)((N + 15) / 16) * 2 <= (int64_t)per_sm * num_sms) rw = 16, ks = 2;
  out->func = ks == 2    ? (const void*)k_gemv_mma_roll<InT, OutT, 16, 2>
              : static_b ? (const void*)k_gemv_mma<InT, OutT>
                         : (const void*)k_gemv_mma_roll<InT, OutT, 8, 1>;
  out->grid = dim3((unsigned)((N + rw - 1) / rw * ks), 1, 1);
  out->block = dim3(GV_THREADS, 1, 1);
  out->smem = 0;
  out->cluster = (unsigned)ks;
  out->kind = ARGS_GEMV;
  const int S = (K / 8 + 8 * ks - 1) / (8 * ks), JJ = (S + 3) / 4, gj = GM_J / (rw / 8);
  *pf = static_b ? 0 : prefetch_groups((JJ + gj - 1) / gj);
  return cudaSuccess;
}

template <typename InT, typename OutT, int MT>
cudaError_t spec_t(int N, int K, int num_sms, bool static_b, LaunchSpec* out, int* pf) {
  // rows of a warp: one at a time; the rolling kernel for one activation row
  // unless B is static
  const bool roll = !static_b && MT == 1 && K % (8 * 32 * GR_V) == 0;
  const void* k = roll ? (const void*)k_gemv_roll<InT, OutT> : (const void*)k_gemv<InT, OutT, MT, 1>;
  const size_t smem = (size_t)MT * (size_t)(K / 8) * 16;
  cudaError_t e = allow_dynamic_smem(k, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, GV_THREADS, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int rows_per_block = GV_THREADS / 32;
  const int need = (N + rows_per_block - 1) / rows_per_block;
  const int grid = std::max(1, std::min(need, per_sm * num_sms));
  out->func = k;
  out->grid = dim3((unsigned)grid, 1, 1);
  out->block = dim3(GV_THREADS, 1, 1);
  out->smem = smem;
  out->cluster = 1;
  out->kind = ARGS_GEMV;
  const int warps = grid * rows_per_block;
  const int rows_per_warp = (N + warps - 1) / warps;
  *pf = roll ? prefetch_groups(rows_per_warp * (K / 8) / (32 * GR_V)) : 0;
  return cudaSuccess;
}

template <typename InT, typename OutT>
cudaError_t spec_m(int M, int N, int K, int num_sms, bool static_b, LaunchSpec* out, int* pf) {
  // one row per warp at a time for M <= 2: twice the CTAs of two rows per warp,
  // which spreads short weight streams more evenly over the SMs (4096 x 4096:
  // 3.99 -> 4.49 TB/s; 14336 x 4096: 5.70 -> 6.05 TB/s)
  if (M <= 1) return spec_t<InT, OutT, 1>(N, K, num_sms, static_b, out, pf);
  if (M <= 2) return spec_t<InT, OutT, 2>(N, K, num_sms, static_b, out, pf);
  if (M <= 8) return spec_mma<InT, OutT>(N, K, num_sms, static_b, out, pf);
  return spec_t<InT, OutT, 16>(N, K, num_sms, static_b, out, pf);
}

}  // namespace

size_t gemv_smem_bytes(int M, int K) {
  if (M >= 3 && M <= 8) return 0;  // k_gemv_mma keeps its operands in registers
  const int mt = M <= 1 ? 1 : M <= 2 ? 2 : 16;
  return (size_t)mt * (size_t)(K / 8) * 16;
}

cudaError_t spec_gemv(int M, int N, int K, bool in_bf16, bool out_f32, int num_sms, bool static_b, LaunchSpec* out,
                      int* pf_groups) {
  if (in_bf16) {
    return out_f32 ? spec_m<__nv_bfloat16, float>(M, N, K, num_sms, static_b, out, pf_groups)
                   : spec_m<__nv_bfloat16, __nv_bfloat16>(M, N, K, num_sms, static_b, out, pf_groups);
  }
  return out_f32 ? spec_m<__half, float>(M, N, K, num_sms, static_b, out, pf_groups)
                 : spec_m<__half, __nv_bfloat16>(M, N, K, num_sms, static_b, out, pf_groups);
}

}  // namespace dgb
