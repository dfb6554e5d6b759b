// kernels_ladder.cu -- the first six steps of the tiled GEMM, C = A * B^T.
//
// "Modern GPU Programming for MLSys" (reading notes, section "9 步优化")
// builds the GEMM in nine steps; this file holds steps 1-6, each a complete,
// correct kernel on its own:
//
//   step 1  one CTA computes one 128x128 output tile: GMEM -> SMEM (thread
//           copies) -> tcgen05.mma into a TMEM accumulator -> tcgen05.ld -> GMEM;
//   step 2  a K loop of 64-wide blocks accumulating into the same TMEM
//           accumulator, one SMEM staging buffer overwritten every iteration;
//   step 3  a 2-D grid of CTAs, one output tile each;
//   step 4  the SMEM fills become TMA tile copies tracked by an mbarrier with
//           an expected byte count;
//   step 5  a ring of staging buffers (two in the pages' telling, any depth
//           here): block k+S loads while block k computes, but the single
//           issuing thread still waits for each MMA before it refills;
//   step 6  a persistent kernel: about one CTA per SM takes tiles from a
//           scheduler (static stride, a global atomic counter, or hardware
//           cluster launch control) in grouped raster order for L2 reuse.
//
// Steps 1-3 share one kernel (a 1x1 grid with K <= 64 is step 1; a 1x1 grid
// is step 2).  All of them use a 128x128 tile, 128 threads (4 warps: warp w
// reads TMEM lanes 32w..32w+31 in the epilogue) and K-major operand tiles in
// the 128-byte swizzled layout that the Tensor Core reads directly.
#include <mutex>

#include "kernel_common.cuh"
#include "launch.h"

namespace dgb {

namespace {

constexpr int LT_M = 128;            // tile rows (TMEM lanes)
constexpr int LT_N = 128;            // tile columns (TMEM fp32 columns)
constexpr int LT_K = 64;             // K block: 64 x 16-bit = one 128-byte swizzle row
constexpr int LT_TILE_BYTES = LT_M * LT_K * 2;  // 16 KB per operand per stage
constexpr int LT_THREADS = 128;

// TMEM accumulator -> registers -> C (one row per thread, 32 columns at a time)
template <typename OutT>
__device__ __forceinline__ void ladder_epilogue(const KParams& p, uint32_t tmem, int32_t m0,
                                                int32_t n0) {
  const uint32_t warp = warp_idx(), lane = lane_idx();
  const int32_t row = m0 + (int32_t)(warp * 32 + lane);
#pragma unroll 1
  for (int ch = 0; ch < LT_N / 32; ++ch) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tmem + ((warp * 32u) << 16) + (uint32_t)(ch * 32), v);
    tmem_wait_ld();
    const int32_t col0 = n0 + ch * 32;
    if (row < p.M && col0 < p.N) store_row32<OutT>(reinterpret_cast<OutT*>(p.C), p.out_ld, row, col0, p.N, v);
  }
}

// ---------------------------------------------------------------------------
// steps 1-3: thread copies into one staging buffer, one tile per CTA

template <typename OutT>
__global__ void __launch_bounds__(LT_THREADS) k_step123(KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + LT_TILE_BYTES;
  uint64_t* bar_mma = reinterpret_cast<uint64_t*>(smem + 2 * LT_TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t tid = threadIdx.x, warp = warp_idx();
  const int32_t m0 = blockIdx.y * LT_M, n0 = blockIdx.x * LT_N;
  if (tid == 0) {
    mbar_init(smem_u32(bar_mma), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(tmem_slot), LT_N);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.status, p.timeout_ns, 0};

  const int32_t KB = (p.K + LT_K - 1) / LT_K;
  const uint64_t adesc = sdesc_k_sw128(smem_u32(sA));
  const uint64_t bdesc = sdesc_k_sw128(smem_u32(sB));
  uint32_t phase = 0;
  bool ok = true;
  for (int32_t kb = 0; kb < KB && ok; ++kb) {
    // every thread copies 8 of the 1024 16-byte chunks of each operand tile
    for (int i = tid; i < LT_M * (LT_K / 8); i += LT_THREADS) {
      const int r = i >> 3, c = i & 7;
      const int32_t gk = kb * LT_K + c * 8;  // K % 8 == 0: a chunk is wholly in or out
      uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
      if (m0 + r < p.M && gk < p.K) va = *reinterpret_cast<const uint4*>(p.A + (int64_t)(m0 + r) * p.K + gk);
      if (n0 + r < p.N && gk < p.K) vb = *reinterpret_cast<const uint4*>(p.B + (int64_t)(n0 + r) * p.K + gk);
      *reinterpret_cast<uint4*>(sA + sw128_offset(r, c)) = va;
      *reinterpret_cast<uint4*>(sB + sw128_offset(r, c)) = vb;
    }
    fence_proxy_async_smem();  // thread writes -> visible to the Tensor Core
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < LT_K / 16; ++k)
        mma_f16<1>(tmem, adesc + 2 * k, bdesc + 2 * k, p.idesc, (kb | k) != 0);
      mma_commit(smem_u32(bar_mma));
    }
    // the MMA reads the staging buffer asynchronously: wait before overwriting it
    bool mine = mbar_wait(smem_u32(bar_mma), phase, w, WAIT_LADDER_MMA);
    phase ^= 1u;
    ok = __syncthreads_and(mine) != 0;
  }
  if (ok) {
    tc_fence_after();
    ladder_epilogue<OutT>(p, tmem, m0, n0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, LT_N);
  }
}

// ---------------------------------------------------------------------------
// steps 4 and 5: TMA copies; a ring of `stages` buffers (1 = step 4)

template <typename OutT>
__global__ void __launch_bounds__(LT_THREADS) k_step45(const __grid_constant__ CUtensorMap tmA,
                                                       const __grid_constant__ CUtensorMap tmB,
                                                       KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  const int S = p.stages;
  uint8_t* ring = smem;  // stage s: A at s*32K, B at s*32K + 16K
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * 2 * LT_TILE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* done = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t tid = threadIdx.x, warp = warp_idx();
  const int32_t m0 = blockIdx.y * LT_M, n0 = blockIdx.x * LT_N;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(tmem_slot), LT_N);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.status, p.timeout_ns, 0};
  const int32_t KB = (p.K + LT_K - 1) / LT_K;

  if (tid == 0) {
    auto load = [&](int32_t kb) {
      const int s = kb % S;
      uint8_t* sA = ring + s * 2 * LT_TILE_BYTES;
      mbar_arrive_expect_tx(smem_u32(full + s), 2 * LT_TILE_BYTES);
      tma_load_2d(smem_u32(sA), &tmA, smem_u32(full + s), kb * LT_K, m0);
      if (!((p.debug_flags & DEBUG_SKIP_ONE_LOAD) && kb == 0))
        tma_load_2d(smem_u32(sA + LT_TILE_BYTES), &tmB, smem_u32(full + s), kb * LT_K, n0);
    };
    bool ok = true;
    for (int32_t kb = 0; kb < min(S, KB); ++kb) load(kb);
    for (int32_t kb = 0; kb < KB && ok; ++kb) {
      const int s = kb % S;
      const uint32_t ph = (uint32_t)(kb / S) & 1u;
      if (!mbar_wait(smem_u32(full + s), ph, w, WAIT_LADDER_TMA)) { ok = false; break; }
      tc_fence_after();
      const uint32_t a_addr = smem_u32(ring + s * 2 * LT_TILE_BYTES);
      const uint64_t adesc = sdesc_k_sw128(a_addr), bdesc = sdesc_k_sw128(a_addr + LT_TILE_BYTES);
#pragma unroll
      for (int k = 0; k < LT_K / 16; ++k)
        mma_f16<1>(tmem, adesc + 2 * k, bdesc + 2 * k, p.idesc, (kb | k) != 0);
      mma_commit(smem_u32(empty + s));
      if (kb + S < KB) {
        // the same thread refills the slot only after its MMA has drained it
        if (!mbar_wait(smem_u32(empty + s), ph, w, WAIT_LADDER_MMA)) { ok = false; break; }
        load(kb + S);
      }
    }
    mma_commit(smem_u32(done));  // arrives once every MMA issued above is complete
  }
  __syncwarp();
  bool mine = mbar_wait(smem_u32(done), 0, w, WAIT_LADDER_MMA);
  const bool ok = __syncthreads_and(mine && *abort_flag == 0) != 0;
  if (ok) {
    tc_fence_after();
    ladder_epilogue<OutT>(p, tmem, m0, n0);
  } else if (tid == 0) {
    // leave time for copies still in flight before the CTA's SMEM goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {}
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, LT_N);
  }
}

// ---------------------------------------------------------------------------
// step 6: persistent CTAs fed by a tile scheduler

enum Sched6 { S6_STATIC = 0, S6_ATOMIC = 1, S6_CLC = 2 };

template <typename OutT, int SCHED>
__global__ void __launch_bounds__(LT_THREADS, 1) k_step6(const __grid_constant__ CUtensorMap tmA,
                                                         const __grid_constant__ CUtensorMap tmB,
                                                         KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  const int S = p.stages;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * 2 * LT_TILE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* done = empty + S;
  uint64_t* clc_bar = done + 1;
  uint32_t* clc_resp = reinterpret_cast<uint32_t*>(clc_bar + 1);  // 16 bytes, 16-aligned
  uint32_t* tmem_slot = clc_resp + 4;
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int32_t* next_tile = reinterpret_cast<volatile int32_t*>(tmem_slot + 2);

  const uint32_t tid = threadIdx.x, warp = warp_idx();
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(done), 1);
    mbar_init(smem_u32(clc_bar), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(tmem_slot), LT_N);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.status, p.timeout_ns, 0};
  const int32_t KB = (p.K + LT_K - 1) / LT_K;
  const int32_t total = p.tiles_m * p.tiles_n;

  int32_t tile = (SCHED == S6_ATOMIC) ? -1 : (int32_t)blockIdx.x;
  if (SCHED == S6_ATOMIC && tid == 0) {
    const int32_t t = (int32_t)atomicAdd(p.status + 1, 1u);
    *next_tile = t < total ? t : -1;
  }
  if (SCHED == S6_ATOMIC) {
    __syncthreads();
    tile = *next_tile;
  }
  uint32_t g_load = 0, g_mma = 0;  // running k-block counters across tiles (ring state)
  uint32_t tiles_done = 0, clc_phase = 0;
  bool ok = true;
  while (ok && tile >= 0 && tile < total) {
    int32_t tm, tn;
    raster_tile(tile, p.tiles_m, p.tiles_n, p.raster_group, tm, tn);
    const int32_t m0 = tm * LT_M, n0 = tn * LT_N;
    if (tid == 0) {
      auto load = [&](int32_t kb) -> bool {
        const uint32_t s = g_load % (uint32_t)S;
        if (g_load >= (uint32_t)S) {
          const uint32_t ph = ((g_load / (uint32_t)S) - 1u) & 1u;
          if (!mbar_wait(smem_u32(empty + s), ph, w, WAIT_LADDER_MMA)) return false;
        }
        uint8_t* sA = ring + s * 2 * LT_TILE_BYTES;
        mbar_arrive_expect_tx(smem_u32(full + s), 2 * LT_TILE_BYTES);
        tma_load_2d(smem_u32(sA), &tmA, smem_u32(full + s), kb * LT_K, m0);
        tma_load_2d(smem_u32(sA + LT_TILE_BYTES), &tmB, smem_u32(full + s), kb * LT_K, n0);
        ++g_load;
        return true;
      };
      bool tok = true;
      int32_t issued = 0;
      for (; issued < min(S, KB) && tok; ++issued) tok = load(issued);
      for (int32_t kb = 0; kb < KB && tok; ++kb) {
        const uint32_t s = g_mma % (uint32_t)S;
        const uint32_t ph = (g_mma / (uint32_t)S) & 1u;
        if (!mbar_wait(smem_u32(full + s), ph, w, WAIT_LADDER_TMA)) { tok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + s * 2 * LT_TILE_BYTES);
        const uint64_t adesc = sdesc_k_sw128(a_addr), bdesc = sdesc_k_sw128(a_addr + LT_TILE_BYTES);
#pragma unroll
        for (int k = 0; k < LT_K / 16; ++k)
          mma_f16<1>(tmem, adesc + 2 * k, bdesc + 2 * k, p.idesc, (kb | k) != 0);
        mma_commit(smem_u32(empty + s));
        ++g_mma;
        if (issued < KB) { tok = load(issued); ++issued; }
      }
      mma_commit(smem_u32(done));
      // fetch the next tile while the MMAs finish
      int32_t nt = -1;
      if (SCHED == S6_STATIC) {
        nt = tile + (int32_t)gridDim.x;
      } else if (SCHED == S6_ATOMIC) {
        nt = (int32_t)atomicAdd(p.status + 1, 1u);
      } else {
        mbar_arrive_expect_tx(smem_u32(clc_bar), 16);
        clc_try_cancel(smem_u32(clc_resp), smem_u32(clc_bar));
        if (mbar_wait(smem_u32(clc_bar), clc_phase, w, WAIT_CLC)) {
          uint32_t x;
          nt = clc_decode(smem_u32(clc_resp), x) ? (int32_t)x : -1;
        } else {
          tok = false;
        }
        clc_phase ^= 1u;
      }
      *next_tile = (nt >= 0 && nt < total) ? nt : -1;
      if (!tok) *abort_flag = 1u;
    }
    __syncwarp();
    bool mine = mbar_wait(smem_u32(done), tiles_done & 1u, w, WAIT_LADDER_MMA);
    ok = __syncthreads_and(mine && *abort_flag == 0) != 0;
    ++tiles_done;
    if (!ok) break;
    tc_fence_after();
    ladder_epilogue<OutT>(p, tmem, m0, n0);
    if (p.visits != nullptr && tid == 0) atomicAdd(p.visits + tile, 1);
    tile = *next_tile;
    // the accumulator is rewritten by the next tile: all TMEM reads first
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (SCHED == S6_ATOMIC && tid == 0 && ok) {
    // the last CTA to run out of tiles rewinds the counters for the next launch
    __threadfence();
    if (atomicAdd(p.status + 2, 1u) == gridDim.x - 1) {
      atomicExch(p.status + 1, 0u);
      atomicExch(p.status + 2, 0u);
    }
  }
  if (!ok && tid == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {}
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, LT_N);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// launch specs (made once per plan)

static size_t ladder_smem(int stages) {
  return 1024 + (size_t)stages * 2 * LT_TILE_BYTES + (size_t)(2 * stages + 2) * 8 + 64;
}

size_t step6_smem_bytes(int stages) { return ladder_smem(stages) + 32; }

static cudaError_t finish_spec(const void* k, dim3 grid, size_t smem, int kind, LaunchSpec* out) {
  cudaError_t e = allow_dynamic_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  out->func = k;
  out->grid = grid;
  out->block = dim3(LT_THREADS, 1, 1);
  out->smem = smem;
  out->cluster = 1;
  out->kind = kind;
  return cudaSuccess;
}

cudaError_t spec_step123(int M, int N, bool out_f32, LaunchSpec* out) {
  const dim3 grid((N + LT_N - 1) / LT_N, (M + LT_M - 1) / LT_M);
  const void* k = out_f32 ? (const void*)k_step123<float> : (const void*)k_step123<__nv_bfloat16>;
  return finish_spec(k, grid, ladder_smem(1), ARGS_K, out);
}

cudaError_t spec_step45(int M, int N, int stages, bool out_f32, LaunchSpec* out) {
  const dim3 grid((N + LT_N - 1) / LT_N, (M + LT_M - 1) / LT_M);
  const void* k = out_f32 ? (const void*)k_step45<float> : (const void*)k_step45<__nv_bfloat16>;
  return finish_spec(k, grid, ladder_smem(stages), ARGS_AB_K, out);
}

cudaError_t spec_step6(int sched, int stages, bool out_f32, int grid, LaunchSpec* out) {
  const void* k;
  if (out_f32) {
    k = sched == S6_ATOMIC ? (const void*)k_step6<float, S6_ATOMIC>
        : sched == S6_CLC  ? (const void*)k_step6<float, S6_CLC>
                           : (const void*)k_step6<float, S6_STATIC>;
  } else {
    k = sched == S6_ATOMIC ? (const void*)k_step6<__nv_bfloat16, S6_ATOMIC>
        : sched == S6_CLC  ? (const void*)k_step6<__nv_bfloat16, S6_CLC>
                           : (const void*)k_step6<__nv_bfloat16, S6_STATIC>;
  }
  return finish_spec(k, dim3((unsigned)grid, 1, 1), step6_smem_bytes(stages), ARGS_AB_K, out);
}

// The dynamic shared-memory limit is an attribute of the kernel, shared by every
// plan that uses it: raise it when a plan needs more, never lower it (a plan
// with a shallower ring must not make an earlier, deeper one unlaunchable).
cudaError_t allow_dynamic_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, func);
  if (e != cudaSuccess) return e;
  if ((size_t)a.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
  return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_spec(const LaunchSpec& s, void** args, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = s.grid;
  cfg.blockDim = s.block;
  cfg.dynamicSmemBytes = s.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (s.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = s.cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (s.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, s.func, args);
}

}  // namespace dgb
