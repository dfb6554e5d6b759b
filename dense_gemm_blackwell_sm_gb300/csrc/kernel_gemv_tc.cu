// kernel_gemv_tc.cu -- decode-shaped Y (M x N) = X (M x K) * B^T for M <= 16 on
// the Tensor Core, with the operands swapped.
//
// The decode product is bandwidth-bound (reading notes of "Modern GPU
// Programming for MLSys", section "Roofline：找到天花板": about one FLOP per
// byte at M = 1).  With a few activation rows (M = 8) the CUDA cores would
// still need 4 fp32 FMAs per weight byte, close to their own limit, so here
// the MMA does the arithmetic: the weight tile (128 rows of B) is the
// 128-row A operand of tcgen05.mma, the activations (M rows, zero-filled by
// TMA up to 16) are the 16-column B operand, and D[n][m] = sum_k B[n][k] X[m][k]
// lands in 16 TMEM columns.  Only the weight stream matters for time:
//   * one CTA per 128-row block of B, or, when that gives too few CTAs, a
//     cluster of `split` CTAs that share the block's K range;
//   * the producer starts the TMA ring (weight box + activation box per stage)
//     right after barrier set-up, before anything else;
//   * a split block's partial sums are added in rank order through
//     distributed shared memory by the leader CTA, which writes Y.
// No global scratch is used.
#include <algorithm>

#include "idesc.h"
#include "kernel_common.cuh"
#include "launch.h"

namespace dgb {

namespace {

constexpr int TG_THREADS = 128;
constexpr int TG_BK = 64;
constexpr uint32_t TG_B_BYTES = 128u * 128u;  // one weight box: 128 rows x 64 K
constexpr uint32_t TG_X_BYTES = 16u * 128u;   // one activation box: 16 rows x 64 K
constexpr uint32_t TG_STAGE = TG_B_BYTES + TG_X_BYTES;
constexpr int TG_MAX_STAGES = 12;

template <typename OutT>
__global__ void __launch_bounds__(TG_THREADS, 1)
    k_gemv_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX, TgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  const int S = p.stages;
  uint8_t* ring = smem;  // stage s: weight box at s*18K, activation box at s*18K + 16K
  float* partial = reinterpret_cast<float*>(ring + (size_t)S * TG_STAGE);  // 128 x 16 fp32
  uint64_t* full = reinterpret_cast<uint64_t*>(partial + 128 * 16);
  uint64_t* empty = full + TG_MAX_STAGES;
  uint64_t* done = empty + TG_MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const uint32_t tid = threadIdx.x, warp = warp_idx(), lane = lane_idx();
  const uint32_t rank = (p.split > 1) ? cluster_ctarank() : 0u;
  const int32_t rb = (int32_t)(blockIdx.x / (uint32_t)p.split);  // 128-row block of B and Y
  const int32_t n0 = rb * 128;
  const int32_t KB = (p.K + TG_BK - 1) / TG_BK;
  const int32_t kb0 = (int32_t)rank * p.kblocks_per_cta;
  const int32_t nkb = max(0, min(p.kblocks_per_cta, KB - kb0));

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(tmem_slot), 32);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{abort_flag, p.status, p.timeout_ns, 0};

  if (warp == 0 && lane == 0) {
    // producer: weight box + activation box per stage.  The first ring's weight
    // boxes go out before waiting for the previous kernel in the stream (a
    // no-op unless launched as its programmatic dependent), the activation
    // boxes only after it.
    const int32_t pre = min(nkb, S);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int32_t j = 0; j < pre; ++j) {
      const uint32_t fb = smem_u32(full + j);
      mbar_arrive_expect_tx(fb, TG_STAGE);
      tma_load_2d(smem_u32(ring + (size_t)j * TG_STAGE), &tmB, fb, (kb0 + j) * TG_BK, n0);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int32_t j = 0; j < pre; ++j)
      tma_load_2d(smem_u32(ring + (size_t)j * TG_STAGE + TG_B_BYTES), &tmX, smem_u32(full + j), (kb0 + j) * TG_BK, 0);
    for (int32_t j = pre; j < nkb; ++j) {
      const int s = j % S;
      const uint32_t ph = (uint32_t)(j / S) & 1u;
      if (!mbar_wait(smem_u32(empty + s), ph ^ 1u, w, WAIT_PRODUCER_EMPTY)) break;
      const uint32_t fb = smem_u32(full + s);
      mbar_arrive_expect_tx(fb, TG_STAGE);
      uint8_t* st = ring + (size_t)s * TG_STAGE;
      tma_load_2d(smem_u32(st), &tmB, fb, (kb0 + j) * TG_BK, n0);
      tma_load_2d(smem_u32(st + TG_B_BYTES), &tmX, fb, (kb0 + j) * TG_BK, 0);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    for (int32_t j = 0; j < nkb; ++j) {
      const int s = j % S;
      const uint32_t ph = (uint32_t)(j / S) & 1u;
      if (!mbar_wait(smem_u32(full + s), ph, w, WAIT_MMA_FULL)) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(ring + (size_t)s * TG_STAGE);
      const uint64_t ad = sdesc_k_sw128(sa), bd = sdesc_k_sw128(sa + TG_B_BYTES);
#pragma unroll
      for (int k = 0; k < TG_BK / 16; ++k) mma_f16<1>(tmem, ad + 2 * k, bd + 2 * k, p.idesc, (j | k) != 0);
      mma_commit(smem_u32(empty + s));
    }
    mma_commit(smem_u32(done));
  }
  __syncwarp();
  bool ok = mbar_wait(smem_u32(done), 0, w, WAIT_LADDER_MMA);
  ok = __syncthreads_and(ok && *abort_flag == 0u) != 0;
  const uint32_t row = warp * 32u + lane;  // TMEM lane = row of the block
  float acc[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) acc[m] = 0.f;
  if (ok && nkb > 0) {
    tc_fence_after();
    uint32_t v[16];
    tmem_ld_32x32b_x16(tmem + ((warp * 32u) << 16), v);
    tmem_wait_ld();
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = __uint_as_float(v[m]);
  }
  if (p.split > 1) {
    float4* dst = reinterpret_cast<float4*>(partial + row * 16);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    cluster_sync_all();
    if (rank == 0) {
      // leader: add the cluster's partials in rank order
#pragma unroll
      for (int m = 0; m < 16; ++m) acc[m] = 0.f;
      const uint32_t my = smem_u32(partial + row * 16);
      for (int r = 0; r < p.split; ++r) {
        const uint32_t src = mapa_shared(my, (uint32_t)r);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = ld_cluster_f32x4(src + 16u * q);
          acc[4 * q] += f.x;
          acc[4 * q + 1] += f.y;
          acc[4 * q + 2] += f.z;
          acc[4 * q + 3] += f.w;
        }
      }
    }
  }
  const int32_t n = n0 + (int32_t)row;
  if (ok && rank == 0 && n < p.N) {
    OutT* Y = reinterpret_cast<OutT*>(p.Y);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m < p.M) {
        if constexpr (sizeof(OutT) == 4) {
          Y[(int64_t)m * p.N + n] = acc[m];
        } else {
          Y[(int64_t)m * p.N + n] = __float2bfloat16_rn(acc[m]);
        }
      }
    }
  }
  if (!ok && tid == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) {}
  }
  if (p.split > 1) cluster_sync_all();  // peers keep their partials until the leader has read them
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, 32);
  }
}

size_t tg_smem(int stages) {
  return 1024 + (size_t)stages * TG_STAGE + 128 * 16 * 4 + (2 * TG_MAX_STAGES + 1) * 8 + 16;
}

}  // namespace

// CTAs per 128-row block along K (`split`, a cluster when > 1) and ring depth:
// the largest power-of-two split (at most 4) whose CTAs all fit at once with
// two CTAs per SM; an 8-stage ring when one CTA per SM suffices, else 4
// stages so that two CTAs share an SM.  `want_split` / `want_stages` override.
void gemv_tc_config(int N, int K, int num_sms, int want_split, int want_stages, int* split, int* stages,
                    int* kblocks_per_cta) {
  const int KB = (K + TG_BK - 1) / TG_BK;
  const int rbs = (N + 127) / 128;
  int sp = 1;
  if (want_split > 0) {
    while (sp * 2 <= want_split && sp < 8) sp *= 2;
  } else {
    while (sp < 4 && rbs * sp * 2 <= 2 * num_sms) sp *= 2;
  }
  while (sp > 1 && sp > KB) sp /= 2;
  *split = sp;
  *kblocks_per_cta = (KB + sp - 1) / sp;
  *stages = want_stages > 0 ? std::min(want_stages, TG_MAX_STAGES) : (rbs * sp <= num_sms ? 8 : 4);
}

size_t gemv_tc_smem_bytes(int stages) { return tg_smem(stages); }

cudaError_t spec_gemv_tc(int M, int N, int K, bool in_bf16, bool out_f32, int num_sms, int want_split,
                         int want_stages, LaunchSpec* out, TgParams* base) {
  TgParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  gemv_tc_config(N, K, num_sms, want_split, want_stages, &p.split, &p.stages, &p.kblocks_per_cta);
  // instruction descriptor: f32 accumulate, fp16/bf16 operands, K-major, M = 128, N = 16
  p.idesc = idesc_f16(in_bf16, 128, 16);
  const size_t smem = tg_smem(p.stages);
  const void* k = out_f32 ? (const void*)k_gemv_tc<float> : (const void*)k_gemv_tc<__nv_bfloat16>;
  cudaError_t e = allow_dynamic_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  out->func = k;
  out->grid = dim3((unsigned)(((N + 127) / 128) * p.split), 1, 1);
  out->block = dim3(TG_THREADS, 1, 1);
  out->smem = smem;
  out->cluster = (unsigned)p.split;
  out->kind = ARGS_BX_TG;
  *base = p;
  return cudaSuccess;
}

}  // namespace dgb
