// kernels_ws.cu -- instantiations of the step 7-9 kernels (fp16 / bf16 / 8-bit
// float inputs) and their launch shapes; the kernel itself is in kernels_ws.cuh.
#include "kernels_ws.cuh"

namespace dgb {

namespace {

template <typename OutT, int CG, int NCONS = 1>
void* pick_fused(int act) {
  switch (act) {
    case EPI_ACT_RELU: return ws_kernel_ptr<OutT, CG, NCONS, SCHED_STATIC, EPI_ACT_RELU>();
    case EPI_ACT_SILU: return ws_kernel_ptr<OutT, CG, NCONS, SCHED_STATIC, EPI_ACT_SILU>();
    case EPI_ACT_GELU_TANH: return ws_kernel_ptr<OutT, CG, NCONS, SCHED_STATIC, EPI_ACT_GELU_TANH>();
    case EPI_ACT_GELU_ERF: return ws_kernel_ptr<OutT, CG, NCONS, SCHED_STATIC, EPI_ACT_GELU_ERF>();
    default: return ws_kernel_ptr<OutT, CG, NCONS, SCHED_STATIC, EPI_ACT_NONE>();
  }
}

// the fused-epilogue kernels exist for the static scheduler: every activation with
// one MMA consumer (steps 7 and 8) and with two on the CTA pair for bf16 C (step 9,
// whose writeback applies the epilogue while draining each accumulator); fp32 C
// on step 9 with bias / residual / scales alone
template <int CG, int NCONS>
void* pick_kernel(int sched, bool out_f32, int fused_act) {
  if (fused_act >= 0) {
    if constexpr (NCONS == 2) {
      if (CG != 2) return nullptr;
      if (out_f32) return fused_act == EPI_ACT_NONE ? ws_kernel_ptr<float, 2, 2, SCHED_STATIC, EPI_ACT_NONE>() : nullptr;
      return pick_fused<__nv_bfloat16, 2, 2>(fused_act);
    } else {
      return out_f32 ? pick_fused<float, CG>(fused_act) : pick_fused<__nv_bfloat16, CG>(fused_act);
    }
  }
  if (sched == SCHED_STREAM_K) {
    return out_f32 ? reinterpret_cast<void*>(k_ws_sk<float, CG, NCONS>)
                   : reinterpret_cast<void*>(k_ws_sk<__nv_bfloat16, CG, NCONS>);
  }
  if (out_f32) {
    if (sched == SCHED_ATOMIC) return ws_kernel_ptr<float, CG, NCONS, SCHED_ATOMIC>();
    if (sched == SCHED_CLC) return ws_kernel_ptr<float, CG, NCONS, SCHED_CLC>();
    return ws_kernel_ptr<float, CG, NCONS, SCHED_STATIC>();
  }
  if (sched == SCHED_ATOMIC) return ws_kernel_ptr<__nv_bfloat16, CG, NCONS, SCHED_ATOMIC>();
  if (sched == SCHED_CLC) return ws_kernel_ptr<__nv_bfloat16, CG, NCONS, SCHED_CLC>();
  return ws_kernel_ptr<__nv_bfloat16, CG, NCONS, SCHED_STATIC>();
}

// The 224-column tile exists for step 9 with the static schedule and the plain
// writeback (the shapes whose waves it evens out).
void* ws_kernel(int cg, int consumers, int sched, bool out_f32, int fused_act = -1, int bn = WS_BN) {
  if (bn == 224) {
    if (cg != 2 || consumers != 2 || sched != SCHED_STATIC || fused_act >= 0) return nullptr;
    return out_f32 ? ws_kernel_ptr<float, 2, 2, SCHED_STATIC, -1, 224>()
                   : ws_kernel_ptr<__nv_bfloat16, 2, 2, SCHED_STATIC, -1, 224>();
  }
  if (bn != WS_BN) return nullptr;
  if (cg == 1 && consumers == 1) return pick_kernel<1, 1>(sched, out_f32, fused_act);
  if (cg == 1 && consumers == 2) return pick_kernel<1, 2>(sched, out_f32, fused_act);
  if (cg == 2 && consumers == 1) return pick_kernel<2, 1>(sched, out_f32, fused_act);
  if (cg == 2 && consumers == 2) return pick_kernel<2, 2>(sched, out_f32, fused_act);
  return nullptr;
}

}  // namespace

WsShape ws_shape(int cg, int consumers, int bn) {
  WsShape s{};
  s.cg = cg;
  s.consumers = consumers;
  s.tile_m = 128 * cg * consumers;
  s.tile_n = bn;
  s.a_box_rows = 128;
  s.b_box_rows = (cg == 1) ? bn : bn / 2;
  s.stage_bytes = consumers * (int)WS_A_BYTES + s.b_box_rows * 128;
  s.threads = WS_THREADS;
  return s;
}

size_t ws_sk_slot_floats(int cg, int consumers) { return (size_t)cg * consumers * 4 * SK_WARP_FLOATS; }

size_t ws_smem_bytes(int cg, int consumers, int stages, int bn) {
  return 1024 + (size_t)stages * ws_shape(cg, consumers, bn).stage_bytes + WS_STAGING + WS_CTRL;
}

int ws_max_stages(int cg, int consumers, int bn) {
  int s = WS_MAX_STAGES;
  while (s > 1 && ws_smem_bytes(cg, consumers, s, bn) > WS_SMEM_LIMIT) --s;
  return s;
}

static cudaLaunchConfig_t ws_config(int cg, int clusters, size_t smem, cudaStream_t st,
                                    cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(clusters * cg), 1, 1);
  cfg.blockDim = dim3(WS_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int ws_max_active_clusters(int cg, int consumers, int sched, bool out_f32, int stages, int bn) {
  void* k = ws_kernel(cg, consumers, sched, out_f32, -1, bn);
  if (!k) return 0;
  const size_t smem = ws_smem_bytes(cg, consumers, stages, bn);
  if (allow_dynamic_smem((const void*)k, smem) != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = ws_config(cg, 1, smem, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename OutT, int CG>
void* ks_kernel(bool l2) {
  return l2 ? reinterpret_cast<void*>(k_ws_ks<OutT, true, CG>) : reinterpret_cast<void*>(k_ws_ks<OutT, false, CG>);
}

cudaError_t spec_ws_ks(int cg, bool out_f32, int stages, int tiles, int split, LaunchSpec* out) {
  if ((cg != 1 && cg != 2) || split < 2 || split * cg > 8) return cudaErrorInvalidValue;
  const bool l2 = split > 2;
  void* k = cg == 1 ? (out_f32 ? ks_kernel<float, 1>(l2) : ks_kernel<__nv_bfloat16, 1>(l2))
                    : (out_f32 ? ks_kernel<float, 2>(l2) : ks_kernel<__nv_bfloat16, 2>(l2));
  // two slices exchange their 128 KB partials through their stage rings
  if (!l2 && (size_t)stages * ws_shape(cg, 1).stage_bytes < (size_t)128 * 1024) return cudaErrorInvalidValue;
  const size_t smem = ws_smem_bytes(cg, 1, stages);
  cudaError_t e = allow_dynamic_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  out->func = k;
  out->grid = dim3((unsigned)(tiles * split * cg), 1, 1);
  out->block = dim3(WS_THREADS, 1, 1);
  out->smem = smem;
  out->cluster = (unsigned)(split * cg);
  out->kind = ARGS_ABC_K;
  return cudaSuccess;
}

cudaError_t spec_ws(int cg, int consumers, int sched, bool out_f32, int stages, int clusters, LaunchSpec* out,
                    int fused_act, int bn) {
  void* k = ws_kernel(cg, consumers, fused_act >= 0 ? SCHED_STATIC : sched, out_f32, fused_act, bn);
  if (!k) return cudaErrorInvalidValue;
  const size_t smem = ws_smem_bytes(cg, consumers, stages, bn);
  cudaError_t e = allow_dynamic_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  out->func = k;
  out->grid = dim3((unsigned)(clusters * cg), 1, 1);
  out->block = dim3((unsigned)ws_threads(consumers, fused_act), 1, 1);
  out->smem = smem;
  out->cluster = (unsigned)cg;
  out->kind = ARGS_ABC_K;
  return cudaSuccess;
}

}  // namespace dgb
