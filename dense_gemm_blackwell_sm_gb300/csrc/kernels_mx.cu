// kernels_mx.cu -- instantiations of the step-7 kernel (one CTA, 128x256 tile)
// and the step-8 kernel (CTA pair, 256x256 tile), one MMA consumer each, and of
// the step-9 kernel (CTA pair, two consumers, 512x224 tile, bf16 C, plain
// writeback, static schedule), for 8-bit float inputs with MX block scales (a
// UE8M0 scale per 32 consecutive K elements of every row of A and B,
// tcgen05.mma kind::mxf8f6f4); the kernel itself is in kernels_ws.cuh.
#include "kernels_ws.cuh"

namespace dgb {

namespace {

template <typename OutT, int CG>
void* pick_mx(int sched, int fused_act) {
  switch (fused_act) {
    case EPI_ACT_NONE: return mx_kernel_ptr<OutT, CG, SCHED_STATIC, EPI_ACT_NONE>();
    case EPI_ACT_RELU: return mx_kernel_ptr<OutT, CG, SCHED_STATIC, EPI_ACT_RELU>();
    case EPI_ACT_SILU: return mx_kernel_ptr<OutT, CG, SCHED_STATIC, EPI_ACT_SILU>();
    case EPI_ACT_GELU_TANH: return mx_kernel_ptr<OutT, CG, SCHED_STATIC, EPI_ACT_GELU_TANH>();
    case EPI_ACT_GELU_ERF: return mx_kernel_ptr<OutT, CG, SCHED_STATIC, EPI_ACT_GELU_ERF>();
    default: break;
  }
  if (sched == SCHED_ATOMIC) return mx_kernel_ptr<OutT, CG, SCHED_ATOMIC>();
  if (sched == SCHED_CLC) return mx_kernel_ptr<OutT, CG, SCHED_CLC>();
  return mx_kernel_ptr<OutT, CG, SCHED_STATIC>();
}

void* mx_kernel(int cg, int consumers, int sched, bool out_f32, int fused_act) {
  if (consumers == 2) {
    if (cg != 2 || out_f32 || fused_act >= 0 || sched != SCHED_STATIC) return nullptr;
    return mx_kernel_ptr<__nv_bfloat16, 2, SCHED_STATIC, -1, 2, 224>();
  }
  if (cg == 1) return out_f32 ? pick_mx<float, 1>(sched, fused_act) : pick_mx<__nv_bfloat16, 1>(sched, fused_act);
  if (cg == 2) return out_f32 ? pick_mx<float, 2>(sched, fused_act) : pick_mx<__nv_bfloat16, 2>(sched, fused_act);
  return nullptr;
}

}  // namespace

size_t mx_smem_bytes(int cg, int stages, int consumers) {
  const size_t stage = (consumers == 2) ? WsCfg<2, 2, 224>::STAGE + WsCfg<2, 2, 224>::MX_BYTES
                       : (cg == 1)      ? WsCfg<1, 1>::STAGE + WsCfg<1, 1>::MX_BYTES
                                        : WsCfg<2, 1>::STAGE + WsCfg<2, 1>::MX_BYTES;
  return 1024 + (size_t)stages * stage + WS_STAGING / 2 + WS_CTRL;
}

int mx_max_stages(int cg, int consumers) {
  // two consumers: TMEM holds their 224-column accumulators (448 columns) and
  // one 16-column scale slot per stage
  int s = (consumers == 2) ? 4 : WS_MAX_STAGES;
  while (s > 1 && mx_smem_bytes(cg, s, consumers) > WS_SMEM_LIMIT) --s;
  return s;
}

cudaError_t spec_mx(int cg, int sched, bool out_f32, int stages, int clusters, LaunchSpec* out, int fused_act,
                    int consumers) {
  void* k = mx_kernel(cg, consumers, sched, out_f32, fused_act);
  if (!k || stages < 1 || stages > mx_max_stages(cg, consumers)) return cudaErrorInvalidValue;
  const size_t smem = mx_smem_bytes(cg, stages, consumers);
  cudaError_t e = allow_dynamic_smem((const void*)k, smem);
  if (e != cudaSuccess) return e;
  out->func = k;
  out->grid = dim3((unsigned)(clusters * cg), 1, 1);
  out->block = dim3((unsigned)mx_threads(consumers), 1, 1);
  out->smem = smem;
  out->cluster = (unsigned)cg;
  out->kind = ARGS_ABCSS_K;
  return cudaSuccess;
}

}  // namespace dgb
