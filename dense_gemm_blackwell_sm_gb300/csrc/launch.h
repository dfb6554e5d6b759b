// launch.h -- internal interface between the host planner (api.cu) and the
// kernel translation units.  Not part of the public C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dgb {

struct KParams;

// Everything needed to launch one kernel, fixed when a plan is made: the
// function, its launch shape and dynamic shared memory (whose attribute is set
// once, at plan time), and which argument list it takes.
enum ArgKind {
  ARGS_K = 0,      // (KParams)
  ARGS_AB_K = 1,   // (tmA, tmB, KParams)
  ARGS_ABC_K = 2,  // (tmA, tmB, tmC, KParams)
  ARGS_GEMV = 3,   // (GemvParams)
  ARGS_BX_TG = 4,  // (tmB, tmX, TgParams)
  ARGS_ABCSS_K = 5,  // (tmA, tmB, tmC, tmScaleA, tmScaleB, KParams)
};

struct LaunchSpec {
  const void* func = nullptr;
  dim3 grid{1, 1, 1};
  dim3 block{1, 1, 1};
  size_t smem = 0;
  unsigned cluster = 1;  // CTAs per cluster along x
  int kind = ARGS_K;
  bool pdl = false;      // launch as a programmatic dependent of the previous kernel
};

// one launch of a prepared kernel (cluster dimension attached when > 1)
cudaError_t launch_spec(const LaunchSpec& s, void** args, cudaStream_t st);
// raise (never lower) a kernel's dynamic shared-memory limit to `bytes`
cudaError_t allow_dynamic_smem(const void* func, size_t bytes);

// steps 1-3 (thread copies), 4-5 (TMA ring), 6 (persistent + scheduler)
cudaError_t spec_step123(int M, int N, bool out_f32, LaunchSpec* out);
cudaError_t spec_step45(int M, int N, int stages, bool out_f32, LaunchSpec* out);
cudaError_t spec_step6(int sched, int stages, bool out_f32, int grid, LaunchSpec* out);
size_t step6_smem_bytes(int stages);

// steps 7-9: warp-specialised persistent kernels
//   cg = 1 (one CTA per 128x256 tile) or 2 (CTA pair, cta_group::2)
//   consumers = 1 or 2 (second MMA consumer, step 9)
//   sched: 0 static stride, 1 atomic counter, 2 cluster launch control, 3 stream-K
struct WsShape {
  int cg;
  int consumers;
  int tile_m;       // rows of one (cluster) tile
  int tile_n;       // columns of one tile
  int a_box_rows;   // rows of one A TMA box
  int b_box_rows;   // rows of one B TMA box
  int stage_bytes;  // per CTA
  int threads;
};
// bn: tile columns, 256, or 224 for step 9 (cg 2, 2 consumers) with the static
// schedule and the plain writeback
WsShape ws_shape(int cg, int consumers, int bn = 256);
size_t ws_smem_bytes(int cg, int consumers, int stages, int bn = 256);
int ws_max_stages(int cg, int consumers, int bn = 256);
int ws_max_active_clusters(int cg, int consumers, int sched, bool out_f32, int stages, int bn = 256);
// stream-K (sched 3): fp32 floats of one cluster's workspace slot; one flag per
// writeback warp, cg * consumers * 4 per slot
size_t ws_sk_slot_floats(int cg, int consumers);
// fused_act >= 0: the writeback applies bias / activation fused_act / residual
// (one MMA consumer, static scheduler); -1: plain writeback
cudaError_t spec_ws(int cg, int consumers, int sched, bool out_f32, int stages, int clusters, LaunchSpec* out,
                    int fused_act = -1, int bn = 256);
// step 7 (cg 1) or step 8 (cg 2, CTA pairs) with each tile's K split into `split`
// slices (split * cg <= 8 CTAs per cluster), the partials exchanged over
// distributed shared memory (2 slices) or through KParams::sk_ws (one 128 KB slot
// per CTA); grid = tiles x split x cg
cudaError_t spec_ws_ks(int cg, bool out_f32, int stages, int tiles, int split, LaunchSpec* out);

// steps 7-9 with MX block scales (8-bit inputs, UE8M0 scale per 32 K
// elements): cg = 1 (one CTA per 128x256 tile) or 2 (CTA pair, 256x256), one
// consumer and a single TMEM accumulator; or cg = 2 with two consumers (step 9:
// 512x224 tiles, bf16 C, plain writeback, static schedule)
size_t mx_smem_bytes(int cg, int stages, int consumers = 1);
int mx_max_stages(int cg, int consumers = 1);
cudaError_t spec_mx(int cg, int sched, bool out_f32, int stages, int clusters, LaunchSpec* out,
                    int fused_act = -1, int consumers = 1);

// decode GEMV, C (M x N) = X (M x K) * B^T for M <= 16, on CUDA cores
struct GemvParams {
  const void* X;
  const void* B;
  void* Y;
  int32_t M, N, K;
  int32_t early_b;  // 1: B may be read before the previous kernel on the stream has completed
  int32_t pf_rows;  // groups of each warp's weight stream prefetched into L2 before waiting for
                    // the previous kernel (the rolling kernels, early_b == 0)
};
size_t gemv_smem_bytes(int M, int K);
// static_b: B is not written by the previous kernel on the stream (it may be
// read before that kernel completes); *pf_groups receives GemvParams::pf_rows
cudaError_t spec_gemv(int M, int N, int K, bool in_bf16, bool out_f32, int num_sms, bool static_b, LaunchSpec* out,
                      int* pf_groups);

// the same product on the Tensor Core (weight as the 128-row MMA operand),
// K split over the CTAs of a cluster
struct TgParams {
  const uint16_t* X;
  void* Y;
  int32_t M, N, K;
  int32_t kblocks_per_cta;  // K blocks in one CTA's slice
  int32_t split;            // CTAs per cluster along K
  int32_t stages;
  uint32_t idesc;
  uint32_t* status;
  uint64_t timeout_ns;
};
void gemv_tc_config(int N, int K, int num_sms, int want_split, int want_stages, int* split, int* stages,
                    int* kblocks_per_cta);
size_t gemv_tc_smem_bytes(int stages);
cudaError_t spec_gemv_tc(int M, int N, int K, bool in_bf16, bool out_f32, int num_sms, int want_split,
                         int want_stages, LaunchSpec* out, TgParams* base);

}  // namespace dgb
