// launch.h -- internal interface between the host planner (api.cu) and the
// kernel translation units.  Not part of the public C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dgb {

struct KParams;

// steps 1-3 (thread copies), 4-5 (TMA ring), 6 (persistent + scheduler)
cudaError_t launch_step123(const KParams& p, bool out_f32, cudaStream_t st);
cudaError_t launch_step45(const KParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                          bool out_f32, cudaStream_t st);
cudaError_t launch_step6(const KParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         bool out_f32, int sched, int grid, cudaStream_t st);
size_t step6_smem_bytes(int stages);

// steps 7-9: warp-specialised persistent kernels
//   cg = 1 (one CTA per 128x256 tile) or 2 (CTA pair, cta_group::2)
//   consumers = 1 or 2 (second MMA consumer, step 9)
//   sched: 0 static stride, 1 atomic counter, 2 cluster launch control
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
WsShape ws_shape(int cg, int consumers);
size_t ws_smem_bytes(int cg, int consumers, int stages);
int ws_max_stages(int cg, int consumers);
cudaError_t launch_ws(int cg, int consumers, int sched, const KParams& p, const CUtensorMap& tmA,
                      const CUtensorMap& tmB, const CUtensorMap& tmC, bool out_f32, int clusters,
                      cudaStream_t st);
int ws_max_active_clusters(int cg, int consumers, int sched, bool out_f32, int stages);

// decode GEMV, C (M x N) = X (M x K) * B^T for M <= 16
struct GemvParams {
  const void* X;
  const void* B;
  void* Y;
  int32_t M, N, K;
};
size_t gemv_smem_bytes(int M, int K);
// the same product on the Tensor Core (weight as the 128-row MMA operand),
// K split over the CTAs of a cluster
void gemv_tc_config(int N, int K, int num_sms, int* split, int* stages, int* kblocks_per_cta);
size_t gemv_tc_smem_bytes(int N, int K, int num_sms);
cudaError_t launch_gemv_tc(const GemvParams& g, const CUtensorMap& tmB, bool in_bf16, bool out_f32,
                           int num_sms, uint32_t* status, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_gemv(const GemvParams& g, bool in_bf16, bool out_f32, int num_sms, cudaStream_t st);

}  // namespace dgb
