// noalloc.cu -- gemm_run_noalloc: C = A * B^T without any memory allocation.
//
// Some callers cannot allocate device memory at the moment they need a GEMM:
// code that runs while a memory pool is locked or being torn down, allocator
// hooks and out-of-memory handlers, callbacks that must not re-enter the CUDA
// allocator, or embedders whose memory is all pre-assigned.  For them this
// entry point runs the warp-specialised kernel (the step 7-9 family) with its
// atomic tile scheduler, whose scratch -- a status word, the tile counter and
// a finished-cluster counter -- lives in a fixed array in this file instead of
// in memory that gemm_plan would allocate.  No plan object is made: the launch
// state and the TMA descriptors live on the stack of the call.
//
// The array has a fixed size (NOALLOC_SCRATCH_BYTES) and every GPU that loads
// the library keeps it until the process exits.  Device code could name it
// directly, but host code must not: on the host its name is only a stand-in,
// not a device address.  So the first call on each device, with that device
// current, asks the runtime for the array's device address
// (cudaGetSymbolAddress) and keeps it.  The same first call also resolves the
// six kernels this entry point can launch (three tiles, two output types) and
// sets their shared-memory limits, so that any code loading the driver does
// lazily happens then and never on a later call.  That first call may
// therefore let the driver reserve memory for code: make it once per device
// outside any no-allocation region (or run with CUDA_MODULE_LOADING=EAGER),
// and before any stream capture.  A first call that fails is not remembered:
// the next call tries the set-up again.
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "gemm.h"
#include "idesc.h"
#include "kernel_common.cuh"
#include "launch.h"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 256;
constexpr int kMaxDevices = 64;

// status word, tile counter, finished-cluster counter (3 of the 64 words used)
constexpr size_t NOALLOC_SCRATCH_USED = 3 * sizeof(uint32_t);
static_assert(NOALLOC_SCRATCH_USED <= NOALLOC_SCRATCH_BYTES, "the scheduler's scratch must fit the fixed array");
static __device__ __align__(256) uint32_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES / sizeof(uint32_t)];

struct DeviceSetup {
  std::mutex mu;
  std::atomic<bool> done{false};  // set only once the set-up has succeeded
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
  bool arch_ok = false;
  int clusters[3][2] = {};  // active clusters per (variant 7/8/9, out fp32?)
};

DeviceSetup g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 2-D row-major [outer][inner] tensor, 128-byte swizzled boxes, zero fill
bool encode(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, uint64_t inner, uint64_t outer,
            uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (uint64_t)esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return f(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (variant 7 / 8 / 9) -> (CTAs per cluster, MMA consumers)
constexpr int kCg[3] = {1, 2, 2};
constexpr int kCons[3] = {1, 1, 2};

// once per device, with that device current; on failure nothing is kept and
// the next call tries again
cudaError_t setup_device(int dev, DeviceSetup& d) {
  int major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  d.sms = sms;
  d.arch_ok = (major == 10 && minor == 3);
  if (!d.arch_ok) return cudaSuccess;
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  // resolve every kernel this entry point launches now (loading its code and
  // setting its shared-memory limit), not on the first call that needs it
  for (int vi = 0; vi < 3; ++vi)
    for (int of = 0; of < 2; ++of) {
      const int stages = dgb::ws_max_stages(kCg[vi], kCons[vi]);
      int n = dgb::ws_max_active_clusters(kCg[vi], kCons[vi], /*atomic scheduler*/ 1, of != 0, stages);
      if (n < 1) return cudaErrorInvalidConfiguration;
      d.clusters[vi][of] = n;
    }
  d.scratch = ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" GEMM_API gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                                                   void* C, gemm_dtype_t dtype, gemm_stream_t stream) {
  using namespace dgb;
  if ((int)dtype < 0 || (int)dtype > 3) return GEMM_ERR_UNSUPPORTED_DTYPE;
  if (M < 1 || N < 1 || K < 1 || M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31))
    return GEMM_ERR_INVALID_ARG;
  if (K % 8 != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;
  const bool out_f32 = (dtype == GEMM_F16_F32 || dtype == GEMM_BF16_F32);
  const bool in_bf16 = (dtype == GEMM_BF16_F32 || dtype == GEMM_BF16_BF16);
  // rows of C must start 16-byte aligned for the TMA stores of this kernel
  if ((N * (out_f32 ? 4 : 2)) % 16 != 0) return GEMM_ERR_UNSUPPORTED_SHAPE;
  if (!A || !B || !C) return GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15u)
    return GEMM_ERR_MISALIGNED;

  int n = 0, dev = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
  DeviceSetup& d = g_dev[dev];
  if (!d.done.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(d.mu);
    if (!d.done.load(std::memory_order_relaxed)) {
      if (setup_device(dev, d) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
      }
      d.done.store(true, std::memory_order_release);
    }
  }
  if (!d.arch_ok) return GEMM_ERR_ARCH;

  // tile: the largest cluster tile that still gives every CTA pair a tile
  const int64_t tn = (N + 255) / 256;
  const int64_t pairs = std::max(1, d.sms / 2);
  int cg = 1, cons = 1;
  if (((M + 511) / 512) * tn >= pairs) {
    cg = 2;
    cons = 2;
  } else if (((M + 255) / 256) * tn >= pairs) {
    cg = 2;
  }
  const WsShape sh = ws_shape(cg, cons);
  const int stages = ws_max_stages(cg, cons);
  const int vi = (cg == 1) ? 0 : (cons == 1 ? 1 : 2);
  const int active = d.clusters[vi][out_f32 ? 1 : 0];

  KParams k{};
  k.M = (int32_t)M;
  k.N = (int32_t)N;
  k.K = (int32_t)K;
  k.tiles_m = (int32_t)((M + sh.tile_m - 1) / sh.tile_m);
  k.tiles_n = (int32_t)tn;
  k.raster_group = std::min(8, k.tiles_m);
  k.stages = stages;
  k.status = static_cast<uint32_t*>(d.scratch);
  k.visits = nullptr;
  k.timeout_ns = 2000000000ull;
  k.debug_flags = 0;
  k.out_ld = (int32_t)N;
  k.A = static_cast<const uint16_t*>(A);
  k.B = static_cast<const uint16_t*>(B);
  k.C = C;
  k.idesc = idesc_f16(in_bf16, 128 * cg, 256);

  CUtensorMap tmA, tmB, tmC;
  const CUtensorMapDataType in_t = in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const bool ok = encode(&tmA, in_t, 2, A, (uint64_t)K, (uint64_t)M, 64, (uint32_t)sh.a_box_rows) &&
                  encode(&tmB, in_t, 2, B, (uint64_t)K, (uint64_t)N, 64, (uint32_t)sh.b_box_rows) &&
                  (out_f32 ? encode(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, (uint64_t)N, (uint64_t)M, 32, 32)
                           : encode(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, (uint64_t)N, (uint64_t)M, 64, 32));
  if (!ok) return GEMM_ERR_CUDA;

  const int tiles = k.tiles_m * k.tiles_n;
  LaunchSpec spec;
  if (spec_ws(cg, cons, /*atomic scheduler*/ 1, out_f32, stages, std::min(tiles, active), &spec) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the status word and both
  // counters must start at zero
  if (cudaMemsetAsync(d.scratch, 0, NOALLOC_SCRATCH_USED, s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  void* args[] = {&tmA, &tmB, &tmC, &k};
  if (launch_spec(spec, args, s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}
