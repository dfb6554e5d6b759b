/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library, libdgbgemm.so.
 *
 * Computes C = A * B^T on one GPU:
 *   A  M x K, row-major (K-major), fp16, bf16, or 8-bit float (E4M3 / E5M2,
 *      optionally with MX block scales)
 *   B  N x K, row-major (K-major), same type as A
 *   C  M x N, row-major (leading dimension N), fp32 or bf16
 * with fp32 accumulation in Tensor Memory.  This is the tiled GEMM of
 * "Modern GPU Programming for MLSys" (reading notes, section "9 步优化"),
 * whose nine steps are exposed as kernel variants below, and the decode-stage
 * vector-matrix product of section "Roofline：找到天花板" (1 x 4096 x 4096,
 * bandwidth-bound) served by a GEMV path for M <= 16.
 *
 * Every argument is a plain integer or pointer; no C++ or framework type
 * crosses this boundary and no exception escapes it.  Device pointers are
 * owned by the caller; the library never allocates, frees or retains user
 * buffers.  A plan owns host state (cached TMA descriptors) and 256 bytes of
 * device scratch (a status word and scheduler counters), plus, for the
 * stream-K schedule, a workspace of one fp32 tile per cluster (about 38 MB on
 * 76 CTA pairs with 512 x 256 tiles), or for a K split over a cluster of 3-8
 * CTAs one fp32 128 x 256 partial per CTA (19 MB at most for an automatic split
 * on 152 SMs),
 * all released by gemm_plan_destroy.  Two launches of one plan must not
 * overlap on the device.
 *
 * Errors: argument problems are returned at once and nothing is launched.
 * Kernels never trap: every wait inside them is bounded in time, and a wait
 * that runs out records a code in the plan's device status word and ends the
 * kernel early, leaving C undefined.  gemm_check() synchronises the stream and
 * reports such a code as GEMM_ERR_DEVICE_TIMEOUT.
 */
#ifndef DGB_GEMM_H
#define DGB_GEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* gemm_stream_t;

/* Input / output element types: A and B share the input type. */
typedef enum {
  GEMM_F16_F32 = 0,   /* fp16 in, fp32 out */
  GEMM_F16_BF16 = 1,  /* fp16 in, bf16 out (round to nearest even) */
  GEMM_BF16_F32 = 2,  /* bf16 in, fp32 out */
  GEMM_BF16_BF16 = 3, /* bf16 in, bf16 out (round to nearest even) */
  GEMM_E4M3_F32 = 4,  /* 8-bit float E4M3 (OCP FP8) in, fp32 out; variants 7-9, K-major */
  GEMM_E4M3_BF16 = 5, /* E4M3 in, bf16 out */
  GEMM_E5M2_F32 = 6,  /* 8-bit float E5M2 in, fp32 out */
  GEMM_E5M2_BF16 = 7, /* E5M2 in, bf16 out */
  /* MX block-scaled 8-bit inputs (OCP Microscaling formats MXFP8): every 32
   * consecutive K elements of a row of A or B share one UE8M0 scale 2^(e-127);
   * run with gemm_plan_run_mx, which takes the two scale arrays.  Variants 7
   * and 8 (one MMA consumer; the automatic plan picks the one whose tiles
   * finish first, see gemm_auto_variant), and on request (opts.variant = 9,
   * bf16 C, static schedule) variant 9's two consumers on 512 x 224 cluster
   * tiles; other variants give GEMM_ERR_UNSUPPORTED_SHAPE. */
  GEMM_MXE4M3_F32 = 8,  /* MXFP8 E4M3 in, fp32 out */
  GEMM_MXE4M3_BF16 = 9, /* MXFP8 E4M3 in, bf16 out */
  GEMM_MXE5M2_F32 = 10, /* MXFP8 E5M2 in, fp32 out */
  GEMM_MXE5M2_BF16 = 11 /* MXFP8 E5M2 in, bf16 out */
} gemm_dtype_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1,       /* NULL pointer, dimension < 1 or >= 2^31, bad option */
  GEMM_ERR_UNSUPPORTED_SHAPE = 2, /* K * sizeof(input) % 16 != 0, or a shape the requested variant cannot do */
  GEMM_ERR_MISALIGNED = 3,        /* A, B or C not 16-byte aligned */
  GEMM_ERR_UNSUPPORTED_DTYPE = 4, /* dtype outside gemm_dtype_t */
  GEMM_ERR_ARCH = 5,              /* current device is not compute capability 10.3 */
  GEMM_ERR_CUDA = 6,              /* a CUDA runtime/driver call failed */
  GEMM_ERR_OOM = 7,               /* plan scratch could not be allocated */
  GEMM_ERR_DEVICE_TIMEOUT = 8,    /* a bounded device-side wait gave up */
  GEMM_ERR_NO_DEVICE = 9          /* no CUDA device is visible */
} gemm_status_t;

/* Kernel variants: the nine steps of "9 步优化" plus the GEMV. */
typedef enum {
  GEMM_VARIANT_AUTO = 0,
  GEMM_VARIANT_S1_SINGLE_TILE = 1,   /* step 1: one CTA, one 128x128 tile; needs M,N <= 128, K <= 64 */
  GEMM_VARIANT_S2_KLOOP = 2,         /* step 2: + K loop into one TMEM accumulator; M,N <= 128 */
  GEMM_VARIANT_S3_MULTI_CTA = 3,     /* step 3: + 2-D grid of 128x128 tiles */
  GEMM_VARIANT_S4_TMA = 4,           /* step 4: + TMA loads tracked by an mbarrier */
  GEMM_VARIANT_S5_PIPELINE = 5,      /* step 5: + multi-stage SMEM ring (opts.stages, default 2) */
  GEMM_VARIANT_S6_PERSISTENT = 6,    /* step 6: + persistent CTAs and a tile scheduler */
  GEMM_VARIANT_S7_WARP_SPECIALIZED = 7, /* step 7: producer / MMA / writeback warps, 128x256 tiles */
  GEMM_VARIANT_S8_CTA_PAIR = 8,      /* step 8: 2-CTA cluster, cta_group::2 MMA, 256x256 tiles */
  GEMM_VARIANT_S9_TWO_CONSUMERS = 9, /* step 9: + second MMA consumer, 512x256 cluster tiles */
  GEMM_VARIANT_GEMV = 10,            /* decode GEMV (CUDA cores), M <= 16 */
  GEMM_VARIANT_GEMV_TC = 11          /* decode GEMV on the Tensor Core (weight as the 128-row
                                        MMA operand, K split over a cluster), M <= 16 */
} gemm_variant_t;

/* Tile schedulers of the persistent variants (6-9). */
typedef enum {
  GEMM_SCHED_AUTO = 0,
  GEMM_SCHED_STATIC = 1, /* fixed stride over the raster order */
  GEMM_SCHED_ATOMIC = 2, /* global atomic tile counter */
  GEMM_SCHED_CLC = 3,    /* hardware cluster launch control (work stealing) */
  GEMM_SCHED_STREAM_K = 4 /* variants 7-9: every cluster takes an equal share of the (tile, K
                             block) iterations; a tile split between two clusters is finished
                             by the one holding its first K blocks, from the other's fp32
                             partial in a plan-owned workspace.  The automatic plan uses it
                             where a fitted cost model says it finishes sooner than whole
                             tiles: those keep the clusters busy for under 80 % of the waves
                             (70 % on variant 9), K has at least 32 K blocks (64 on variant
                             9), and every cluster gets at least a tile's work.  Fused
                             epilogues and MX plans use whole tiles. */
} gemm_sched_t;

/* Tuning and test options; zero-initialise and set what you need.
 * A NULL options pointer means all-automatic. */
typedef struct {
  int32_t variant;      /* gemm_variant_t, 0 = automatic choice */
  int32_t sched;        /* gemm_sched_t, 0 = automatic (static) */
  int32_t stages;       /* SMEM ring depth, 0 = automatic (at most 12) */
  int32_t raster_group; /* tile rows per L2 raster group, 0 = automatic */
  int32_t max_ctas;     /* cap on persistent CTAs / clusters, 0 = no cap */
  int32_t split_k;      /* GEMV_TC: CTAs (a cluster) sharing one 128-row block's K range,
                           1, 2, 4 or 8.  Variant 7: CTAs (a cluster, 2-8) sharing one
                           128 x 256 tile's K range; variant 8: CTA pairs (2-4 slices,
                           clusters of 4-8 CTAs) sharing one 256 x 256 tile's.  The fp32
                           partials of two slices are exchanged over distributed shared
                           memory, of 3-8 through a plan workspace of 128 KB per CTA (a
                           split needing over 512 MB gives GEMM_ERR_UNSUPPORTED_SHAPE).
                           1 = never; 0 = automatic: when step 7's tiles would fill at
                           most half the SMs, the K range is split into as many slices
                           as the SMs hold with every cluster resident at once, at most
                           4, each keeping at least 16 K blocks, on step 8's pairs
                           unless they would occupy fewer SMs than step 7's CTAs */
  int64_t timeout_ns;   /* bound on every device-side wait, 0 = 2 s */
  int32_t debug_flags;  /* test hooks: 1 = leave out one TMA load (forces a timeout) */
  int32_t flags;        /* GEMM_FLAG_* */
  int32_t layout;       /* GEMM_LAYOUT_* bits; 0 = both operands K-major */
  int32_t reserved[5];
} gemm_opts_t;

/* Operand storage (variants 7-9).  C = A * B^T always; by default A is M x K and
 * B is N x K row-major (K-major).  GEMM_LAYOUT_A_MN: A is stored K x M row-major
 * (M-major, needs M % 8 == 0); GEMM_LAYOUT_B_MN: B is stored K x N row-major
 * (N-major, needs N % 8 == 0).  The reading notes name k-major and mn-major as
 * the two element orders a tile can have (section "三个核心概念", layout). */
#define GEMM_LAYOUT_A_MN 1
#define GEMM_LAYOUT_B_MN 2

/* B is not written by the work queued before the call on the same stream
 * (weights of a decode step).  The GEMV variants then start streaming B while
 * the previous kernel still runs and read A (the activations) only after it has
 * completed.  (Variants 7-9 and the CUDA-core GEMV always launch as programmatic
 * dependents of the previous kernel, but without the flag they wait for it to
 * complete before any access to global memory.) */
#define GEMM_FLAG_STATIC_B 1

typedef struct gemm_plan_s* gemm_plan_t;

/* What a plan chose. */
typedef struct {
  int32_t variant, sched, stages, raster_group;
  int32_t tile_m, tile_n;  /* output tile of one CTA (or CTA pair / cluster) */
  int32_t cluster;         /* CTAs per cluster: 1, or 2 for a CTA pair (variants 8-9); with a
                              K split over a cluster, slices x CTAs per tile (2-8); the
                              CUDA-core GEMV for 3 <= M <= 8 takes 2 when its 16-row
                              clusters fit one wave */
  int32_t consumers;       /* MMA consumers per CTA */
  int32_t grid;            /* CTAs launched */
  int32_t smem_bytes;      /* dynamic shared memory per CTA */
  int32_t num_sms;
  int32_t tiles;           /* output tiles (cluster tiles for variants 8-9) */
  int32_t narrow_tile_n;   /* variant 9 with tile_n 224: 0, or the width (208) of the tile
                              columns after the first wide_cols, chosen when the two widths
                              add up to N and even out the CTA pairs' work */
  int32_t wide_cols;
} gemm_plan_info_t;

/* The kernel variant the automatic plan (opts.variant = 0, K-major operands)
 * takes for these sizes and types on a GPU with num_sms SMs, without a device:
 * the decode GEMVs for M <= 16, the plain-store persistent kernel when C's rows
 * are not 16-byte aligned, step 7 with its K split over a cluster for outputs
 * whose 128 x 256 tiles fill at most half the SMs (and K has at least 32 blocks),
 * otherwise step 9, 8 or 7, whichever a cost model (waves of resident clusters x
 * a tile's area per SM / the step's per-SM rate, or the stream-K schedule's even
 * shares plus its partial sums where it applies) says finishes soonest; below 32
 * K blocks, a fit of launch ramp and per-wave times with whole tiles.  The tile
 * width, schedule and split are settled by gemm_plan with the device's
 * occupancy.  Errors: GEMM_ERR_INVALID_ARG (null variant, sizes out of range,
 * num_sms < 2), GEMM_ERR_UNSUPPORTED_DTYPE, GEMM_ERR_UNSUPPORTED_SHAPE (K's row
 * pitch); *variant is 0 then. */
GEMM_API gemm_status_t gemm_auto_variant(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                         int32_t num_sms, int32_t* variant);

/* Build a plan for C = A * B^T of the given sizes and types on the current
 * device.  Validates sizes (M, N, K >= 1 and < 2^31; K % 8 == 0), the dtype,
 * the options and the device (compute capability 10.3), picks the kernel
 * variant, tile, ring depth, raster and launch size, and allocates the plan's
 * device scratch.  On success *out receives the plan. */
GEMM_API gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                        const gemm_opts_t* opts, gemm_plan_t* out);

/* Launch the plan's kernel on `stream` (asynchronous).  A, B and C are device
 * pointers, 16-byte aligned, laid out as described at the top of this file;
 * C must not overlap A or B.  One plan runs on one stream at a time. */
GEMM_API gemm_status_t gemm_plan_run(gemm_plan_t plan, const void* A, const void* B, void* C,
                            gemm_stream_t stream);

/* Activations of the fused epilogue.  The reading notes list the nonlinear
 * nodes that follow a linear layer in an LLM's DAG (softmax, layer norm, GeLU /
 * SiLU); the formulas are the standard definitions. */
typedef enum {
  GEMM_ACT_NONE = 0,
  GEMM_ACT_RELU = 1,      /* max(x, 0) */
  GEMM_ACT_SILU = 2,      /* x / (1 + exp(-x)) */
  GEMM_ACT_GELU_TANH = 3, /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
  /* SiLU and the tanh form of GeLU are evaluated as x * logistic(t) with the
   * hardware's approximate exp2 and reciprocal: within 2^-20 |x| of the exact
   * value, well inside a bf16 or fp32 rounding of results of that size */
  GEMM_ACT_GELU_ERF = 4   /* 0.5 x (1 + erf(x / sqrt(2))) */
} gemm_activation_t;

/* Fused epilogue of the writeback:
 *   C[i][j] = act(scale_a[i] * scale_b[j] * sum_k A[i][k] B[j][k] + bias[j]) + residual[i][j],
 * computed in fp32 and rounded once to C's type (absent terms are skipped). */
typedef struct {
  const float* bias;    /* N fp32 values (device, 4-byte aligned), or NULL */
  const void* residual; /* M x N device array of C's type, row-major, 16-byte aligned, or
                           NULL; may be C itself (each element is read before it is
                           overwritten) */
  int32_t activation;   /* gemm_activation_t */
  int32_t reserved[3];
  const float* scale_a; /* M fp32 values multiplying row i of the product before the bias
                           (dequantisation of 8-bit inputs), or NULL */
  const float* scale_b; /* N fp32 values multiplying column j, or NULL */
} gemm_epilogue_t;

/* gemm_plan_run with the fused epilogue.  Needs a plan of variant 7, 8 or 9
 * (the automatic plan of most shapes with M > 16); other plans return
 * GEMM_ERR_UNSUPPORTED_SHAPE.  The epilogue kernel uses the static scheduler
 * and 256-column tiles; a variant-9 plan keeps its two consumers for bf16 C,
 * and for fp32 C with bias / residual / scales alone (an fp32 activation runs
 * on variant 8's 256 x 256 tile). */
GEMM_API gemm_status_t gemm_plan_run_epilogue(gemm_plan_t plan, const void* A, const void* B, void* C,
                                              const gemm_epilogue_t* epilogue, gemm_stream_t stream);

/* Block-scaled product of a plan made with an MX dtype (GEMM_MXE4M3_* or
 * GEMM_MXE5M2_*), the low-precision GEMM named among the kernels that decide
 * MLSys speed ("Modern GPU Programming for MLSys", background section):
 *
 *   C[i][j] = epi( sum_k (X_A[i][k/32] * A[i][k]) * (X_B[j][k/32] * B[j][k]) )
 *
 * with X = 2^(e - 127) for the UE8M0 byte e (255 is NaN), accumulated in fp32
 * in Tensor Memory by tcgen05.mma kind::mxf8f6f4.  A, B and C as for
 * gemm_plan_run (K-major 8-bit operands, K * 1 % 16 == 0).
 *
 * scale_a / scale_b are device arrays of UE8M0 bytes for A's M rows and B's N
 * rows, 16-byte aligned, each in the tiled layout: 512-byte blocks of 128 rows
 * x 4 scales (128 K elements), block (rb, cb) at byte (rb * ceil(K/128) + cb) *
 * 512, and inside a block the scale of row r, scale column c at byte
 * (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4.  Each array holds
 * gemm_mx_scale_bytes(rows, K) bytes; bytes of padding rows and of scale
 * columns past ceil(K/32) are never used.
 *
 * epilogue may be NULL (plain rounding to C's type) or a fused epilogue as for
 * gemm_plan_run_epilogue.  Plans of other dtypes return GEMM_ERR_UNSUPPORTED_DTYPE;
 * gemm_plan_run / gemm_run on an MX plan or dtype return GEMM_ERR_INVALID_ARG. */
GEMM_API gemm_status_t gemm_plan_run_mx(gemm_plan_t plan, const void* A, const void* B, void* C,
                                        const void* scale_a, const void* scale_b,
                                        const gemm_epilogue_t* epilogue, gemm_stream_t stream);

/* Bytes of one tiled MX scale array for `rows` rows and inner dimension K:
 * ceil(rows/128) * ceil(K/128) * 512; -1 for rows < 1 or K < 1. */
GEMM_API int64_t gemm_mx_scale_bytes(int64_t rows, int64_t K);

/* One-shot form: plan (cached per shape, dtype and device) and run.  A cached
 * plan keeps its device scratch, and any stream-K or split-K workspace (at most
 * about 38 MB), until gemm_clear_cache; launches through one cached plan on
 * different streams must not overlap. */
GEMM_API gemm_status_t gemm_run(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                       gemm_dtype_t dtype, gemm_stream_t stream);

/* End-to-end form with HOST operands: copies A_host and B_host into the
 * caller's device buffers dA and dB, runs the GEMM into dC and copies dC back
 * into C_host, then returns with everything complete and the device status
 * checked.  The work starts after what `stream` holds at the call; internally
 * B is copied first (in two column halves when C is the larger transfer) and
 * A, the GEMM and C go in up to 8 row panels on the library's own per-device
 * copy and compute streams, so the copies of later panels and the return of
 * earlier blocks of C overlap the GEMMs (host-to-device and device-to-host
 * copies run concurrently).  Calls are serialised per process.  Host buffers
 * should be pinned for full copy speed. */
GEMM_API gemm_status_t gemm_run_host(int64_t M, int64_t N, int64_t K, const void* A_host,
                            const void* B_host, void* C_host, gemm_dtype_t dtype, void* dA,
                            void* dB, void* dC, gemm_stream_t stream);

/* C = A * B^T like gemm_run, for callers that must not allocate memory while
 * they compute: code running inside an allocator hook or an out-of-memory
 * handler, while a memory pool is locked or being torn down, in a callback
 * that must not re-enter the CUDA allocator, or in an embedder whose device
 * memory is all pre-assigned.  The reading notes have no counterpart of this
 * entry point; it exists for those callers only.
 *
 * It makes no plan and calls no cudaMalloc, cudaFree or other allocating
 * routine: it runs the warp-specialised kernel of variants 7-9 with the atomic
 * tile scheduler, whose scratch (a status word and two counters, 12 bytes,
 * whatever the shape) lives in a fixed 256-byte device array inside the
 * library that every GPU loading the library keeps until the process exits.
 * The first call on a device, with that device current, looks up the array's
 * device address and loads the six kernels this entry point can launch (three
 * tiles, two output types) and sets their shared-memory limits, so any lazy
 * code loading by the driver happens then and never in a later call.  That
 * first call may therefore let the driver reserve memory for code: make it
 * once per device outside any no-allocation region (or run the process with
 * CUDA_MODULE_LOADING=EAGER), and before any stream capture.  If it fails
 * (GEMM_ERR_CUDA), nothing is kept and the next call tries again.  Every call
 * shares the array and clears it on `stream` before its kernel starts, so calls
 * that overlap on the GPU (different streams, or different threads) race and
 * must be serialised by the caller.  Needs N * sizeof(C element) % 16 == 0
 * besides the usual preconditions, and 16-bit inputs (dtypes 0-3; the 8-bit
 * ones return GEMM_ERR_UNSUPPORTED_DTYPE).  Asynchronous on `stream`; a
 * device-side wait that times out leaves C undefined and is not reported by
 * this entry point. */
GEMM_API gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                                        void* C, gemm_dtype_t dtype, gemm_stream_t stream);

/* Synchronise `stream`, then report (and clear) a device-side error recorded
 * by the plan's kernels.  plan == NULL checks every plan gemm_run cached. */
GEMM_API gemm_status_t gemm_check(gemm_plan_t plan, gemm_stream_t stream);

/* Fill *info with the plan's choices. */
GEMM_API gemm_status_t gemm_plan_info(gemm_plan_t plan, gemm_plan_info_t* info);

/* Test hook: when `visits` (a device int32 array with one entry per tile) is
 * non-NULL, persistent variants add 1 to visits[tile] for every tile written. */
GEMM_API gemm_status_t gemm_plan_set_visits(gemm_plan_t plan, int32_t* visits);

/* Release the plan's device scratch and host state.  NULL is ignored. */
GEMM_API void gemm_plan_destroy(gemm_plan_t plan);

/* Drop every plan cached by gemm_run (and gemm_run_host), releasing their device
 * memory; no launch through them may still be running. */
GEMM_API void gemm_clear_cache(void);

/* Static description of a status code. */
GEMM_API const char* gemm_status_string(gemm_status_t status);

/* Library version string. */
GEMM_API const char* gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DGB_GEMM_H */
