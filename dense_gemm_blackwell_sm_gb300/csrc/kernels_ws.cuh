// kernels_ws.cuh -- steps 7-9 of the tiled GEMM, C = A * B^T: persistent,
// warp-specialised kernels with TMEM double buffering, CTA pairs and a
// second MMA consumer.
//
// "Modern GPU Programming for MLSys" (reading notes, section "9 步优化",
// third stage) adds, on top of the persistent TMA pipeline of step 6:
//
//   step 7  warp specialisation: a producer warp (TMA), an MMA warp and
//           writeback warps hand tiles to each other through mbarriers, so
//           loads, MMAs and stores overlap continuously;
//   step 8  a 2-CTA cluster computes one 256x256 tile: the pair MMA
//           (cta_group::2) reads both CTAs' shared memory, the accumulator
//           spans both CTAs' TMEM, and each loaded byte feeds about twice the
//           work;
//   step 9  a second MMA consumer per CTA: both consumers share the B stage,
//           each owns half of the output rows, so the cluster tile grows to
//           512x256 with no extra B traffic per stage.
//
// Roles (256 threads):
//   warp 0      producer: one lane issues the TMA loads into a `stages`-deep ring
//   warp 1      MMA consumer 0 (one lane issues tcgen05.mma); owns TMEM alloc
//   warp 2      tile scheduler: static stride, a global atomic counter, or
//               hardware cluster launch control; publishes tile ids to a ring
//   warp 3      MMA consumer 1 (step 9 only)
//   warps 4-7   writeback: tcgen05.ld -> fp32 or bf16 -> 128B-swizzled SMEM
//               staging -> TMA tile stores (vectorised and coalesced by TMA)
//
// TMEM holds two 256-column fp32 accumulators.  Steps 7 and 8 alternate them
// between consecutive tiles (the writeback of tile i overlaps the MMAs of
// tile i+1); step 9 gives one to each consumer, so its writeback first drains
// the accumulator into registers (bf16 C: packed; fp32 C on 224-column tiles:
// two chunks staged, five held) and hands it back before the stores.
//
// All of steps 7-9 launch as programmatic dependents of the previous kernel on
// the stream: the set-up below overlaps that kernel's end, and every thread
// waits for it to complete before its first access to global memory.
//
// MX block scaling (k_ws_mx: one consumer, one CTA or a CTA pair): each stage
// also brings the UE8M0 scales of its 128 K-elements (one 512-byte block for
// the CTA's 128 rows of A, two for the tile's 256 rows of B) into shared memory
// with TMA copies of 128 x 4-byte boxes, and tcgen05.cp moves them into TMEM
// ahead of the block-scaled MMAs.  On the CTA pair, warp 3 (idle with one
// consumer) issues those copies and signals each stage's on a barrier, so the
// MMA thread only issues MMAs: that single thread's issue rate bounds the pair
// kernel, and three copies per stage on it cost about a tenth of the
// throughput.  The one-CTA kernel, whose 4-stage ring leaves less time to hide
// the extra hand-off, issues the copies from the MMA thread itself.  In a pair each CTA holds
// the scales of its own A rows and of all the tile's B rows, and its copies
// complete on the leader's barrier like its operand copies.  The scales take
// TMEM columns 256 and up, so the tile keeps a single accumulator, and the
// writeback stages through one 4 KB buffer per warp instead of two to leave
// shared memory for the scale blocks.
//
// Stream-K (SK template flag, static schedule, plain writeback): instead of
// whole tiles, every cluster takes an equal, contiguous share of the flattened
// (tile, K block) iterations, so the last wave no longer leaves clusters idle
// (80 tiles on 76 CTA pairs are two waves of whole tiles; a 1024^2 output in
// 128 x 256 tiles keeps 32 of 152 SMs busy).  A tile is split between
// consecutive clusters: every cluster but the first whose share covers part of
// it computes that part as its FIRST segment ("head" part, K blocks from the
// middle of the tile on) and writes the fp32 partial to its workspace slot,
// with one flag per writeback warp; the cluster holding the tile's first K
// blocks does them as its LAST segment ("owner" part), waits (bounded) for the
// flags of all the following clusters whose shares start inside the tile, adds
// their partials and stores the tile.  No cluster waits on one that has not
// started, the owner clears the flags it consumed, and a slot holds each
// writeback warp's 32-column chunks in the layout of sk_add32, so both sides
// move whole 4 KB runs with 512 contiguous bytes per warp access.
//
// Split-K within a cluster (KS template parameter, step 7's 128x256 tile or step
// 8's 256x256 pair tile, plain writeback): for outputs with too few tiles for the
// GPU, a cluster of 2-8 CTAs (2-4 pairs) shares one tile, CTA (pair) r
// accumulating K blocks [KB r / s, KB (r+1) / s) in its own TMEM; in a pair each
// CTA exchanges partials with the CTAs of the same pair half.  Every CTA puts its fp32 partial where the others can read it (its
// idle stage ring for a cluster of two; otherwise, except the columns it owns,
// its slot of the plan's workspace in L2) in the writeback warps' (warp, chunk,
// lane) order and arrives on the barrier of every CTA of the cluster; then each
// CTA adds all the partials of its share of the tile's columns and stores that
// share.  The cluster synchronises once more before any CTA exits, so no shared
// memory is read after its owner has gone.
//
// In a CTA pair, each CTA loads its own 128 rows of A and its own 128 rows of B
// (the pair MMA splits A along M and B along N) with the cta_group::2 TMA form,
// whose completion is counted on the leader CTA's barrier; only the leader
// issues MMAs, and its commits arrive on the barriers of both CTAs.  No load is
// multicast.  Every wait is bounded (see ptx.cuh).
#pragma once
#include "idesc.h"
#include "kernel_common.cuh"
#include "launch.h"

namespace dgb {

namespace {

enum SchedWs { SCHED_STATIC = 0, SCHED_ATOMIC = 1, SCHED_CLC = 2, SCHED_STREAM_K = 3 };

constexpr int WS_THREADS = 256;
// step 9's fused-epilogue kernels have four writeback warps per consumer, so that both
// accumulators get their epilogue at the same time: 12 warps
__host__ __device__ constexpr int ws_threads(int ncons, int epi) { return (ncons == 2 && epi >= 0) ? 384 : WS_THREADS; }
constexpr int WS_BN = 256;          // tile columns (MMA N)
constexpr uint32_t WS_A_BYTES = 128u * 128u;  // 128 rows x 128 B
constexpr int WS_RING = 4;          // depth of the tile-id ring
constexpr int WS_STAGING = 4 * 2 * 4096;      // 4 writeback warps x 2 buffers x 32 rows x 128 B
constexpr int WS_CTRL = 512;        // barriers and small state
constexpr int WS_MAX_STAGES = 8;
constexpr size_t WS_SMEM_LIMIT = 232448;  // 227 KB per CTA
constexpr int SK_WARP_FLOATS = (WS_BN / 32) * 32 * 32;  // one writeback warp's 32 x 256 fp32 part
constexpr uint32_t MX_BLOCK = 512;  // scales of 128 rows x 128 K-elements (4 per row)
constexpr uint32_t MX_TMEM_COL = 256;  // first TMEM column of the per-stage scale slots
constexpr uint32_t MX_TMEM_SLOT = 16;  // TMEM columns per stage: 4 for A, 8 for B (step 9: 4 + 4 + 8)
// threads of the MX kernels: 8 warps, and a ninth on step 9 (two consumers) that
// regroups the B scales and copies every scale block into TMEM
__host__ __device__ constexpr int mx_threads(int consumers) { return consumers == 2 ? 288 : 256; }

// A warp's partial accumulator (32 rows x 256 columns, fp32) is kept as 8 chunks of
// 32 columns, each [j][lane][4 values]: lane L's values 4j..4j+3 of a chunk sit at
// float4 index j*32 + L, so each 16-byte access of the warp covers 512 contiguous
// bytes (coalesced in global memory, free of bank conflicts in shared memory)
constexpr int SK_CHUNK_FLOATS = 32 * 32;

// Programmatic dependent launch: let the next kernel on the stream begin its own
// set-up, and wait until the previous one has completed and its memory is visible
// (both are no-ops for a launch that did not ask for it)
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The K blocks of a cluster's i-th tile run backwards when i is odd.  A wave of
// tiles streams its A and B panels through L2 from the first K block to the
// last; the next wave, started at the last K block, first asks for the blocks
// the previous wave loaded most recently, which are the ones still in L2.  The
// order of the K blocks changes only the fp32 summation order.  Stream-K and
// split-K segments keep the forward order.
template <bool PARTIAL_K>
__device__ __forceinline__ bool k_reversed(uint32_t i) {
  return !PARTIAL_K && (i & 1u) != 0u;
}

// v[j] += the lane's 32 values of one partial chunk, for fp32 values held as bit patterns
__device__ __forceinline__ void sk_add32(uint32_t (&v)[32], const float* chunk, uint32_t lane) {
  const float4* s4 = reinterpret_cast<const float4*>(chunk) + lane;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 a = s4[j * 32];
    v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + a.x);
    v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + a.y);
    v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + a.z);
    v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + a.w);
  }
}

// stores the lane's 32 values as one partial chunk in the layout sk_add32 reads
__device__ __forceinline__ void sk_store32(float* chunk, uint32_t lane, const uint32_t (&v)[32]) {
  float4* d4 = reinterpret_cast<float4*>(chunk) + lane;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    d4[j * 32] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                             __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
}

// BN: tile columns (MMA N), 256 or 224 (the narrower tile evens out the waves
// of shapes such as 4096^3, whose 512 x 256 tiles fill 1.68 waves of CTA pairs)
template <int CG, int NCONS, int BN = WS_BN>
struct WsCfg {
  static constexpr int B_ROWS = (CG == 1) ? BN : BN / 2;
  static constexpr uint32_t B_BYTES = (uint32_t)B_ROWS * 128u;
  static constexpr uint32_t STAGE = NCONS * WS_A_BYTES + B_BYTES;  // per CTA
  static constexpr int TILE_M = 128 * CG * NCONS;
  // arrivals that free one tile-ring slot: producer + 4 writeback warps in
  // every CTA of the cluster, plus the leader's MMA consumers
  static constexpr uint32_t RING_CONSUMERS = (uint32_t)(CG * 5 + NCONS);
  // MX scale blocks per stage and CTA: one for the CTA's 128 rows of A, two for
  // the tile's 256 rows of B; on step 9 (224-column tiles) two for A (one per
  // consumer), the three 128-row blocks of B holding the tile's 224 rows as
  // loaded, and the two blocks they are regrouped into
  static constexpr uint32_t MX_BYTES = MX_BLOCK * (NCONS == 2 ? 7u : 3u);
};

// The kernel body.  EPI < 0: plain writeback; EPI >= 0: fused epilogue with
// activation EPI.  MX: 8-bit inputs with UE8M0 block scales read through
// tmSA / tmSB (one consumer only).  The tensor maps are kernel parameters of
// the entry points below.  KS: K split over a cluster, the partials exchanged
// over distributed shared memory (1, a cluster of two) or through L2 (2).
template <typename OutT, int CG, int NCONS, int SCHED, int EPI, bool MX, bool SK = false, int BN = WS_BN,
          int KS = 0>
__device__ __forceinline__ void ws_body(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmC,
                                        const CUtensorMap* tmSA, const CUtensorMap* tmSB, const KParams& p) {
  using Cfg = WsCfg<CG, NCONS, BN>;
  // MX on step 9: two consumers on the CTA pair's 512 x 224 tile
  constexpr bool MX9 = MX && NCONS == 2;
  static_assert(!MX9 || (CG == 2 && BN == 224 && EPI < 0 && sizeof(OutT) == 2 && !SK && !KS),
                "MX with two consumers: CTA pair, 224-column tiles, plain bf16 writeback");
  static_assert(BN == WS_BN || ((!MX || MX9) && !SK && EPI < 0), "narrow tiles: plain writeback, whole tiles");
  static_assert(!KS || (NCONS == 1 && !MX && !SK && EPI < 0 && BN == WS_BN),
                "split-K clusters: step 7 or step 8 tile, plain writeback");
  static_assert(!SK || (!MX && EPI < 0 && SCHED == SCHED_STATIC), "stream-K: plain writeback, static schedule");
  // MX on the pair: a separate warp copies the scales and takes tile ids from the ring
  // (warp 3 of the leader with one consumer).  On step 9 warp 8 of both CTAs
  // regroups the B scales and also reads the ring, and one thread (warp 1 of the
  // leader) issues both consumers' MMAs, each stage's scale copies first.
  constexpr bool MX_COPIER = MX && CG == 2 && !MX9;
  constexpr uint32_t MMA_THREADS = MX9 ? 1u : (uint32_t)NCONS;  // MMA-issuing threads
  // step 9 with a fused epilogue: eight writeback warps, four per consumer (see below)
  constexpr bool WB8 = EPI >= 0 && NCONS == 2 && CG == 2 && !MX && !SK && !KS && BN == WS_BN;
  static_assert(ws_threads(NCONS, EPI) == (WB8 ? 384 : WS_THREADS) || MX, "thread count of the fused step-9 kernels");
  constexpr uint32_t RING_CONS = Cfg::RING_CONSUMERS - (uint32_t)NCONS + MMA_THREADS + (MX_COPIER ? 1u : 0u) +
                                 (MX9 ? (uint32_t)CG : 0u) + (WB8 ? 4u * (uint32_t)CG : 0u);
  // TMEM columns: consumer c's accumulator at c * 256; the per-stage scale slots
  // from MX_TMEM_COL, or on step 9 MX in the two 32-column gaps the 224-column
  // accumulators leave (columns 224-255 and 480-511, two 16-column slots each)
  auto sf_slot_col = [&](uint32_t st) -> uint32_t {
    if constexpr (MX9) {
      return (st < 2u ? (uint32_t)BN : 256u + (uint32_t)BN) + (st & 1u) * MX_TMEM_SLOT;
    } else {
      return MX_TMEM_COL + st * MX_TMEM_SLOT;
    }
  };
  constexpr uint32_t STAGING = MX ? WS_STAGING / 2 : WS_STAGING;
  constexpr uint32_t WARP_STAGING = STAGING / 4;
  constexpr int CW = (sizeof(OutT) == 4) ? 32 : 64;  // output columns per 128-byte staging row
  constexpr int NCH = BN / CW;      // whole 128-byte staging chunks of a row
  constexpr int TAIL = BN % CW;     // bf16 with BN = 224: 32 more columns, stored from registers
  // writeback that first drains a single accumulator into registers (see below)
  constexpr bool DRAIN = (MX || (NCONS == 2 && !SK)) && CW == 64 && EPI < 0;
  // the same for fp32 C on step 9's 224-column tile: two chunks into the staging
  // buffers, the other five into registers
  constexpr bool DRAIN32 = CG == 2 && NCONS == 2 && !SK && !MX && BN == 224 && CW == 32 && EPI < 0;
  // the 224-column kernel may run tiles of two widths (KParams wide_n / narrow_n)
  constexpr bool BAL = BN != WS_BN && !MX;
  auto tile_cols = [&](int32_t tn, int32_t& c0, int32_t& width) {
    if constexpr (BAL) {
      tile_columns(p, tn, BN, c0, width);
    } else {
      c0 = tn * BN;
      width = BN;
    }
  };
  // fused epilogue on step 9: each consumer's single accumulator is held while
  // the epilogue runs, so the rows are stored straight from registers (no wait
  // for a staging buffer inside that window), and the staging buffers hold the
  // tile's bias and scale_b columns instead
  constexpr bool EPI_DIRECT = WB8;
  static_assert(!EPI_DIRECT || WS_STAGING / 8 >= 2 * WS_BN * 4, "a warp's staging holds two column vectors");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  const int S = p.stages;
  uint8_t* ring = smem;
  uint8_t* staging = smem + (size_t)S * Cfg::STAGE;
  uint8_t* mx_ring = staging + STAGING;  // S x Cfg::MX_BYTES (MX only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(mx_ring + (MX ? (size_t)S * Cfg::MX_BYTES : 0));
  uint64_t* full = bars;                       // [8]  TMA -> MMA
  uint64_t* empty = bars + 8;                  // [8]  MMA -> TMA
  uint64_t* acc_full = bars + 16;              // [2]  MMA -> writeback
  uint64_t* acc_empty = bars + 18;             // [2]  writeback -> MMA
  uint64_t* ring_full = bars + 20;             // [4]  scheduler -> roles
  uint64_t* ring_empty = bars + 24;            // [4]  roles -> scheduler
  uint64_t* clc_bar = bars + 28;
  uint64_t* drain_bar = bars + 29;
  uint64_t* sf_ready = bars + 36;              // [8]  scale copies -> MMA (MX)
  uint64_t* cp_drain = bars + 44;              // scale-copy warp's last copies done (MX)
  uint64_t* red_full = bars + 45;              // split-K partials parked (every CTA of the cluster)
  uint64_t* sf_land = bars + 46;               // [8]  this CTA's B scale blocks landed (step 9 MX)
  uint64_t* sf_grouped = bars + 54;            // [8]  B scales regrouped in both CTAs (step 9 MX, leader)
  uint32_t* clc_resp = reinterpret_cast<uint32_t*>(bars + 30);   // 16 B, 16-aligned
  volatile int32_t* ring_tile = reinterpret_cast<volatile int32_t*>(clc_resp + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(clc_resp + 4 + WS_RING);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* zero_word = tmem_slot + 2;

  const uint32_t warp = warp_idx(), lane = lane_idx();
  // cluster rank; the CTA's half of its pair (ranks 2j and 2j + 1 form a pair); the
  // cluster rank of the pair's leader (the CTA itself without pairs), a compile-time
  // 0 where a cluster is one pair or one CTA (a run-time leader rank in the commit
  // masks and barrier addresses cost step 8 2 %)
  const uint32_t crank = (CG == 2 || KS != 0) ? cluster_ctarank() : 0u;
  const uint32_t rank = (CG == 2) ? (KS != 0 ? (crank & 1u) : crank) : 0u;
  const uint32_t lead = (KS != 0) ? (CG == 2 ? (crank & ~1u) : crank) : 0u;
  const bool leader = (rank == 0);
  // split-K: this CTA's (or pair's) slice of the tile's K blocks and the number of slices
  const int32_t ks_n = KS ? (int32_t)(cluster_nctarank() / (uint32_t)CG) : 1;
  const int32_t ks_r = KS ? (int32_t)(crank / (uint32_t)CG) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), MMA_THREADS);
      if constexpr (MX_COPIER) mbar_init(smem_u32(sf_ready + s), 1);
      if constexpr (MX9) {
        mbar_init(smem_u32(sf_land + s), 1);
        mbar_init(smem_u32(sf_grouped + s), CG);
      }
    }
    if constexpr (MX_COPIER) mbar_init(smem_u32(cp_drain), 1);
    if constexpr (KS != 0) mbar_init(smem_u32(red_full), 4u * (uint32_t)ks_n);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(acc_full + i), 1);
      mbar_init(smem_u32(acc_empty + i), 4 * CG);
    }
    for (int i = 0; i < WS_RING; ++i) {
      mbar_init(smem_u32(ring_full + i), 1);
      mbar_init(smem_u32(ring_empty + i), RING_CONS);
    }
    mbar_init(smem_u32(clc_bar), 1);
    mbar_init(smem_u32(drain_bar), MMA_THREADS);
    *abort_flag = 0u;
    *zero_word = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(tmA);
    tma_prefetch_desc(tmB);
    tma_prefetch_desc(tmC);
    if constexpr (MX) {
      tma_prefetch_desc(tmSA);
      tma_prefetch_desc(tmSB);
    }
  }
  if (warp == 1) {
    tmem_alloc<CG>(smem_u32(tmem_slot), 512);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (CG == 2 || KS != 0) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above touched only this CTA's (or cluster's) shared memory and TMEM;
  // from here on global memory is read and written
  grid_launch_dependents();
  grid_wait_prior();
  const uint32_t peer_abort = (CG == 2) ? mapa_shared(smem_u32((const void*)abort_flag), crank ^ 1u) : 0u;
  const WaitCtl w{abort_flag, p.status, p.timeout_ns, peer_abort};
  // K elements per stage: one 128-byte swizzle row of A / B (64 x 16-bit or 128 x 8-bit)
  const int32_t BKE = (p.bk > 0) ? p.bk : 64;
  const int32_t KB = (p.K + BKE - 1) / BKE;
  const bool f8 = (p.mma_kind == 1);
  const bool a_mn = (p.layout & LAYOUT_A_MN) != 0u;
  const bool b_mn = (p.layout & LAYOUT_B_MN) != 0u;

  // stream-K: this cluster's share [sk_b, sk_e) of the flattened (tile, K block)
  // iterations, walked as segments of one tile each
  const int64_t sk_total = (int64_t)p.tiles_m * p.tiles_n * KB;
  const int64_t sk_units = (int64_t)(gridDim.x / CG), sk_cid = (int64_t)(blockIdx.x / CG);
  const int64_t sk_b = sk_total * sk_cid / sk_units, sk_e = sk_total * (sk_cid + 1) / sk_units;
  auto sk_next = [&](int64_t& it, int32_t& tile, int32_t& kb0, int32_t& kb1) -> bool {
    if (it >= sk_e) return false;
    tile = (int32_t)(it / KB);
    kb0 = (int32_t)(it - (int64_t)tile * KB);
    kb1 = (int32_t)min((int64_t)KB, kb0 + (sk_e - it));
    it += kb1 - kb0;
    return true;
  };

  // one lane takes the next entry of the tile-id ring; -1 ends the stream
  auto ring_get = [&](uint32_t i, int32_t& tile) -> bool {
    const uint32_t slot = i % WS_RING, ph = (i / WS_RING) & 1u;
    if (!mbar_wait<CG == 2>(smem_u32(ring_full + slot), ph, w, WAIT_RING_FULL)) return false;
    tile = ring_tile[slot];
    if constexpr (CG == 1) {
      mbar_arrive(smem_u32(ring_empty + slot));
    } else {
      mbar_arrive_cluster(mapa_shared(smem_u32(ring_empty + slot), lead));
    }
    return true;
  };

  if (warp == 2 && !SK && !KS) {
    // ------------------------------------------------------------- scheduler
    if (lane == 0 && leader) {
      const int32_t total = p.tiles_m * p.tiles_n;
      const int32_t nclusters = (int32_t)(gridDim.x / CG);
      const int32_t cid = (int32_t)(blockIdx.x / CG);
      int32_t next_static = cid;
      uint32_t clc_phase = 0;
      bool first = true, exhausted = false, ok = true;
      for (uint32_t i = 0;; ++i) {
        const uint32_t slot = i % WS_RING, ph = (i / WS_RING) & 1u;
        if (!mbar_wait<CG == 2>(smem_u32(ring_empty + slot), ph ^ 1u, w, WAIT_RING_EMPTY)) { ok = false; break; }
        int32_t t = -1;
        if (!exhausted) {
          if (SCHED == SCHED_STATIC) {
            t = next_static;
            next_static += nclusters;
          } else if (SCHED == SCHED_ATOMIC) {
            t = (int32_t)atomicAdd(p.status + 1, 1u);
          } else if (first) {
            t = cid;
          } else {
            mbar_arrive_expect_tx(smem_u32(clc_bar), 16);
            clc_try_cancel(smem_u32(clc_resp), smem_u32(clc_bar));
            if (!mbar_wait(smem_u32(clc_bar), clc_phase, w, WAIT_CLC)) { ok = false; break; }
            clc_phase ^= 1u;
            uint32_t x;
            t = clc_decode(smem_u32(clc_resp), x) ? (int32_t)(x / CG) : -1;
          }
          first = false;
        }
        if (t >= total) t = -1;
        if (t < 0) exhausted = true;
        ring_tile[slot] = t;
        mbar_arrive(smem_u32(ring_full + slot));
        if constexpr (CG == 2) {
          st_cluster_u32(mapa_shared(smem_u32((const void*)(ring_tile + slot)), lead + 1u), (uint32_t)t);
          mbar_arrive_cluster(mapa_shared(smem_u32(ring_full + slot), lead + 1u));
        }
        if (t < 0) break;
      }
      if (SCHED == SCHED_ATOMIC && ok) {
        // the last cluster to run out of tiles rewinds the counters for the next launch
        __threadfence();
        if (atomicAdd(p.status + 2, 1u) == (uint32_t)(nclusters - 1)) {
          atomicExch(p.status + 1, 0u);
          atomicExch(p.status + 2, 0u);
        }
      }
    }
  } else if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, sphase = 0, issued = 0;
      bool skip = (p.debug_flags & DEBUG_SKIP_ONE_LOAD) != 0u;
      bool ok = true;
      int64_t sk_it = sk_b;
      for (uint32_t i = 0; ok; ++i) {
        int32_t tile, kb0 = 0, kb1 = KB;
        if constexpr (SK) {
          if (!sk_next(sk_it, tile, kb0, kb1)) break;
        } else if constexpr (KS != 0) {
          if (i > 0) break;  // one tile per cluster, this CTA's share of K
          tile = (int32_t)(blockIdx.x / (uint32_t)(ks_n * CG));
          kb0 = KB * ks_r / ks_n;
          kb1 = KB * (ks_r + 1) / ks_n;
        } else {
          if (!ring_get(i, tile)) { ok = false; break; }
          if (tile < 0) break;
        }
        int32_t tm, tn;
        raster_tile(tile, p.tiles_m, p.tiles_n, p.raster_group, tm, tn);
        const int32_t m_cta = tm * Cfg::TILE_M + (int32_t)rank * 128;
        int32_t tc0, tw;
        tile_cols(tn, tc0, tw);
        // the pair's second CTA holds the tile's second half of B rows
        const int32_t n_cta = tc0 + (CG == 2 ? (int32_t)rank * (tw / 2) : 0);
        const bool rev = k_reversed<SK || KS != 0>(i);
        for (int32_t it = 0; it < kb1 - kb0; ++it) {
          const int32_t kb = rev ? kb1 - 1 - it : kb0 + it;
          if (!mbar_wait(smem_u32(empty + stage), sphase ^ 1u, w, WAIT_PRODUCER_EMPTY)) { ok = false; break; }
          const uint32_t fb = smem_u32(full + stage);
          // MX: one block of A scales and one box holding the two blocks of B scales
          // (a block past the array's last row group arrives as zeros)
          const int32_t n_tile = tn * BN;
          // (step 9: the scales count on this CTA's own barrier instead)
          const uint32_t mx_tx = MX9 ? 0u : MX ? 3u * MX_BLOCK : 0u;
          if (leader) mbar_arrive_expect_tx(fb, (Cfg::STAGE + mx_tx) * CG);
          if constexpr (MX9) {
            // step 9 MX: the scales first, on this CTA's own barrier: A's 128-row
            // block of each consumer (rows m_cta and m_cta + 256) and the three
            // 128-row blocks of B from the one holding the tile's first row, so the
            // regrouping warp works on them while the operands are still landing
            uint8_t* sd = mx_ring + (size_t)stage * Cfg::MX_BYTES;
            const uint32_t lb = smem_u32(sf_land + stage);
            mbar_arrive_expect_tx(lb, 5u * MX_BLOCK);
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_2d(smem_u32(sd + c * MX_BLOCK), tmSA, lb, 0, 4 * (((m_cta + c * 256) / 128) * KB + kb));
            tma_load_4d(smem_u32(sd + 2 * MX_BLOCK), tmSB, lb, 0, 0, kb, n_tile / 128);
          }
          uint8_t* st = ring + (size_t)stage * Cfg::STAGE;
#pragma unroll
          for (int c = 0; c < NCONS; ++c) {
            const int32_t row = m_cta + c * 128 * CG;
            uint8_t* dst = st + c * WS_A_BYTES;
            if (a_mn) {
              // K x M in memory: two 64-row-of-K x 64-M boxes, 8 KB apart
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                if constexpr (CG == 1) {
                  tma_load_2d(smem_u32(dst + h * 8192), tmA, fb, row + 64 * h, kb * BKE);
                } else {
                  tma_load_2d_pair(smem_u32(dst + h * 8192), tmA, mapa_shared(fb, lead), row + 64 * h, kb * BKE);
                }
              }
            } else if constexpr (CG == 1) {
              tma_load_2d(smem_u32(dst), tmA, fb, kb * BKE, row);
            } else {
              tma_load_2d_pair(smem_u32(dst), tmA, mapa_shared(fb, lead), kb * BKE, row);
            }
          }
          uint8_t* bdst = st + NCONS * WS_A_BYTES;
          if (skip) {
            skip = false;  // test hook: this stage's B bytes never arrive
          } else if (b_mn) {
#pragma unroll
            for (int h = 0; h < Cfg::B_ROWS / 64; ++h) {
              if constexpr (CG == 1) {
                tma_load_2d(smem_u32(bdst + h * 8192), tmB, fb, n_cta + 64 * h, kb * BKE);
              } else {
                tma_load_2d_pair(smem_u32(bdst + h * 8192), tmB, mapa_shared(fb, lead), n_cta + 64 * h, kb * BKE);
              }
            }
          } else if constexpr (CG == 1) {
            tma_load_2d(smem_u32(bdst), tmB, fb, kb * BKE, n_cta);
          } else {
            tma_load_2d_pair(smem_u32(bdst), tmB, mapa_shared(fb, lead), kb * BKE, n_cta);
          }
          if constexpr (MX && !MX9) {
            // tiled scale layout: block (row block, K block) at ((row block) * KB + kb) * 512,
            // i.e. rows 4 * block .. 4 * block + 3 of A's 128-byte-wide map, and entry
            // (0, 0, kb, row block) of B's 4-D map (whose boxes span two row blocks).
            // Every extra copy on the pair costs throughput, hence the one B box.
            uint8_t* sd = mx_ring + (size_t)stage * Cfg::MX_BYTES;
            const int32_t ya = 4 * ((m_cta / 128) * KB + kb);
            if constexpr (CG == 1) {
              tma_load_2d(smem_u32(sd), tmSA, fb, 0, ya);
              tma_load_4d(smem_u32(sd + MX_BLOCK), tmSB, fb, 0, 0, kb, n_tile / 128);
            } else {
              tma_load_2d_pair(smem_u32(sd), tmSA, mapa_shared(fb, lead), 0, ya);
              tma_load_4d_pair(smem_u32(sd + MX_BLOCK), tmSB, mapa_shared(fb, lead), 0, 0, kb, n_tile / 128);
            }
          }
          ++issued;
          if (++stage == (uint32_t)S) { stage = 0; sphase ^= 1u; }
        }
      }
      if (!ok) {
        // Copies may still be in flight into this CTA's ring: they must land before
        // its shared memory is released.  Each issued stage's full barrier (in this
        // CTA, or in the leader of a pair) completes when its bytes have arrived, so
        // where this thread can see the barrier it waits for the last min(S, issued)
        // stages, each wait bounded (a stage whose load was never issued, as in the
        // missing-load test, gives up after the bound).  The other CTA of a pair
        // cannot wait on the leader's barriers; it waits the same bound in wall time,
        // far longer than a ring of at most 8 x 48 KB takes to land at the slowest
        // per-SM copy rate seen (about 40 GB/s: 10 us).
        volatile uint32_t never = 0u;  // a timeout here sets this flag only
        const WaitCtl wd{&never, nullptr, 2000000ull, 0};
        const uint32_t n = issued < (uint32_t)S ? issued : (uint32_t)S;
        if constexpr (MX9) {
          // the scale blocks land on this CTA's own barriers
          for (uint32_t back = 1; back <= n; ++back) {
            const uint32_t sb = (stage + (uint32_t)S - back) % (uint32_t)S;
            mbar_wait(smem_u32(sf_land + sb), back <= stage ? sphase : sphase ^ 1u, wd, 0u);
          }
        }
        if (CG == 1 || leader) {
          for (uint32_t back = 1; back <= n; ++back) {
            const uint32_t sb = (stage + (uint32_t)S - back) % (uint32_t)S;
            mbar_wait(smem_u32(full + sb), back <= stage ? sphase : sphase ^ 1u, wd, 0u);
          }
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < wd.timeout_ns) {}
        }
      }
    }
  } else if (MX9 && warp == 1 && leader) {
    // -------------------------------------------------- MMA (step 9 MX)
    // One thread issues the tcgen05.cp of each stage's scales into the stage's
    // TMEM slot and then both consumers' MMAs: the tensor pipe runs one thread's
    // tcgen05 operations in order, so no copy completion has to travel back
    // through an mbarrier before the MMAs may be issued.  A slot was last read
    // by MMAs this thread issued S stages earlier.
    if (lane == 0) {
      uint32_t g = 0;  // stages issued so far (ring position g % S, phase (g / S) & 1)
      bool ok = true;
      auto copy_stage = [&](uint32_t gg) {
        const uint32_t st = gg % (uint32_t)S;
        const uint32_t sft = tmem + sf_slot_col(st);
        const uint32_t sfs = smem_u32(mx_ring + (size_t)st * Cfg::MX_BYTES);
        tmem_cp_32x128b_x4<CG>(sft, sdesc_rows16(sfs));                      // consumer 0's A rows
        tmem_cp_32x128b_x4<CG>(sft + 4, sdesc_rows16(sfs + MX_BLOCK));       // consumer 1's A rows
        tmem_cp_32x128b_x4<CG>(sft + 8, sdesc_rows16(sfs + 5 * MX_BLOCK));   // B rows 0-127
        tmem_cp_32x128b_x4<CG>(sft + 12, sdesc_rows16(sfs + 6 * MX_BLOCK));  // B rows 128-223
      };
      for (uint32_t i = 0; ok; ++i) {
        int32_t tile;
        if (!ring_get(i, tile) || tile < 0) break;
        const uint32_t apar = i & 1u;
        for (int c = 0; c < 2 && ok; ++c)
          ok = mbar_wait<true>(smem_u32(acc_empty + c), apar ^ 1u, w, WAIT_MMA_ACC_EMPTY);
        if (!ok) break;
        tc_fence_after();
        const bool rev = k_reversed<false>(i);
        for (int32_t it = 0; it < KB; ++it, ++g) {
          const int32_t kb = rev ? KB - 1 - it : it;
          const uint32_t stage = g % (uint32_t)S, sphase = (g / (uint32_t)S) & 1u;
          const uint32_t acc0 = (it != 0) ? 1u : 0u;
          if (!mbar_wait(smem_u32(full + stage), sphase, w, WAIT_MMA_FULL)) { ok = false; break; }
          // the B scales regrouped in both CTAs
          if (!mbar_wait<true>(smem_u32(sf_grouped + stage), sphase, w, WAIT_MMA_FULL)) { ok = false; break; }
          tc_fence_after();
          copy_stage(g);
          const uint32_t sft = tmem + sf_slot_col(stage);
          const uint32_t sb = smem_u32(ring + (size_t)stage * Cfg::STAGE + NCONS * WS_A_BYTES);
          const uint64_t bd = sdesc_k_sw128(sb);
          const int32_t rem = p.K - kb * BKE;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint64_t ad = sdesc_k_sw128(smem_u32(ring + (size_t)stage * Cfg::STAGE + c * WS_A_BYTES));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k * 32 < rem)
                mma_mxf8f6f4<CG>(tmem + (uint32_t)c * 256u, ad + 2 * k, bd + 2 * k,
                                 p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29), sft + 4u * (uint32_t)c, sft + 8u,
                                 acc0 | (uint32_t)k);
          }
          mma_commit_pair(smem_u32(empty + stage), 3u << lead);
        }
        if (!ok) break;
        for (int c = 0; c < 2; ++c) mma_commit_pair(smem_u32(acc_full + c), 3u << lead);
      }
      // every MMA and copy this thread issued must be complete before TMEM is released
      mma_commit_cg<CG>(smem_u32(drain_bar));
      const WaitCtl wd{zero_word, p.status, p.timeout_ns, 0};
      mbar_wait(smem_u32(drain_bar), 0, wd, WAIT_DRAIN);
    }
  } else if ((warp == 1 || (NCONS == 2 && !MX9 && warp == 3)) && leader) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      const int cons = (warp == 1) ? 0 : 1;
      uint32_t stage = 0, sphase = 0;
      int64_t sk_it = sk_b;
      for (uint32_t i = 0;; ++i) {
        int32_t tile, kb0 = 0, kb1 = KB;
        if constexpr (SK) {
          if (!sk_next(sk_it, tile, kb0, kb1)) break;
        } else if constexpr (KS != 0) {
          if (i > 0) break;
          tile = (int32_t)(blockIdx.x / (uint32_t)(ks_n * CG));
          kb0 = KB * ks_r / ks_n;
          kb1 = KB * (ks_r + 1) / ks_n;
        } else {
          if (!ring_get(i, tile) || tile < 0) break;
        }
        const uint32_t slot = (NCONS == 2) ? (uint32_t)cons : MX ? 0u : (i & 1u);
        const uint32_t apar = (MX || NCONS == 2) ? (i & 1u) : ((i >> 1) & 1u);
        uint32_t idesc = p.idesc;
        if constexpr (BAL) {
          // this tile's width as the MMA's N
          int32_t tm, tn, tc0, tw;
          raster_tile(tile, p.tiles_m, p.tiles_n, p.raster_group, tm, tn);
          tile_cols(tn, tc0, tw);
          if (tw != BN) idesc = idesc_with_n(p.idesc, tw);
        }
        if (!mbar_wait<CG == 2>(smem_u32(acc_empty + slot), apar ^ 1u, w, WAIT_MMA_ACC_EMPTY)) break;
        tc_fence_after();
        const uint32_t d = tmem + slot * 256u;
        bool ok = true;
        const bool rev = k_reversed<SK || KS != 0>(i);
        for (int32_t it = 0; it < kb1 - kb0; ++it) {
          const int32_t kb = rev ? kb1 - 1 - it : kb0 + it;
          const uint32_t acc0 = (it != 0) ? 1u : 0u;  // the segment's first MMA overwrites D
          // MX pair: this stage's scales are in TMEM; the copy warp saw the stage land
          // before copying, so this one wait covers the operands too
          const uint32_t ready = MX_COPIER ? smem_u32(sf_ready + stage) : smem_u32(full + stage);
          if (!mbar_wait(ready, sphase, w, WAIT_MMA_FULL)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + (size_t)stage * Cfg::STAGE + cons * WS_A_BYTES);
          const uint32_t sb = smem_u32(ring + (size_t)stage * Cfg::STAGE + NCONS * WS_A_BYTES);
          // K-major: a K step of 16 moves 32 B inside the swizzle row; MN-major: two 1 KB atoms
          const uint64_t ad = a_mn ? sdesc_mn_sw128(sa, 8192) : sdesc_k_sw128(sa);
          const uint64_t bd = b_mn ? sdesc_mn_sw128(sb, 8192) : sdesc_k_sw128(sb);
          const uint64_t astep = a_mn ? 128 : 2, bstep = b_mn ? 128 : 2;
          // four MMAs per stage, each over 32 bytes of K (16 x 16-bit or 32 x 8-bit)
          if constexpr (MX) {
            if constexpr (!MX_COPIER) {
              // one CTA: the scales precede their MMAs in this thread's issue order
              const uint32_t sft0 = tmem + MX_TMEM_COL + stage * MX_TMEM_SLOT;
              const uint32_t sfs = smem_u32(mx_ring + (size_t)stage * Cfg::MX_BYTES);
              tmem_cp_32x128b_x4<CG>(sft0, sdesc_rows16(sfs));
              tmem_cp_32x128b_x4<CG>(sft0 + 4, sdesc_rows16(sfs + MX_BLOCK));
              tmem_cp_32x128b_x4<CG>(sft0 + 8, sdesc_rows16(sfs + 2 * MX_BLOCK));
            }
            const uint32_t sft = tmem + sf_slot_col(stage);
            const uint32_t sfa = sft, sfb = sft + 4u;  // A scales: 4 columns, then B's
            // byte k of each scale word belongs to the k-th 32-element K block; blocks
            // wholly past K are not issued (their scale bytes are padding)
            const int32_t rem = p.K - kb * BKE;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k * 32 < rem)
                mma_mxf8f6f4<CG>(d, ad + 2 * k, bd + 2 * k, p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29), sfa,
                                 sfb, acc0 | (uint32_t)k);
          } else if (f8) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8f6f4<CG>(d, ad + astep * k, bd + bstep * k, idesc, acc0 | (uint32_t)k);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f16<CG>(d, ad + astep * k, bd + bstep * k, idesc, acc0 | (uint32_t)k);
          }
          if constexpr (CG == 1) {
            mma_commit(smem_u32(empty + stage));
          } else {
            mma_commit_pair(smem_u32(empty + stage), 3u << lead);
          }
          if (++stage == (uint32_t)S) { stage = 0; sphase ^= 1u; }
        }
        if (!ok) break;
        if constexpr (CG == 1) {
          mma_commit(smem_u32(acc_full + slot));
        } else {
          mma_commit_pair(smem_u32(acc_full + slot), 3u << lead);
        }
      }
      // every MMA this thread issued must be complete before TMEM is released
      mma_commit_cg<CG>(smem_u32(drain_bar));
      const WaitCtl wd{zero_word, p.status, p.timeout_ns, 0};
      mbar_wait(smem_u32(drain_bar), 0, wd, WAIT_DRAIN);
    }
  } else if (MX_COPIER && warp == 3 && leader) {
    // --------------------------------------------------- scale copies (MX only)
    if (lane == 0) {
      uint32_t stage = 0, sphase = 0;
      bool ok = true;
      for (uint32_t i = 0; ok; ++i) {
        int32_t tile;
        if (!ring_get(i, tile) || tile < 0) break;
        for (int32_t kb = 0; kb < KB; ++kb) {
          // the stage's slot was last read by MMAs that completed before the stage was
          // refilled, so it is free once the stage has landed
          if (!mbar_wait(smem_u32(full + stage), sphase, w, WAIT_MMA_FULL)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sft = tmem + MX_TMEM_COL + stage * MX_TMEM_SLOT;
          const uint32_t sfs = smem_u32(mx_ring + (size_t)stage * Cfg::MX_BYTES);
          tmem_cp_32x128b_x4<CG>(sft, sdesc_rows16(sfs));           // A's 128 rows: 4 columns
          tmem_cp_32x128b_x4<CG>(sft + 4, sdesc_rows16(sfs + MX_BLOCK));      // B's 256 rows: 8
          tmem_cp_32x128b_x4<CG>(sft + 8, sdesc_rows16(sfs + 2 * MX_BLOCK));
          mma_commit_cg<CG>(smem_u32(sf_ready + stage));
          if (++stage == (uint32_t)S) { stage = 0; sphase ^= 1u; }
        }
      }
      // the copies this thread issued must be complete before TMEM is released
      mma_commit_cg<CG>(smem_u32(cp_drain));
      const WaitCtl wd{zero_word, p.status, p.timeout_ns, 0};
      mbar_wait(smem_u32(cp_drain), 0, wd, WAIT_DRAIN);
    }
  } else if (MX9 && warp == 8) {
    // ------------------------------------------- B scale regrouping (step 9 MX)
    // The tile's 224 B rows start at a multiple of 32 but not of 128, so their
    // scales, loaded as the three 128-row blocks that hold them, are regrouped into
    // the two blocks of 128 rows the MMA reads: in the tiled layout a block holds
    // 32 rows of 16 bytes, word j of row l being the four K scales of matrix row
    // 32 j + l, so 32-row group G of the tile (global group 7 tn + G) moves from
    // word (7 tn + G) % 4 of loaded block (7 tn + G) / 4 - (7 tn) / 4 to word G % 4
    // of block G / 4; lane l moves row l of every group, and group 7 (rows 224-255,
    // outside the tile) is zeroed.  Both CTAs regroup their own copy (the copies
    // into TMEM read each CTA's shared memory) and arrive on the leader's barrier,
    // which the MMA thread waits on before it copies the stage's scales.
    uint32_t stage = 0, sphase = 0;
    bool ok = true;
    for (uint32_t i = 0; ok; ++i) {
      int32_t tile = -1;
      uint32_t okr = 1;
      if (lane == 0) okr = ring_get(i, tile) ? 1u : 0u;
      okr = __shfl_sync(0xffffffffu, okr, 0);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (!okr || tile < 0) break;
      int32_t tm, tn;
      raster_tile(tile, p.tiles_m, p.tiles_n, p.raster_group, tm, tn);
      const int32_t g0 = tn * (BN / 32);  // the tile's first 32-row group of B
      for (int32_t kb = 0; kb < KB; ++kb) {
        uint32_t got = 1;
        if (lane == 0) got = mbar_wait(smem_u32(sf_land + stage), sphase, w, WAIT_MMA_FULL) ? 1u : 0u;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        uint8_t* sd = mx_ring + (size_t)stage * Cfg::MX_BYTES;
        const uint8_t* loaded = sd + 2 * MX_BLOCK;
        uint8_t* grouped = sd + 5 * MX_BLOCK;
#pragma unroll
        for (int32_t G = 0; G < 8; ++G) {
          uint32_t v = 0u;
          if (G < BN / 32) {
            const int32_t gg = g0 + G;
            v = *reinterpret_cast<const uint32_t*>(loaded + ((gg >> 2) - (g0 >> 2)) * MX_BLOCK + lane * 16u +
                                                   (uint32_t)(gg & 3) * 4u);
          }
          *reinterpret_cast<uint32_t*>(grouped + (G >> 2) * MX_BLOCK + lane * 16u + (uint32_t)(G & 3) * 4u) = v;
        }
        // the regrouped blocks are read by tcgen05.cp (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (leader) {
            mbar_arrive(smem_u32(sf_grouped + stage));
          } else {
            mbar_arrive_cluster(mapa_shared(smem_u32(sf_grouped + stage), lead));
          }
        }
        if (++stage == (uint32_t)S) { stage = 0; sphase ^= 1u; }
      }
    }
  } else if (warp >= 4 && warp < (WB8 ? 12u : 8u)) {
    // ------------------------------------------------------------ writeback
    const uint32_t q = warp & 3u;  // TMEM lane quarter this warp may access
    // step 9 with a fused epilogue: warps 4-7 serve consumer 0 and warps 8-11
    // consumer 1, each with a quarter of the staging space of its own
    const int my_cons = WB8 ? (int)((warp - 4u) >> 2) : -1;
    uint8_t* my_staging = WB8 ? staging + (warp - 4u) * (STAGING / 8u) : staging + q * WARP_STAGING;
    uint32_t tog = 0;
    int64_t sk_it = sk_b;
    for (uint32_t i = 0;; ++i) {
      int32_t tile = -1, kb0 = 0, kb1 = KB;
      if constexpr (SK) {
        if (!sk_next(sk_it, tile, kb0, kb1)) break;
      } else if constexpr (KS != 0) {
        if (i > 0) break;
        tile = (int32_t)(blockIdx.x / (uint32_t)(ks_n * CG));
      } else {
        uint32_t okr = 1;
        if (lane == 0) okr = ring_get(i, tile) ? 1u : 0u;
        okr = __shfl_sync(0xffffffffu, okr, 0);
        tile = __shfl_sync(0xffffffffu, tile, 0);
        if (!okr || tile < 0) break;
      }
      int32_t tm, tn;
      raster_tile(tile, p.tiles_m, p.tiles_n, p.raster_group, tm, tn);
      bool ok = true;
      float* epi_cols = reinterpret_cast<float*>(my_staging);  // EPI_DIRECT: bias, then scale_b
      if constexpr (EPI_DIRECT) {
        __syncwarp();  // every lane is done with the previous tile's columns
        if (p.bias != nullptr) stage_columns<BN>(epi_cols, p.bias, tn * BN, p.N, lane);
        if (p.scale_b != nullptr) stage_columns<BN>(epi_cols + BN, p.scale_b, tn * BN, p.N, lane);
        __syncwarp();
      }
#pragma unroll 1
      for (int cons = 0; cons < NCONS; ++cons) {
        if (WB8 && cons != my_cons) continue;
        const uint32_t slot = (NCONS == 2) ? (uint32_t)cons : MX ? 0u : (i & 1u);
        const uint32_t apar = (MX || NCONS == 2) ? (i & 1u) : ((i >> 1) & 1u);
        const int32_t row0 = tm * Cfg::TILE_M + cons * 128 * CG + (int32_t)rank * 128 + (int32_t)q * 32;
        int32_t col_base, tile_w;
        tile_cols(tn, col_base, tile_w);
        // fused epilogue: while the MMAs still run, read the first chunk of the
        // lane's residual row segment and scale_a, and have L2 fetch the rest of
        // the segment, so the held accumulator waits on no DRAM round trip
        uint32_t res_next[EPI >= 0 ? 32 : 1];
        float epi_sa = 1.f;
        bool epi_res = false;
        // 32-byte row accesses when C's and the residual's rows allow them (32-byte
        // aligned and N a multiple of 16 columns, so a 32-byte group lies wholly
        // inside C or outside)
        const bool v8_rows = EPI_DIRECT && (p.N % 16 == 0) &&
                             (((reinterpret_cast<uintptr_t>(p.C) | reinterpret_cast<uintptr_t>(p.residual) |
                                (uintptr_t)((int64_t)p.out_ld * (int64_t)sizeof(OutT))) & 31u) == 0);
        if constexpr (EPI >= 0) {
          const int32_t row = row0 + (int32_t)lane;
          epi_res = p.residual != nullptr && row < p.M;
          if (epi_res) {
            if constexpr (EPI_DIRECT) {
              load_residual_cols32<OutT>(res_next, p, row, col_base, v8_rows);
            } else {
              load_residual128<OutT>(res_next, p, row, col_base, v8_rows);
            }
            const uint8_t* seg = reinterpret_cast<const uint8_t*>(reinterpret_cast<const OutT*>(p.residual) +
                                                                  (int64_t)row * p.out_ld + col_base);
            const int32_t seg_bytes = min(BN, p.N - col_base) * (int32_t)sizeof(OutT);
#pragma unroll 1
            // with evict_last priority, so that less of it is gone again when the epilogue
            // runs (8192^3 bias + SiLU + residual: DRAM reads 1019 -> 930 MB per launch,
            // 1840 -> 1847 TFLOP/s)
            for (int32_t b = 128; b < seg_bytes + 127; b += 128)
              asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(seg + min(b, seg_bytes - 1)));
          }
          if (p.scale_a != nullptr) epi_sa = (row < p.M) ? __ldg(p.scale_a + row) : 0.f;
        }
        uint32_t got = 1;
        if (lane == 0) got = mbar_wait(smem_u32(acc_full + slot), apar, w, WAIT_EPI_ACC_FULL) ? 1u : 0u;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        tc_fence_after();
        const uint32_t tbase = tmem + ((q * 32u) << 16) + slot * 256u;
        if constexpr (EPI_DIRECT) {
          // 32 columns per step: the TMEM load, the epilogue (the residual read one
          // step ahead; bias and scale_b from the warp's staging copy) and the row's
          // 64 or 128 bytes stored from registers; the accumulator goes back as soon
          // as the last step's columns are in registers
          constexpr int RW = 32 * (int)sizeof(OutT) / 4;  // words of 32 columns
          constexpr int per16 = 16 / (int)sizeof(OutT);
          const int32_t row = row0 + (int32_t)lane;
#pragma unroll 1
          for (int s32 = 0; s32 < BN / 32; ++s32) {
            uint32_t res[RW];
#pragma unroll
            for (int j = 0; j < RW; ++j) res[j] = res_next[j];
            if (epi_res && s32 + 1 < BN / 32) load_residual_cols32<OutT>(res_next, p, row, col_base + (s32 + 1) * 32, v8_rows);
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + (uint32_t)(s32 * 32), v);
            tmem_wait_ld();
            if (s32 == BN / 32 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty + slot), lead));
            }
            const int32_t col0 = col_base + s32 * 32;
            apply_epilogue32<OutT, EPI>(v, p, col0, epi_sa, epi_res, res, epi_cols + s32 * 32, epi_cols + BN + s32 * 32);
            if (row < p.M) {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<OutT*>(p.C) + (int64_t)row * p.out_ld + col0);
              uint32_t o[RW];  // the row's 32 columns in C's type
#pragma unroll
              for (int j = 0; j < RW; ++j) o[j] = (sizeof(OutT) == 4) ? v[j] : pack_bf16x2(v[2 * j], v[2 * j + 1]);
              if (v8_rows) {
#pragma unroll
                for (int j = 0; j < RW / 8; ++j)
                  if (col0 + 2 * per16 * j < p.N) st_global_v8(dst + 2 * j, o + 8 * j);
              } else {
#pragma unroll
                for (int j = 0; j < RW / 4; ++j)
                  if (col0 + per16 * j < p.N) dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
              }
            }
          }
          continue;
        }
        // stream-K: this warp's 32 x 256 part of a split tile, in a workspace slot of
        // SK_WARP_FLOATS floats (8 chunks of 32 columns, see sk_add32); the owner adds
        // sk_nparts partials from consecutive slots
        const float* sk_part = nullptr;
        int32_t sk_nparts = 0;
        constexpr int64_t SK_SLOT_STRIDE = (int64_t)CG * NCONS * 4;  // flags / warp slots per cluster
        if constexpr (SK) {
          const int64_t own = ((sk_cid * CG + rank) * NCONS + cons) * 4 + q;
          if (kb0 > 0) {
            // head part (the tile's last K blocks): publish it for the previous cluster
            float* dst = p.sk_ws + own * SK_WARP_FLOATS;
#pragma unroll 1
            for (int c32 = 0; c32 < WS_BN / 32; ++c32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tbase + (uint32_t)(c32 * 32), v);
              tmem_wait_ld();
              if (c32 == WS_BN / 32 - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                  if constexpr (CG == 1) {
                    mbar_arrive(smem_u32(acc_empty + slot));
                  } else {
                    mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty + slot), lead));
                  }
                }
              }
              sk_store32(dst + c32 * SK_CHUNK_FLOATS, lane, v);
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu_u32(p.sk_flags + own, 1u);
            continue;
          }
          if (kb1 < KB) {
            // owner part (the first K blocks): wait for the head parts of the following
            // clusters whose shares start inside this tile (empty shares write nothing)
            const int64_t tile_end = (int64_t)(tile + 1) * KB;
            uint32_t okf = 1;
            for (int64_t c2 = sk_cid + 1; c2 < sk_units && sk_total * c2 / sk_units < tile_end; ++c2) {
              if (sk_total * (c2 + 1) / sk_units == sk_total * c2 / sk_units) continue;
              ++sk_nparts;
              if (lane == 0 && okf)
                okf = wait_flag_gpu(p.sk_flags + own + (c2 - sk_cid) * SK_SLOT_STRIDE, w, WAIT_SK_PARTIAL) ? 1u : 0u;
            }
            okf = __shfl_sync(0xffffffffu, okf, 0);
            if (!okf) { ok = false; break; }
            sk_part = p.sk_ws + (own + SK_SLOT_STRIDE) * SK_WARP_FLOATS;
          }
        }
        if constexpr (KS != 0) {
          // a tile split over the cluster: slice r's CTA adds, in slice order, the ks_n
          // partials of its share of the tile's 32-column chunks (of its pair half) and
          // stores them.  The partials are kept as [warp quarter][32-column chunk] in the
          // chunk layout of sk_add32 (each 16-byte access of the warp covers 512
          // contiguous bytes), and every CTA arrives on the barriers of the CTAs it
          // exchanges with once its own are in place.  Distributed shared memory moves
          // only about 15 bytes per clock per SM, so two slices park their partials in
          // their (idle) stage rings and read each other's there (512 x 4096 x 4096 on
          // step 7: 775 TFLOP/s, 747 through L2), while more slices write the chunks the
          // others own to their slots of the plan's workspace in L2 and read them back
          // from there, each CTA's own chunks straight from TMEM (1024 x 1024 x 4096 on
          // four CTAs: 541 TFLOP/s, 520 over distributed shared memory)
          constexpr bool via_l2 = KS == 2;
          const int32_t cb = (WS_BN / 32) * ks_r / ks_n, ce = (WS_BN / 32) * (ks_r + 1) / ks_n;
          const int64_t cta0 = (int64_t)blockIdx.x - crank + rank;  // slice 0's CTA of this pair half
          if constexpr (via_l2) {
            float* mine = p.sk_ws + ((int64_t)blockIdx.x * 4 + q) * SK_WARP_FLOATS;
#pragma unroll 1
            for (int c32 = 0; c32 < WS_BN / 32; ++c32) {
              if (c32 >= cb && c32 < ce) continue;
              uint32_t v[32];
              tmem_ld_32x32b_x32(tbase + (uint32_t)(c32 * 32), v);
              tmem_wait_ld();
              sk_store32(mine + c32 * SK_CHUNK_FLOATS, lane, v);
            }
          } else {
            float* mine = reinterpret_cast<float*>(ring) + (int64_t)q * SK_WARP_FLOATS;
#pragma unroll 1
            for (int c32 = 0; c32 < WS_BN / 32; ++c32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tbase + (uint32_t)(c32 * 32), v);
              tmem_wait_ld();
              sk_store32(mine + c32 * SK_CHUNK_FLOATS, lane, v);
            }
          }
          fence_cluster();
          __syncwarp();
          if (lane < (uint32_t)ks_n) mbar_arrive_cluster(mapa_shared(smem_u32(red_full), lane * CG + rank));
          uint32_t got2 = 1;
          if (lane == 0) got2 = mbar_wait<true>(smem_u32(red_full), 0, w, WAIT_SK_PARTIAL) ? 1u : 0u;
          got2 = __shfl_sync(0xffffffffu, got2, 0);
          if (!got2) { ok = false; break; }
          const int32_t row = row0 + (int32_t)lane;
#pragma unroll 1
          for (int c32 = cb; c32 < ce; ++c32) {
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;  // +0.0f
            // the partials of up to four CTAs are requested together, then added
            for (int32_t pr0 = 0; pr0 < ks_n; pr0 += 4) {
              float4 a4[4][8];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int32_t pr = pr0 + u;
                if (pr < ks_n && !(via_l2 && pr == ks_r)) {
                  if constexpr (via_l2) {
                    const float4* src = reinterpret_cast<const float4*>(
                                            p.sk_ws + ((cta0 + pr * CG) * 4 + q) * SK_WARP_FLOATS + c32 * SK_CHUNK_FLOATS) +
                                        lane;
#pragma unroll
                    for (int j = 0; j < 8; ++j) a4[u][j] = ld_cg_f32x4(src + j * 32);
                  } else {
                    const uint32_t base =
                        mapa_shared(smem_u32(ring), (uint32_t)pr * CG + rank) +
                        (uint32_t)(((int)q * (WS_BN / 32) + c32) * SK_CHUNK_FLOATS + (int)lane * 4) * 4u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) a4[u][j] = ld_cluster_f32x4(base + 512u * j);
                  }
                }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int32_t pr = pr0 + u;
                if (pr < ks_n) {
                  if (via_l2 && pr == ks_r) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tbase + (uint32_t)(c32 * 32), o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(o[j]));
                  } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                      v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + a4[u][j].x);
                      v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + a4[u][j].y);
                      v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + a4[u][j].z);
                      v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + a4[u][j].w);
                    }
                  }
                }
              }
            }
            if (row < p.M) store_row32<OutT>(reinterpret_cast<OutT*>(p.C), p.out_ld, row, col_base + 32 * c32, p.N, v);
          }
          continue;
        }
        if constexpr (DRAIN32) {
          // fp32 C, 7 chunks of 32 columns: one accumulator per consumer, so hand it back
          // as early as possible.  Chunks 0 and 1 go to the two staging buffers once the
          // previous tile's stores have read them, chunks 2-6 into registers; then the
          // accumulator is free and the stores follow (4096^3 fp16 -> fp32 on 512 x 224
          // tiles: the next tile's MMAs no longer wait for seven store round trips)
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * 32), v);
            tmem_wait_ld();
            uint8_t* buf = my_staging + ch * 4096;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(buf + sw128_offset(lane, (uint32_t)j)) =
                  make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
          uint32_t r[NCH - 2][32];
#pragma unroll
          for (int ch = 2; ch < NCH; ++ch) tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * 32), r[ch - 2]);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty + slot), lead));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              const int32_t col0 = col_base + ch * 32;
              if (row0 < p.M && col0 < p.N) tma_store_2d(tmC, smem_u32(my_staging + ch * 4096), col0, row0);
              bulk_commit_group();
            }
          }
#pragma unroll
          for (int ch = 2; ch < NCH; ++ch) {
            if (ch * 32 + 32 > tile_w) {
              // a narrow tile's last 16 columns (208 = 6 x 32 + 16): straight from
              // registers, so no store reaches into the next tile's columns
              const int32_t row = row0 + (int32_t)lane, col = col_base + ch * 32;
              if (ch * 32 < tile_w && row < p.M) {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<OutT*>(p.C) + (int64_t)row * p.out_ld + col);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (col + 4 * j < p.N)
                    dst[j] = make_uint4(r[ch - 2][4 * j], r[ch - 2][4 * j + 1], r[ch - 2][4 * j + 2], r[ch - 2][4 * j + 3]);
              }
              continue;
            }
            uint8_t* buf = my_staging + (ch & 1) * 4096;
            if (lane == 0) bulk_wait_group_read<1>();  // the store issued from `buf` two chunks ago is done reading
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(buf + sw128_offset(lane, (uint32_t)j)) =
                  make_uint4(r[ch - 2][4 * j], r[ch - 2][4 * j + 1], r[ch - 2][4 * j + 2], r[ch - 2][4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int32_t col0 = col_base + ch * 32;
              if (row0 < p.M && col0 < p.N) tma_store_2d(tmC, smem_u32(buf), col0, row0);
              bulk_commit_group();
            }
          }
          continue;
        }
        if constexpr (DRAIN) {
          // single accumulator (MX, and each consumer of step 9): first pull this warp's
          // 32 x 256 (or 224) slice into registers as packed bf16 and hand the
          // accumulator back, so the next tile's MMAs start while the stores below
          // drain (step 9, 8192 x 14336 x 4096: +1 %)
          uint32_t pk[NCH][32];
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * CW), v0);
            tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * CW + 32), v1);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              pk[ch][m] = pack_bf16x2(v0[2 * m], v0[2 * m + 1]);
              pk[ch][16 + m] = pack_bf16x2(v1[2 * m], v1[2 * m + 1]);
            }
          }
          uint32_t pt[TAIL > 0 ? 16 : 1];  // 224-column tile: columns 192-223
          if constexpr (TAIL > 0) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + (uint32_t)(NCH * CW), v);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 16; ++m) pt[m] = pack_bf16x2(v[2 * m], v[2 * m + 1]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (CG == 1) {
              mbar_arrive(smem_u32(acc_empty + slot));
            } else {
              mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty + slot), lead));
            }
          }
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            // two staging buffers in turn (MX: one), so a chunk is staged while the
            // store of the one before is still reading its buffer; the second
            // consumer's accumulator is handed back that much sooner
            uint8_t* buf = my_staging + (MX ? 0u : (tog & 1u) * 4096u);
            if (lane == 0) bulk_wait_group_read<MX ? 0 : 1>();  // the store issued from `buf` is done reading
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(buf + sw128_offset(lane, (uint32_t)j)) =
                  make_uint4(pk[ch][4 * j], pk[ch][4 * j + 1], pk[ch][4 * j + 2], pk[ch][4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int32_t col0 = col_base + ch * CW;
              if (row0 < p.M && col0 < p.N) tma_store_2d(tmC, smem_u32(buf), col0, row0);
              bulk_commit_group();
            }
            ++tog;
          }
          if constexpr (TAIL > 0) {
            // straight from registers to C: 64 bytes of the lane's row, 32 bytes in a
            // 208-column tile (N % 8 == 0, so each 8-column group is wholly in or out)
            const int32_t row = row0 + (int32_t)lane, col = col_base + NCH * CW;
            const int32_t col_end = min(p.N, col_base + tile_w);
            if (row < p.M) {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<OutT*>(p.C) + (int64_t)row * p.out_ld + col);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (col + 8 * j < col_end) dst[j] = make_uint4(pt[4 * j], pt[4 * j + 1], pt[4 * j + 2], pt[4 * j + 3]);
            }
          }
          continue;
        }
        if constexpr (KS == 0 && !DRAIN && !DRAIN32) {
          static_assert(TAIL == 0, "224-column tiles drain their accumulator first");
#pragma unroll 1
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t v0[32], v1[32];
            uint32_t res[EPI >= 0 ? 32 : 1];
            if constexpr (EPI >= 0) {
              // this chunk's residual, and the next chunk's on its way
#pragma unroll
              for (int j = 0; j < 32; ++j) res[j] = res_next[j];
              if (epi_res && ch + 1 < NCH)
                load_residual128<OutT>(res_next, p, row0 + (int32_t)lane, col_base + (ch + 1) * CW, v8_rows);
            }
            tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * CW), v0);
            if constexpr (CW == 64) tmem_ld_32x32b_x32(tbase + (uint32_t)(ch * CW + 32), v1);
            tmem_wait_ld();
            if constexpr (SK) {
              // add the other clusters' parts of this tile (clusters with an empty share
              // wrote nothing and are skipped, as in the count above)
              int32_t np = 0;
              for (int64_t c2 = sk_cid + 1; np < sk_nparts; ++c2) {
                if (sk_total * (c2 + 1) / sk_units == sk_total * c2 / sk_units) continue;
                const float* part = sk_part + (c2 - sk_cid - 1) * SK_SLOT_STRIDE * SK_WARP_FLOATS;
                sk_add32(v0, part + (ch * CW) / 32 * SK_CHUNK_FLOATS, lane);
                if constexpr (CW == 64) sk_add32(v1, part + ((ch * CW) / 32 + 1) * SK_CHUNK_FLOATS, lane);
                ++np;
              }
            }
            if (ch == NCH - 1) {
              // the whole accumulator is in registers: hand it back to the MMA warp
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                if constexpr (CG == 1) {
                  mbar_arrive(smem_u32(acc_empty + slot));
                } else {
                  mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty + slot), lead));
                }
              }
            }
            if constexpr (EPI >= 0) {
              // scales, bias, activation and residual, in fp32, before the single
              // rounding to C's type
              const int32_t col0 = col_base + ch * CW;
              apply_epilogue32<OutT, EPI>(v0, p, col0, epi_sa, epi_res, res);
              if constexpr (CW == 64) apply_epilogue32<OutT, EPI>(v1, p, col0 + 32, epi_sa, epi_res, res + 16);
            }
            uint8_t* buf = my_staging + (MX ? 0u : (tog & 1u) * 4096u);
            // the store issued from `buf` (two chunks ago; MX: one) is done reading
            if (lane == 0) bulk_wait_group_read<MX ? 0 : 1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4 val;
              if constexpr (CW == 32) {
                val = make_uint4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
              } else {
                const uint32_t* src = (j < 4) ? (v0 + 8 * j) : (v1 + 8 * (j - 4));
                val = make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]),
                                 pack_bf16x2(src[4], src[5]), pack_bf16x2(src[6], src[7]));
              }
              *reinterpret_cast<uint4*>(buf + sw128_offset(lane, (uint32_t)j)) = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int32_t col0 = col_base + ch * CW;
              if (row0 < p.M && col0 < p.N) tma_store_2d(tmC, smem_u32(buf), col0, row0);
              bulk_commit_group();
            }
            ++tog;
          }
        }
      }
      if (!ok) break;
      if constexpr (SK) {
        // the owner part consumed the following clusters' flags: clear them for the next launch
        if (kb0 == 0 && kb1 < KB) {
          __syncwarp();
          if (lane == 0) {
            const int64_t tile_end = (int64_t)(tile + 1) * KB;
            for (int64_t c2 = sk_cid + 1; c2 < sk_units && sk_total * c2 / sk_units < tile_end; ++c2)
#pragma unroll 1
              for (int cons = 0; cons < NCONS; ++cons) p.sk_flags[((c2 * CG + rank) * NCONS + cons) * 4 + q] = 0u;
          }
        }
      }
      if (p.visits != nullptr && q == 0 && my_cons <= 0 && lane == 0 && leader && (!SK || kb0 == 0) &&
          (!KS || ks_r == 0))
        atomicAdd(p.visits + tile, 1);
    }
    if (lane == 0) bulk_wait_group<0>();
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2 || KS != 0) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem, 512);
  }
}

// entry point of the fp16 / bf16 / 8-bit float kernels
template <typename OutT, int CG, int NCONS, int SCHED, int EPI = -1, int BN = WS_BN>
__global__ void __launch_bounds__(ws_threads(NCONS, EPI), 1)
    k_ws(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
         const __grid_constant__ CUtensorMap tmC, KParams p) {
  ws_body<OutT, CG, NCONS, SCHED, EPI, false, false, BN>(&tmA, &tmB, &tmC, nullptr, nullptr, p);
}

// entry point of the MX block-scaled kernels (one consumer; or two on the CTA
// pair's 512 x 224 tile, step 9)
template <typename OutT, int CG, int SCHED, int EPI = -1, int NCONS = 1, int BN = WS_BN>
__global__ void __launch_bounds__(mx_threads(NCONS), 1)
    k_ws_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSA,
            const __grid_constant__ CUtensorMap tmSB, KParams p) {
  ws_body<OutT, CG, NCONS, SCHED, EPI, true, false, BN>(&tmA, &tmB, &tmC, &tmSA, &tmSB, p);
}

// entry point of the split-K cluster kernels (step 7 tile, plain writeback);
// L2: clusters of more than two CTAs, partials exchanged through L2.  Each form
// is its own kernel: with both in one, the larger writeback code slowed the
// two-CTA form by 4 % (512 x 4096 x 4096: 742 against 770 TFLOP/s)
template <typename OutT, bool L2, int CG = 1>
__global__ void __launch_bounds__(WS_THREADS, 1)
    k_ws_ks(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, KParams p) {
  ws_body<OutT, CG, 1, SCHED_STATIC, -1, false, false, WS_BN, L2 ? 2 : 1>(&tmA, &tmB, &tmC, nullptr, nullptr, p);
}

// entry point of the stream-K kernels (static schedule, plain writeback)
template <typename OutT, int CG, int NCONS>
__global__ void __launch_bounds__(WS_THREADS, 1)
    k_ws_sk(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, KParams p) {
  ws_body<OutT, CG, NCONS, SCHED_STATIC, -1, false, true>(&tmA, &tmB, &tmC, nullptr, nullptr, p);
}

template <typename OutT, int CG, int NCONS, int SCHED, int EPI = -1, int BN = WS_BN>
void* ws_kernel_ptr() {
  return reinterpret_cast<void*>(k_ws<OutT, CG, NCONS, SCHED, EPI, BN>);
}

template <typename OutT, int CG, int SCHED, int EPI = -1, int NCONS = 1, int BN = WS_BN>
void* mx_kernel_ptr() {
  return reinterpret_cast<void*>(k_ws_mx<OutT, CG, SCHED, EPI, NCONS, BN>);
}

}  // namespace

}  // namespace dgb
