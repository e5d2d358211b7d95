// The warp-specialised, persistent 2-SM (cta_group::2) tcgen05 main loop shared
// by the library's tensor-core kernels (linear-logp calls of at most 128 rows
// use the one-CTA variant in rlk_solo.cuh instead).
//
// A cluster of two CTAs on two SMs computes one 256 x 256 FP32 accumulator
// tile per MMA chain: rank r holds rows [128 r, 128 r + 128) of the left
// operand and rows [128 r, 128 r + 128) of the right operand's 256-row tile in
// its own shared memory, and its own 128 rows of the accumulator in its own
// TMEM.  Rank 0 issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) for both.
//   warp 0, lane 0  TMA producer in each CTA; both CTAs' copies complete on
//                   rank 0's full barrier (rank 0 arms it for both halves).
//   warp 1          allocates 512 TMEM columns collectively with the peer; in
//                   rank 0, lane 0 issues the MMAs and commits to both CTAs'
//                   empty / accumulator-full barriers (multicast).
//   warps 2..5      epilogue on the CTA's own 128 accumulator rows; each warp
//                   releases the accumulator on rank 0's barrier (8 arrivals).
// Compared with one CTA owning a 128 x 256 tile, each SM reads half the
// right-operand bytes from shared memory per MMA for the same accumulator shape.
#pragma once

#include "rlk_device.cuh"

namespace rlk {

// Dynamic shared memory: alignment slack, the barrier block, then the stage ring.
constexpr int kSmemLimit = 232448;                    // 227 KiB per CTA
constexpr int kBarrierBlockBytes = 1024;              // keeps the ring 1024-byte aligned
constexpr int kMaxStages = 11;                        // barrier slots; the rings use at most 7

// The stage ring: each stage holds this CTA's 128 rows of the left operand and
// its kBHalf rows of the right-operand tile (half of the tile's 2 kBHalf
// columns), kK reduction columns each (64: 16 KiB apiece for 256-wide tiles, 7
// stages; 128: 32 KiB apiece, 3 stages), in two areas: left-operand blocks of all
// stages first, then the right-operand blocks.
template <int kBHalf_, int kK_ = kBK>
struct PairRingT {
  static constexpr int kBHalf = kBHalf_;
  static constexpr int kK = kK_;                                    // reduction elements per stage
  static constexpr int kTileN = 2 * kBHalf;                         // MMA N
  static constexpr int kABytes = kHalfRows * kK * 2;               // 16 or 32 KiB
  static constexpr int kBBytes = kBHalf * kK * 2;                  // 8 - 32 KiB
  static constexpr int kStages =
      (kSmemLimit - 1024 - kBarrierBlockBytes) / (kABytes + kBBytes) < kMaxStages
          ? (kSmemLimit - 1024 - kBarrierBlockBytes) / (kABytes + kBBytes)
          : kMaxStages;                                             // 7
  // Bytes rank 0's full barrier counts per stage (both CTAs' copies).
  static constexpr uint32_t kTxBytes = 2u * (kABytes + kBBytes);
  static constexpr int kSmemBytes = 1024 + kBarrierBlockBytes + kStages * (kABytes + kBBytes);
  static __device__ __forceinline__ uint32_t a_stage(uint32_t ring, int s) {
    return ring + s * kABytes;
  }
  static __device__ __forceinline__ uint32_t b_stage(uint32_t ring, int s) {
    return ring + kStages * kABytes + s * kBBytes;
  }
  static_assert(kSmemBytes <= kSmemLimit, "exceeds the 227 KiB per-CTA shared memory limit");
  // One CTA per SM: a second resident CTA could not get TMEM columns.
  static_assert(kSmemBytes > kSmemLimit / 2, "tcgen05 kernels must own their SM");
  static_assert(kBHalf == kHalfRows || kBHalf == kHalfRows / 2 || kBHalf == 112,
                "256-, 224- or 128-wide tiles");
};
using PairRing = PairRingT<kHalfRows>;                              // 256 x 256 tiles, 7 stages

// Row-operand extent above which the linear-logp 2-SM loops (the partials and the
// backward's G kernel) stage 128 reduction columns at a time (PairRingT<128, 128>,
// three 64 KiB stages) instead of 64 (seven 32 KiB stages).  Each stage carries a
// fixed cost besides its MMAs: with 128-column stages the MMA issuer spends about
// a tenth fewer cycles per 256 x 256 tile (mid shape 39,180 -> 35,010 cycles for
// 32,768 cycles of MMAs, debug-build role counters), while a call of a single
// 256-row block streams W from HBM and keeps the deeper ring (128-column stages
// made ragged N = 255 4.6% slower).  Either way the same 16-element MMAs run in
// the same order, so the bits do not depend on the choice.
constexpr int kWideStageRows = kPairRows;
constexpr int kSmemBytes = PairRing::kSmemBytes;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Acquire at cluster scope: sees what the peer CTA released before arriving.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded like mbar_wait (abort flag, time limit, poll cap), acquiring at cluster scope.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned int* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 31u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs || n > (1u << 30)) {
        *abort_flag = 1;
        atomicOr(err, kDevErrTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, int value) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(value) : "memory");
}

__device__ __forceinline__ void umma_pair_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once, on the barrier at this shared offset in every CTA of `mask`,
// when all MMAs issued so far by this thread are done.
__device__ __forceinline__ void umma_pair_commit(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Work units reach every role through a small ring that rank 0's scheduler
// fills (in both CTAs) and that each consumer releases on rank 0's barrier.
// A cluster's first unit is its own index and bypasses the ring, so the first
// tiles start without waiting on the counter.
constexpr int kUnitSlots = 4;
// Consumers of each slot: rank 0's producer, MMA issuer and 4 epilogue warps;
// rank 1's producer and 4 epilogue warps.
constexpr int kUnitConsumers = 2 + 4 + 1 + 4;
constexpr int kUnitDone = -1;      // no more units
constexpr int kUnitAbort = -2;     // the CTA is winding down

struct PipeBarriers {
  uint64_t full[kMaxStages];    // used in rank 0 only: both CTAs' copies for a stage
  uint64_t empty[kMaxStages];   // per CTA: the stage's shared memory may be refilled
  uint64_t acc_full[2];       // per CTA: accumulator b holds a finished tile
  uint64_t acc_empty[2];      // rank 0: both CTAs' epilogues released accumulator b
  uint64_t drained;           // rank 0: every issued MMA has completed
  uint64_t unit_full[kUnitSlots];    // per CTA: slot k holds the next unit
  uint64_t unit_empty[kUnitSlots];   // rank 0: every consumer has read slot k
  int unit_id[kUnitSlots];           // per CTA copy of the ring
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PipeBarriers) <= kBarrierBlockBytes, "barrier block overflows its bytes");

struct PipeSmem {
  uint32_t stages;   // the ring (1024-byte aligned)
  PipeBarriers* bars;
  uint32_t rank;
  __device__ __forceinline__ uint32_t full(int s) const { return smem_u32(&bars->full[s]); }
  __device__ __forceinline__ uint32_t empty(int s) const { return smem_u32(&bars->empty[s]); }
  __device__ __forceinline__ uint32_t acc_full(int b) const { return smem_u32(&bars->acc_full[b]); }
  __device__ __forceinline__ uint32_t acc_empty(int b) const {
    return smem_u32(&bars->acc_empty[b]);
  }
  __device__ __forceinline__ uint32_t unit_full(int k) const { return smem_u32(&bars->unit_full[k]); }
  __device__ __forceinline__ uint32_t unit_empty(int k) const {
    return smem_u32(&bars->unit_empty[k]);
  }
  __device__ __forceinline__ volatile int* abort_flag() const { return &bars->abort_flag; }
};

__device__ __forceinline__ PipeSmem pipe_smem(uint8_t* raw) {
  const uint32_t base = smem_u32(raw);
  const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
  PipeSmem p;
  p.bars = reinterpret_cast<PipeBarriers*>(raw + pad);
  p.stages = base + pad + kBarrierBlockBytes;
  p.rank = cluster_rank();
  return p;
}

// Barrier initialisation, collective TMEM allocation, then a cluster barrier
// so that no CTA touches its peer's barriers before they exist; then the wait
// for the previous kernel in the stream (programmatic dependent launch).
__device__ __forceinline__ uint32_t pipe_setup(const PipeSmem& ps) {
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(ps.full(s), 1);
      mbar_init(ps.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ps.acc_full(b), 1);
      mbar_init(ps.acc_empty(b), 2 * (kEpilogueThreads / 32));
    }
    mbar_init(smem_u32(&ps.bars->drained), 1);
    for (int k = 0; k < kUnitSlots; ++k) {
      mbar_init(ps.unit_full(k), 1);
      mbar_init(ps.unit_empty(k), kUnitConsumers);
    }
    ps.bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ps.bars->tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  // The prologue above touched only this CTA's shared memory and TMEM.
  griddep_wait();
  return ps.bars->tmem_base;
}

// Cluster barrier (no CTA leaves while its peer may still signal it or read
// its shared memory), then the collective TMEM release.
__device__ __forceinline__ void pipe_teardown(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (threadIdx.x / 32 == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Rank 0, warp 0, lane 1: hands out this cluster's units, in order, through the
// ring.  With a counter (a zeroed int in the caller's workspace) each cluster
// takes the next unit the moment it has room for it, so the units in flight
// stay a compact, in-order window of the schedule: clusters cannot drift apart
// over a long launch and evict each other's operand tiles from L2.  Without a
// counter there is no ring: every role takes units c, c + C, c + 2C, ... of
// cluster c directly.  Which cluster computes a unit never changes its
// arithmetic.
template <class Sched>
__device__ __forceinline__ void scheduler_role(const Sched& sc, const PipeSmem& ps,
                                               unsigned int* err) {
  if (sc.counter == nullptr) return;   // every role computes the round-robin order itself
  const int units = sc.num_units();
  // Unit 0 of cluster c is unit c (every role knows it without the ring); the
  // counter hands out units C, C + 1, ... from the second unit on, so ring
  // position j carries the cluster's unit j + 1.
  const int first_shared = (int)cluster_count();
  for (int j = 0;; ++j) {
    const int slot = j % kUnitSlots;
    const uint32_t parity = (uint32_t)(j / kUnitSlots) & 1u;
    if (!mbar_wait_cluster(ps.unit_empty(slot), parity ^ 1u, ps.abort_flag(), err)) return;
    int u = first_shared + atomicAdd(sc.counter, 1);
    if (u >= units) u = kUnitDone;
    ps.bars->unit_id[slot] = u;
    st_shared_cluster(mapa_shared(smem_u32(&ps.bars->unit_id[slot]), 1), u);
    mbar_arrive(ps.unit_full(slot));
    mbar_arrive_cluster(mapa_shared(ps.unit_full(slot), 1));
    if (u == kUnitDone) return;
  }
}

// Release slot `slot` after reading it (one arrival per consumer).  The arrival
// carries no data, and the consumer has already used the value it read, so it
// is relaxed: a release-ordered arrival from a thread with copies in flight
// would stall that thread until they land.
__device__ __forceinline__ void unit_release(const PipeSmem& ps, int slot) {
  if (ps.rank == 0)
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(ps.unit_empty(slot))
                 : "memory");
  else
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     mapa_shared(ps.unit_empty(slot), 0))
                 : "memory");
}

// The k-th unit of this cluster in the round-robin order (no counter).
template <class Sched>
__device__ __forceinline__ int unit_static(const Sched& sc, int k) {
  const int u = (int)cluster_index() + k * (int)cluster_count();
  return u < sc.num_units() ? u : kUnitDone;
}

// The k-th unit for a single-thread role: a unit id, kUnitDone or kUnitAbort.
template <class Sched>
__device__ __forceinline__ int unit_take(const Sched& sc, const PipeSmem& ps, int k,
                                         unsigned int* err) {
  if (sc.counter == nullptr || k == 0) return unit_static(sc, k);
  const int slot = (k - 1) % kUnitSlots;
  const uint32_t parity = (uint32_t)((k - 1) / kUnitSlots) & 1u;
  if (!mbar_wait_cluster(ps.unit_full(slot), parity, ps.abort_flag(), err)) return kUnitAbort;
  const int u = *reinterpret_cast<volatile int*>(&ps.bars->unit_id[slot]);
  unit_release(ps, slot);
  return u;
}

// The k-th unit for a whole warp (all lanes agree; lane 0 releases the slot).
template <class Sched>
__device__ __forceinline__ int warp_unit_take(const Sched& sc, const PipeSmem& ps, int k,
                                              unsigned int* err) {
  if (sc.counter == nullptr || k == 0) return unit_static(sc, k);
  const int slot = (k - 1) % kUnitSlots;
  const uint32_t parity = (uint32_t)((k - 1) / kUnitSlots) & 1u;
  const bool ok = mbar_wait_cluster(ps.unit_full(slot), parity, ps.abort_flag(), err);
  if (!__all_sync(0xffffffffu, ok)) return kUnitAbort;
  const int u = *reinterpret_cast<volatile int*>(&ps.bars->unit_id[slot]);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) unit_release(ps, slot);
  return u;
}

// Work description: a Schedule provides
//   int  num_units() const;                    units, handed out by scheduler_role
//   int* counter;                              zeroed unit counter, or nullptr
//   int  unit_tiles(int u) const;              accumulator tiles in unit u
//   void tile_coords(int u, int i, int& a0, int& b0) const;
//        a0 = first row of the pair's 256-row block of the left operand,
//        b0 = first row of the 256-row right-operand tile
//   int  nkb;                                  reduction stages (R::kK wide) per tile
//   int  nkb64;                                64-wide reduction blocks per tile
//        (read only by rings of 128-wide stages)
// The reduction of every tile runs over its blocks in ascending order and starts
// from zero, so a tile's arithmetic depends only on its operand tiles, never on
// the schedule, the grid or the row count.  TA / TB are the 128-row operand
// halves (OperandTile<majorness, 128>).
template <class TA, class TB, class Sched, class R = PairRing>
__device__ __forceinline__ void producer_role(const CUtensorMap* ta, const CUtensorMap* tb,
                                               const Sched& sc, const PipeSmem& ps,
                                               unsigned int* err) {
  static_assert(TA::kBytes == R::kABytes && TB::kBytes == R::kBBytes, "operand halves fit the ring");
  static_assert(TA::kK == R::kK && TB::kK == R::kK, "operand tiles and ring stage the same depth");
  constexpr int kStages = R::kStages;
  int stage = 0;
  uint32_t phase = 0, issued = 0, last_parity = 0;
  bool run = true;
  const int32_t half = (int32_t)ps.rank * kHalfRows;         // this CTA's left-operand rows
  const int32_t half_b = (int32_t)ps.rank * R::kBHalf;       // and right-operand rows
  const long long c_begin = RLK_CYCLES();                   // debug-build counters
  long long c_slot = 0;
  for (int k = 0; run; ++k) {
    const int u = unit_take(sc, ps, k, err);
    if (u < 0) {
      run = u != kUnitAbort;
      break;
    }
    const int nt = sc.unit_tiles(u);
    for (int i = 0; run && i < nt; ++i) {
      int a0, b0;
      sc.tile_coords(u, i, a0, b0);
      for (int kb = 0; kb < sc.nkb; ++kb) {
        const long long c0 = RLK_CYCLES();
        if (!mbar_wait(ps.empty(stage), phase ^ 1u, ps.abort_flag(), err)) {
          run = false;
          break;
        }
        c_slot += RLK_CYCLES() - c0;
        if (ps.rank == 0) mbar_arrive_expect_tx(ps.full(stage), R::kTxBytes);
        const uint32_t leader_full = mapa_shared(ps.full(stage), 0);
        TA::template load<true>(R::a_stage(ps.stages, stage), ta, leader_full, a0 + half,
                                kb * R::kK);
        TB::template load<true>(R::b_stage(ps.stages, stage), tb, leader_full, b0 + half_b,
                                kb * R::kK);
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  RLK_TRACE_SET(kTraceLoadSlotWait, c_slot);
  RLK_TRACE_SET(kTraceLoadCycles, RLK_CYCLES() - c_begin);
  // No more units for this CTA: the next kernel in the stream may start its
  // prologue on the SMs this grid frees from here on (it waits for this grid
  // to complete before it touches memory).  Signalling only now keeps its
  // blocks from sitting resident beside the main loop.
  griddep_launch_dependents();
  if (ps.rank == 0) {
    // Rank 0's full barriers count both CTAs' bytes: once they complete, every
    // copy of the pair has landed.
    for (int s = 0; s < kStages; ++s)
      if ((issued >> s) & 1u) mbar_wait_drain(ps.full(s), (last_parity >> s) & 1u, err);
  } else if (!run) {
    // Winding down early: rank 1 cannot observe rank 0's barriers, so it gives
    // its last copies a bounded 1 ms to land before the CTA may exit.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
}

template <class TA, class TB, class Sched, class R = PairRing>
__device__ __forceinline__ void mma_role(const Sched& sc, const PipeSmem& ps, uint32_t tmem,
                                          uint32_t idesc, unsigned int* err) {
  constexpr int kStages = R::kStages;
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool run = true;
  const long long c_begin = RLK_CYCLES();                   // debug-build counters
  long long c_operand = 0, c_acc = 0, tiles = 0;
  for (int k = 0; run; ++k) {
    const int u = unit_take(sc, ps, k, err);
    if (u < 0) break;
    const int nt = sc.unit_tiles(u);
    for (int i = 0; run && i < nt; ++i) {
      long long c0 = RLK_CYCLES();
      if (!mbar_wait(ps.acc_empty(acc), acc_phase ^ 1u, ps.abort_flag(), err)) {
        run = false;
        break;
      }
      c_acc += RLK_CYCLES() - c0;
      tc_fence_after();
      const uint32_t d = tmem + acc * kAccCols;
      for (int kb = 0; kb < sc.nkb; ++kb) {
        c0 = RLK_CYCLES();
        if (!mbar_wait(ps.full(stage), phase, ps.abort_flag(), err)) {
          run = false;
          break;
        }
        if (k == 0 && i == 0 && kb == 0)
          RLK_TRACE(2);                                    // the CTA's first stage has landed
        else
          c_operand += RLK_CYCLES() - c0;                  // (the first wait is start-up)
        tc_fence_after();
        const uint32_t sa = R::a_stage(ps.stages, stage);
        const uint32_t sb = R::b_stage(ps.stages, stage);
        // A 128-wide last stage that holds a single 64-wide block (an odd block
        // count) runs only that block's MMAs: every tile issues exactly the MMAs
        // of 64-wide staging, never an all-zero one (adding +0 would turn an
        // accumulated -0 into +0).
        bool one_block = false;
        if constexpr (R::kK > kBK) one_block = kb == sc.nkb - 1 && (sc.nkb64 & 1);
#pragma unroll
        for (int k = 0; k < R::kK / kUmmaK; ++k)
          if (k < kBK / kUmmaK || !one_block)
            umma_pair_bf16(d, TA::desc(sa, k), TB::desc(sb, k), idesc, (kb | k) != 0 ? 1u : 0u);
        umma_pair_commit(ps.empty(stage), 0x3);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!run) break;
      umma_pair_commit(ps.acc_full(acc), 0x3);
      ++tiles;
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  RLK_TRACE_SET(kTraceMmaOperandWait, c_operand);
  RLK_TRACE_SET(kTraceMmaAccWait, c_acc);
  RLK_TRACE_SET(kTraceMmaCycles, RLK_CYCLES() - c_begin);
  RLK_TRACE_SET(kTraceMmaTiles, tiles);
  umma_pair_commit(smem_u32(&ps.bars->drained), 0x1);
  mbar_wait_drain(smem_u32(&ps.bars->drained), 0, err);
}

__device__ __forceinline__ bool epilogue_acquire(const PipeSmem& ps, int acc, uint32_t parity,
                                                  unsigned int* err) {
  const bool ok = mbar_wait(ps.acc_full(acc), parity, ps.abort_flag(), err);
  const bool all = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  return all;
}

// Warp-level release of an accumulator on rank 0's barrier.
__device__ __forceinline__ void epilogue_release(const PipeSmem& ps, int acc) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (ps.rank == 0)
      mbar_arrive(ps.acc_empty(acc));
    else
      mbar_arrive_cluster(mapa_shared(ps.acc_empty(acc), 0));
  }
}

}  // namespace rlk
