// One-CTA variant of the tcgen05 main loop, for linear-logp calls of at most
// 128 rows.
//
// A CTA owns a whole unit: it stages its left-operand rows and the full 256-row
// right-operand tile per reduction block, and issues tcgen05.mma.cta_group::1
// (M=128, N=256, K=16) into one of two 256-column FP32 accumulators.  For a
// call of few rows the 2-SM loop spends its MMAs on 256 padded rows per tile
// and deals its units to SM pairs in waves; here a tile costs half the MMA time
// per SM and every SM takes a unit of its own.  Each output element still sums
// the same 16-wide products over the same ascending 64-wide blocks, and the
// epilogue is the same code, so a row's bits do not depend on which loop
// computed it (compared bit for bit on GB300 at 17, 300 and 1024 rows).
//
// Roles as in the 2-SM loop: warp 0 lane 0 TMA producer, warp 1 TMEM
// allocation and (lane 0) MMA issue, warps 2..5 epilogue on the 128
// accumulator rows.  Units are dealt round-robin (few rounds at these sizes).
#pragma once

#include "rlk_pipeline.cuh"

namespace rlk {

// Stage ring: kARows rows of the left operand (32 when every row of the call
// lies in the first 32, else 128) and the 256-row right-operand tile, 64
// reduction columns each; left-operand blocks of all stages first, then the
// right-operand blocks.  The MMA always reads 128 left rows: with the thin ring
// the rows past the 32 staged ones hold other data (the next stages' blocks),
// which reaches only accumulator rows that nothing reads (row i of a product
// depends on row i of the left operand alone).
template <int kARows_>
struct SoloRing {
  static constexpr int kARows = kARows_;
  static constexpr int kABytes = kARows * kBK * 2;                 // 4 or 16 KiB
  static constexpr int kBBytes = kBN * kBK * 2;                    // 32 KiB
  static constexpr int kStages =
      (kSmemLimit - 1024 - kBarrierBlockBytes) / (kABytes + kBBytes) < kMaxStages
          ? (kSmemLimit - 1024 - kBarrierBlockBytes) / (kABytes + kBBytes)
          : kMaxStages;
  static constexpr uint32_t kTxBytes = (uint32_t)(kABytes + kBBytes);
  static constexpr int kSmemBytes = 1024 + kBarrierBlockBytes + kStages * (kABytes + kBBytes);
  static __device__ __forceinline__ uint32_t a_stage(uint32_t ring, int s) {
    return ring + s * kABytes;
  }
  static __device__ __forceinline__ uint32_t b_stage(uint32_t ring, int s) {
    return ring + kStages * kABytes + s * kBBytes;
  }
  static_assert(kARows == kHalfRows || kARows == 32, "full or thin left operand");
  static_assert(kSmemBytes <= kSmemLimit, "exceeds the 227 KiB per-CTA shared memory limit");
  static_assert(kSmemBytes > kSmemLimit / 2, "tcgen05 kernels must own their SM");
  static_assert(kStages * (kABytes + kBBytes) >= kHalfRows * kBK * 2 + (kStages - 1) * kABytes,
                "left-operand reads leave the ring");
};
using SoloFull = SoloRing<kHalfRows>;   // 4 stages x 48 KiB
using SoloThin = SoloRing<32>;          // 6 stages x 36 KiB

// k-th unit of this CTA in round-robin order, or kUnitDone.
template <class Sched>
__device__ __forceinline__ int solo_unit(const Sched& sc, int k) {
  const int u = (int)blockIdx.x + k * (int)gridDim.x;
  return u < sc.num_units() ? u : kUnitDone;
}

// Barriers, the 512-column TMEM allocation, then the wait for the previous
// kernel in the stream (programmatic dependent launch).
__device__ __forceinline__ uint32_t solo_setup(const PipeSmem& ps) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(ps.full(s), 1);
      mbar_init(ps.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ps.acc_full(b), 1);
      mbar_init(ps.acc_empty(b), kEpilogueThreads / 32);
    }
    mbar_init(smem_u32(&ps.bars->drained), 1);
    ps.bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x / 32 == 1) {
    tmem_alloc(smem_u32(&ps.bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();
  return ps.bars->tmem_base;
}

__device__ __forceinline__ void solo_teardown(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x / 32 == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <class TA, class TB, class R, class Sched>
__device__ __forceinline__ void solo_producer(const CUtensorMap* ta, const CUtensorMap* tb,
                                              const Sched& sc, const PipeSmem& ps,
                                              unsigned int* err) {
  static_assert(TA::kBytes == R::kABytes && TB::kBytes == R::kBBytes, "operand blocks fit the ring");
  constexpr int kStages = R::kStages;
  int stage = 0;
  uint32_t phase = 0, issued = 0, last_parity = 0;
  bool run = true;
  const long long c_begin = RLK_CYCLES();                   // debug-build counters
  long long c_slot = 0;
  for (int k = 0; run; ++k) {
    const int u = solo_unit(sc, k);
    if (u < 0) break;
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
        const uint32_t full = ps.full(stage);
        mbar_arrive_expect_tx(full, R::kTxBytes);
        TA::load(R::a_stage(ps.stages, stage), ta, full, a0, kb * kBK);
        TB::load(R::b_stage(ps.stages, stage), tb, full, b0, kb * kBK);
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
  griddep_launch_dependents();   // no more units: the next kernel may begin its prologue
  // Every issued copy lands before the CTA can exit.
  for (int s = 0; s < kStages; ++s)
    if ((issued >> s) & 1u) mbar_wait_drain(ps.full(s), (last_parity >> s) & 1u, err);
}

template <class TA, class TB, class R, class Sched>
__device__ __forceinline__ void solo_mma(const Sched& sc, const PipeSmem& ps, uint32_t tmem,
                                         uint32_t idesc, unsigned int* err) {
  constexpr int kStages = R::kStages;
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool run = true;
  const long long c_begin = RLK_CYCLES();                   // debug-build counters
  long long c_operand = 0, c_acc = 0, tiles = 0;
  for (int k = 0; run; ++k) {
    const int u = solo_unit(sc, k);
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
#pragma unroll
        for (int j = 0; j < kBK / kUmmaK; ++j)
          umma_bf16(d, TA::desc(sa, j), TB::desc(sb, j), idesc, (kb | j) != 0 ? 1u : 0u);
        umma_commit(ps.empty(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!run) break;
      umma_commit(ps.acc_full(acc));
      ++tiles;
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  RLK_TRACE_SET(kTraceMmaOperandWait, c_operand);
  RLK_TRACE_SET(kTraceMmaAccWait, c_acc);
  RLK_TRACE_SET(kTraceMmaCycles, RLK_CYCLES() - c_begin);
  RLK_TRACE_SET(kTraceMmaTiles, tiles);
  // Every MMA issued above completes before the CTA frees TMEM.
  umma_commit(smem_u32(&ps.bars->drained));
  mbar_wait_drain(smem_u32(&ps.bars->drained), 0, err);
}

// Warp-level release of an accumulator (one arrival per epilogue warp).
__device__ __forceinline__ void solo_release(const PipeSmem& ps, int acc) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(ps.acc_empty(acc));
}

}  // namespace rlk
