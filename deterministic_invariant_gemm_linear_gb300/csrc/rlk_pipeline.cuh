// The warp-specialised tcgen05 main loop shared by the fused linear-logp
// kernel and the det_gemm kernel.
//
// CTA layout (192 threads, one CTA per SM, persistent over work units):
//   warp 0, lane 0  TMA producer: streams (A, B) reduction blocks of 64 into a
//                   kStages-deep shared-memory ring (full / empty mbarriers).
//   warp 1          allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//                   (M=128, N=256, K=16) into one of two FP32 accumulators and
//                   commits to the stage's empty barrier and, at the end of a
//                   tile, to the accumulator's full barrier.
//   warps 2..5      epilogue: each thread owns one accumulator row (TMEM lane)
//                   and releases the accumulator through its empty barrier.
//
// The reduction of every accumulator tile runs over its blocks in ascending
// order and always starts from zero: the arithmetic of a tile depends only on
// its two operand tiles, never on the schedule, the grid or the row count.
//
// Work description: a Schedule provides
//   int  num_units() const;                       units are dealt round-robin
//   int  unit_tiles(int u) const;                 accumulator tiles in unit u
//   void tile_coords(int u, int i, int& a_row0, int& b_row0) const;
//   int  nkb;                                     reduction blocks per tile
#pragma once

#include "rlk_device.cuh"

namespace rlk {

// Shared-memory bookkeeping that follows the stage buffers.
struct PipeBarriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drained;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PipeBarriers) <= 256, "barrier block overflows its reserved bytes");

struct PipeSmem {
  uint32_t stages;       // shared address of stage 0 (1024-byte aligned)
  PipeBarriers* bars;    // generic pointer to the barrier block
  __device__ __forceinline__ uint32_t full(int s) const { return smem_u32(&bars->full[s]); }
  __device__ __forceinline__ uint32_t empty(int s) const { return smem_u32(&bars->empty[s]); }
  __device__ __forceinline__ uint32_t acc_full(int b) const { return smem_u32(&bars->acc_full[b]); }
  __device__ __forceinline__ uint32_t acc_empty(int b) const {
    return smem_u32(&bars->acc_empty[b]);
  }
  __device__ __forceinline__ volatile int* abort_flag() const { return &bars->abort_flag; }
};

// Carves the dynamic shared memory: stage ring first (1024-byte aligned), then
// the barrier block.
__device__ __forceinline__ PipeSmem pipe_smem(uint8_t* raw) {
  const uint32_t base = smem_u32(raw);
  const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
  PipeSmem p;
  p.stages = base + pad;
  p.bars = reinterpret_cast<PipeBarriers*>(raw + pad + kStages * kStageBytes);
  return p;
}

// Barrier initialisation (one thread) and TMEM allocation (warp 1); ends with
// a CTA barrier so every role sees both.
__device__ __forceinline__ uint32_t pipe_setup(const PipeSmem& ps) {
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(ps.full(s), 1);
      mbar_init(ps.empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(ps.acc_full(b), 1);
      mbar_init(ps.acc_empty(b), kEpilogueThreads);
    }
    mbar_init(smem_u32(&ps.bars->drained), 1);
    ps.bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ps.bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return ps.bars->tmem_base;
}

// Final CTA barrier and TMEM release (warp 1).  Every role has drained its
// asynchronous work before reaching this point.
__device__ __forceinline__ void pipe_teardown(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x / 32 == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <class TA, class TB, class Sched>
__device__ __forceinline__ void producer_role(const CUtensorMap* ta, const CUtensorMap* tb,
                                              const Sched& sc, const PipeSmem& ps,
                                              unsigned int* err) {
  int stage = 0;
  uint32_t phase = 0, issued = 0, last_parity = 0;
  bool run = true;
  const int units = sc.num_units();
  for (int u = blockIdx.x; run && u < units; u += gridDim.x) {
    const int nt = sc.unit_tiles(u);
    for (int i = 0; run && i < nt; ++i) {
      int a0, b0;
      sc.tile_coords(u, i, a0, b0);
      for (int kb = 0; kb < sc.nkb; ++kb) {
        if (!mbar_wait(ps.empty(stage), phase ^ 1u, ps.abort_flag(), err)) {
          run = false;
          break;
        }
        const uint32_t full = ps.full(stage);
        mbar_arrive_expect_tx(full, kStageBytes);
        const uint32_t sa = ps.stages + stage * kStageBytes;
        TA::load(sa, ta, full, a0, kb * kBK);
        TB::load(sa + kAStageBytes, tb, full, b0, kb * kBK);
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
  // Let every issued copy land before the CTA can exit.
  for (int s = 0; s < kStages; ++s)
    if ((issued >> s) & 1u) mbar_wait_drain(ps.full(s), (last_parity >> s) & 1u, err);
}

template <class TA, class TB, class Sched>
__device__ __forceinline__ void mma_role(const Sched& sc, const PipeSmem& ps, uint32_t tmem,
                                         uint32_t idesc, unsigned int* err) {
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool run = true;
  const int units = sc.num_units();
  for (int u = blockIdx.x; run && u < units; u += gridDim.x) {
    const int nt = sc.unit_tiles(u);
    for (int i = 0; run && i < nt; ++i) {
      if (!mbar_wait(ps.acc_empty(acc), acc_phase ^ 1u, ps.abort_flag(), err)) {
        run = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + acc * kAccCols;
      for (int kb = 0; kb < sc.nkb; ++kb) {
        if (!mbar_wait(ps.full(stage), phase, ps.abort_flag(), err)) {
          run = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = ps.stages + stage * kStageBytes;
        const uint32_t sb = sa + kAStageBytes;
#pragma unroll
        for (int k = 0; k < kBK / kUmmaK; ++k)
          umma_bf16(d, TA::desc(sa, k), TB::desc(sb, k), idesc, (kb | k) != 0 ? 1u : 0u);
        umma_commit(ps.empty(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!run) break;
      umma_commit(ps.acc_full(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  // Every MMA issued above completes before the CTA frees TMEM.
  umma_commit(smem_u32(&ps.bars->drained));
  mbar_wait_drain(smem_u32(&ps.bars->drained), 0, err);
}

// Epilogue-side wait for an accumulator: all 32 lanes poll, then agree, so the
// warp-collective tcgen05.ld that follows is never reached by part of a warp.
__device__ __forceinline__ bool epilogue_acquire(const PipeSmem& ps, int acc, uint32_t parity,
                                                 unsigned int* err) {
  const bool ok = mbar_wait(ps.acc_full(acc), parity, ps.abort_flag(), err);
  const bool all = __all_sync(0xffffffffu, ok);
  tc_fence_after();
  return all;
}

__device__ __forceinline__ void epilogue_release(const PipeSmem& ps, int acc) {
  tc_fence_before();
  mbar_arrive(ps.acc_empty(acc));
}

}  // namespace rlk
