// Deterministic BF16 GEMM family on sm_103a.
//
// "feat(musa): add native deterministic gemm kernel", Summary: forward
// C = A B, dA = dC B^T and dB = A^T dC with FP32 accumulation in a fixed,
// ascending K order; BF16 or FP32 output.  Review comment on that page: when the
// forward produced FP32, grad_output is rounded to BF16 before dA / dB.
// "Support musa", review comment: det_gemm never falls back to a
// non-deterministic matmul; unsupported cases fail explicitly.
//
// One kernel template serves all three products through the operands'
// majorness (which of the two extents of each operand is contiguous):
//   forward  A [M,K] reduction-contiguous (K-major), B [K,N] N-contiguous (MN-major)
//   dA       dC [M,N] K-major,                       B [K,N] K-major (N is reduced)
//   dB       A [M,K] MN-major (output rows = K),      dC [M,N] MN-major (M is reduced)
// Output tiles are 256 x 256 per CTA pair (2-SM tcgen05 loop, M=256 x N=256 x
// K=16 per MMA; 256 x 128 for outputs too small to fill the SM pairs and for a
// last wave that would leave most pairs idle; 256 x 224 for a K-major right
// operand where that fills the waves better), the reduction runs in ascending
// order in 16-element MMAs, each tile's accumulation starts from zero, and there is no
// split of the reduction: every output bit is a function of its own row of the
// left operand and column of the right operand only.
#include <mutex>

#include <cuda_bf16.h>

#include "rlk.h"
#include "rlk_internal.h"
#include "rlk_pipeline.cuh"

namespace rlk {

__device__ unsigned int g_err_det_gemm = 0;

namespace {

constexpr int kMidTileN = 224;   // tiles of K-major right operands (112 rows per CTA)

struct GemmSched {
  Banded order; // rows = 256-row output blocks (one per CTA pair), cols = order_n-column blocks
  int* counter; // nullptr: cluster c takes units c, c + C, ... (a few rounds at most sizes)
  int nkb;      // reduction stages (64 or 128 wide)
  int nkb64;    // 64-wide reduction blocks
  int order_n;  // output columns per block of the order (256, or 128 for narrow tiles throughout)
  int first;    // this launch's first block of the order
  int units;    // this launch's units
  int halves;   // 1: unit u is half (u & 1) of block first + u / 2 (128 of its 256 columns)
  __device__ __forceinline__ int num_units() const { return units; }
  __device__ __forceinline__ int unit_tiles(int) const { return 1; }
  __device__ __forceinline__ void tile_coords(int u, int, int& a0, int& b0) const {
    int mb, nb;
    order.unit(first + (halves ? u >> 1 : u), mb, nb);
    a0 = mb * kPairRows;
    b0 = nb * order_n + (halves ? (u & 1) * (order_n / 2) : 0);
  }
};

struct GemmOut {
  int M, N;          // output extent
  void* C;
  int64_t ldc;       // elements
  int fp32;          // 1: FP32 output, 0: BF16
  int accum;         // 1: FP32 C += product (C read once, added after the full reduction)
  int vec_bytes;     // widest vector store (16, 8 or 4 bytes) the base and pitch allow, or 0
};

// The widest vector store width (16, 8 or 4 bytes) that both the output's base
// address and its row pitch are multiples of (a chunk starts at a column that is
// a multiple of 32, so at a multiple of 64 bytes within its row), 0 for none.
inline int store_width(const void* C, int64_t ld, int64_t esize) {
  for (int w = 16; w >= 4; w /= 2)
    if (reinterpret_cast<uintptr_t>(C) % w == 0 && (ld * esize) % w == 0) return w;
  return 0;
}

__device__ __forceinline__ void store_chunk(const GemmOut& o, int row, int col0,
                                            const uint32_t (&r)[32]) {
  // the chunk's 32 columns (clipped to N) lie in row `row` of the M x ldc output
  if (!RLK_STORE_OK(row >= 0 && row < o.M && col0 >= 0 &&
                        (int64_t)min(col0 + 32, o.N) <= o.ldc,
                    &g_err_det_gemm))
    return;
  // whole chunks go out as the widest vector stores the output allows (the same
  // values and roundings as element stores); a row's ragged last chunk element-wise
  const int w = col0 + 32 <= o.N ? o.vec_bytes : 0;
  if (o.fp32) {
    float* dst = static_cast<float*>(o.C) + (int64_t)row * o.ldc + col0;
    if (o.accum) {
      if (w == 16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 c = reinterpret_cast<const float4*>(dst)[i];
          c.x = __fadd_rn(c.x, __uint_as_float(r[4 * i]));
          c.y = __fadd_rn(c.y, __uint_as_float(r[4 * i + 1]));
          c.z = __fadd_rn(c.z, __uint_as_float(r[4 * i + 2]));
          c.w = __fadd_rn(c.w, __uint_as_float(r[4 * i + 3]));
          reinterpret_cast<float4*>(dst)[i] = c;
        }
      } else if (w == 8) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float2 c = reinterpret_cast<const float2*>(dst)[i];
          c.x = __fadd_rn(c.x, __uint_as_float(r[2 * i]));
          c.y = __fadd_rn(c.y, __uint_as_float(r[2 * i + 1]));
          reinterpret_cast<float2*>(dst)[i] = c;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (col0 + i < o.N) dst[i] = __fadd_rn(dst[i], __uint_as_float(r[i]));
      }
    } else if (w == 16) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<uint4*>(dst)[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
    } else if (w == 8) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        reinterpret_cast<uint2*>(dst)[i] = make_uint2(r[2 * i], r[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < o.N) dst[i] = __uint_as_float(r[i]);
    }
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(o.C) + (int64_t)row * o.ldc + col0;
    if (w != 0) {
      uint32_t p[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        p[i] = *reinterpret_cast<uint32_t*>(&b);
      }
      if (w == 16) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<uint4*>(dst)[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
      } else if (w == 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          reinterpret_cast<uint2*>(dst)[i] = make_uint2(p[2 * i], p[2 * i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) reinterpret_cast<uint32_t*>(dst)[i] = p[i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < o.N) dst[i] = __float2bfloat16_rn(__uint_as_float(r[i]));
    }
  }
}

// One 256 x kTileN output tile per CTA pair (2-SM loop): rank r stages rows
// [a0 + 128 r, +128) of the left operand and rows / columns [b0 + kTileN/2 r,
// +kTileN/2) of the right operand, and stores its own 128 output rows.  Every
// output element sums the same 16-wide products over the same ascending 64-wide
// blocks whatever the tile width, so both widths give the same bits (tested).
template <bool kAMN, bool kBMN, int kTileN, int kStageK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    det_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    GemmSched sc, GemmOut out) {
  extern __shared__ uint8_t smem_raw[];
  const PipeSmem ps = pipe_smem(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  const uint32_t tmem = pipe_setup(ps);
  using R = PairRingT<kTileN / 2, kStageK>;
  using TA = OperandTile<kAMN, kHalfRows, kStageK>;
  using TB = OperandTile<kBMN, kTileN / 2, kStageK>;

  if (warp == 0) {
    if (lane == 0) producer_role<TA, TB, GemmSched, R>(&tm_a, &tm_b, sc, ps, &g_err_det_gemm);
    if (lane == 1 && ps.rank == 0) scheduler_role(sc, ps, &g_err_det_gemm);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && ps.rank == 0)
      mma_role<TA, TB, GemmSched, R>(sc, ps, tmem, idesc_bf16_f32(kPairRows, kTileN, kAMN, kBMN),
                                     &g_err_det_gemm);
    __syncwarp();
  } else {
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int k = 0;; ++k) {
      const int u = warp_unit_take(sc, ps, k, &g_err_det_gemm);
      if (u < 0) break;
      if (!epilogue_acquire(ps, acc, acc_phase, &g_err_det_gemm)) break;
      int m0, n0;
      sc.tile_coords(u, 0, m0, n0);
      const int row = m0 + (int)ps.rank * kHalfRows + q * 32 + lane;
      const uint32_t taddr = tmem + acc * kAccCols + lane_off;
#pragma unroll 1
      for (int c = 0; c < kTileN / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= out.N) break;               // uniform: depends on the tile only
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
        if (row < out.M) store_chunk(out, row, col0, r);
      }
      epilogue_release(ps, acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  pipe_teardown(tmem);
}

// out[r, c] = part_0[r, c] + part_1[r, c] + ... + part_{P-1}[r, c], added in FP32
// (round to nearest) in ascending part order, written as FP32 or BF16 (round to
// nearest even).  Consecutive threads take consecutive columns, so every part's
// row is read coalesced.
__global__ void __launch_bounds__(256)
    ordered_sum_kernel(const float* __restrict__ parts, int64_t P, int64_t rows, int64_t cols,
                       int64_t ld_in, int64_t part_stride, void* __restrict__ out, int out_fp32,
                       int64_t ld_out) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  // rows to blocks (blockIdx.y, then in steps of gridDim.y), a row's columns to
  // consecutive threads: coalesced, and no index division
  const int64_t c0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t cstep = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    for (int64_t c = c0; c < cols; c += cstep) {
      const float* p = parts + r * ld_in + c;
      float acc = __ldg(p);
      for (int64_t q = 1; q < P; ++q) acc = __fadd_rn(acc, __ldg(p + q * part_stride));
      if (!RLK_STORE_OK(r < rows && c < cols && c < ld_out, &g_err_det_gemm)) continue;
      if (out_fp32) {
        static_cast<float*>(out)[r * ld_out + c] = acc;
      } else {
        static_cast<__nv_bfloat16*>(out)[r * ld_out + c] = __float2bfloat16_rn(acc);
      }
    }
  }
}

// ---- Two products in one launch --------------------------------------------
// The linear-logp backward needs grad_hidden = G . W (the forward configuration,
// a few very long tiles: K = V) and grad_weight = G^T . hidden (the dB
// configuration, many short tiles).  Run apart, the long product leaves most SM
// pairs idle in its last wave.  Here both products' 256 x 256 tiles form one
// unit list, the product with the longer reduction first, handed out in order
// from one counter, so the short tiles fill the pairs the long ones leave idle.  Each tile is computed
// exactly as by det_gemm_kernel (same operands, same ascending reduction), so
// the outputs are the same bits as the two separate launches.
struct DualSched {
  Banded order1, order2;   // output blocks of product 1 and product 2
  int two_first;           // 1: product 2's units come first (its reduction is longer)
  int* counter;            // zeroed unit counter (ordered hand-out)
  int nkb1, nkb2;          // 64-wide reduction blocks of each product
  __device__ __forceinline__ int num_units() const { return order1.count() + order2.count(); }
  __device__ __forceinline__ int unit_tiles(int) const { return 1; }
  __device__ __forceinline__ bool second(int u) const {
    return two_first ? u < order2.count() : u >= order1.count();
  }
  __device__ __forceinline__ int unit_nkb(int u) const { return second(u) ? nkb2 : nkb1; }
  __device__ __forceinline__ void tile_coords(int u, int, int& a0, int& b0) const {
    int mb, nb;
    if (second(u))
      order2.unit(two_first ? u : u - order1.count(), mb, nb);
    else
      order1.unit(two_first ? u - order2.count() : u, mb, nb);
    a0 = mb * kPairRows;
    b0 = nb * kBN;
  }
};

// The TMA producer of the two-product loop (see producer_role): the unit's
// product selects the tensor maps and the operand layouts.
template <class TA1, class TB1, class TA2, class TB2>
__device__ __forceinline__ void dual_producer(const CUtensorMap* ta1, const CUtensorMap* tb1,
                                              const CUtensorMap* ta2, const CUtensorMap* tb2,
                                              const DualSched& sc, const PipeSmem& ps,
                                              unsigned int* err) {
  using R = PairRing;
  static_assert(TA1::kBytes == R::kABytes && TB1::kBytes == R::kBBytes &&
                    TA2::kBytes == R::kABytes && TB2::kBytes == R::kBBytes,
                "operand halves fit the ring");
  constexpr int kStages = R::kStages;
  int stage = 0;
  uint32_t phase = 0, issued = 0, last_parity = 0;
  bool run = true;
  const int32_t half = (int32_t)ps.rank * kHalfRows;
  for (int k = 0; run; ++k) {
    const int u = unit_take(sc, ps, k, err);
    if (u < 0) {
      run = u != kUnitAbort;
      break;
    }
    const bool two = sc.second(u);
    const int nkb = sc.unit_nkb(u);
    int a0, b0;
    sc.tile_coords(u, 0, a0, b0);
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait(ps.empty(stage), phase ^ 1u, ps.abort_flag(), err)) {
        run = false;
        break;
      }
      if (ps.rank == 0) mbar_arrive_expect_tx(ps.full(stage), R::kTxBytes);
      const uint32_t leader_full = mapa_shared(ps.full(stage), 0);
      const uint32_t sa = R::a_stage(ps.stages, stage), sb = R::b_stage(ps.stages, stage);
      if (two) {
        TA2::template load<true>(sa, ta2, leader_full, a0 + half, kb * kBK);
        TB2::template load<true>(sb, tb2, leader_full, b0 + half, kb * kBK);
      } else {
        TA1::template load<true>(sa, ta1, leader_full, a0 + half, kb * kBK);
        TB1::template load<true>(sb, tb1, leader_full, b0 + half, kb * kBK);
      }
      issued |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  griddep_launch_dependents();
  if (ps.rank == 0) {
    for (int s = 0; s < kStages; ++s)
      if ((issued >> s) & 1u) mbar_wait_drain(ps.full(s), (last_parity >> s) & 1u, err);
  } else if (!run) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
}

// The MMA issuer of the two-product loop (see mma_role).
template <class TA1, class TB1, class TA2, class TB2>
__device__ __forceinline__ void dual_mma(const DualSched& sc, const PipeSmem& ps, uint32_t tmem,
                                         uint32_t idesc1, uint32_t idesc2, unsigned int* err) {
  using R = PairRing;
  constexpr int kStages = R::kStages;
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool run = true;
  for (int k = 0; run; ++k) {
    const int u = unit_take(sc, ps, k, err);
    if (u < 0) break;
    const bool two = sc.second(u);
    const int nkb = sc.unit_nkb(u);
    if (!mbar_wait(ps.acc_empty(acc), acc_phase ^ 1u, ps.abort_flag(), err)) break;
    tc_fence_after();
    const uint32_t d = tmem + acc * kAccCols;
    for (int kb = 0; kb < nkb; ++kb) {
      if (!mbar_wait(ps.full(stage), phase, ps.abort_flag(), err)) {
        run = false;
        break;
      }
      tc_fence_after();
      const uint32_t sa = R::a_stage(ps.stages, stage), sb = R::b_stage(ps.stages, stage);
#pragma unroll
      for (int j = 0; j < kBK / kUmmaK; ++j) {
        if (two)
          umma_pair_bf16(d, TA2::desc(sa, j), TB2::desc(sb, j), idesc2, (kb | j) != 0 ? 1u : 0u);
        else
          umma_pair_bf16(d, TA1::desc(sa, j), TB1::desc(sb, j), idesc1, (kb | j) != 0 ? 1u : 0u);
      }
      umma_pair_commit(ps.empty(stage), 0x3);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!run) break;
    umma_pair_commit(ps.acc_full(acc), 0x3);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  }
  umma_pair_commit(smem_u32(&ps.bars->drained), 0x1);
  mbar_wait_drain(smem_u32(&ps.bars->drained), 0, err);
}

// Product 1: out1 = A1 . B1 with A1 K-major and B1 MN-major (the forward
// configuration, kB1MN) or K-major (the dA configuration); product 2:
// out2 = A2^T . B2 in the dB configuration (both MN-major).
template <bool kB1MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    det_gemm_fwd_db_kernel(const __grid_constant__ CUtensorMap tm_a1,
                           const __grid_constant__ CUtensorMap tm_b1,
                           const __grid_constant__ CUtensorMap tm_a2,
                           const __grid_constant__ CUtensorMap tm_b2, DualSched sc, GemmOut out1,
                           GemmOut out2) {
  extern __shared__ uint8_t smem_raw[];
  const PipeSmem ps = pipe_smem(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_a1);
    tma_prefetch_desc(&tm_b1);
    tma_prefetch_desc(&tm_a2);
    tma_prefetch_desc(&tm_b2);
  }
  const uint32_t tmem = pipe_setup(ps);
  using TA1 = OperandTile<false, kHalfRows>;
  using TB1 = OperandTile<kB1MN, kHalfRows>;
  using TA2 = OperandTile<true, kHalfRows>;
  using TB2 = OperandTile<true, kHalfRows>;
  if (warp == 0) {
    if (lane == 0)
      dual_producer<TA1, TB1, TA2, TB2>(&tm_a1, &tm_b1, &tm_a2, &tm_b2, sc, ps, &g_err_det_gemm);
    if (lane == 1 && ps.rank == 0) scheduler_role(sc, ps, &g_err_det_gemm);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && ps.rank == 0)
      dual_mma<TA1, TB1, TA2, TB2>(sc, ps, tmem, idesc_bf16_f32(kPairRows, kBN, false, kB1MN),
                                   idesc_bf16_f32(kPairRows, kBN, true, true), &g_err_det_gemm);
    __syncwarp();
  } else {
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int k = 0;; ++k) {
      const int u = warp_unit_take(sc, ps, k, &g_err_det_gemm);
      if (u < 0) break;
      if (!epilogue_acquire(ps, acc, acc_phase, &g_err_det_gemm)) break;
      const GemmOut& out = sc.second(u) ? out2 : out1;
      int m0, n0;
      sc.tile_coords(u, 0, m0, n0);
      const int row = m0 + (int)ps.rank * kHalfRows + q * 32 + lane;
      const uint32_t taddr = tmem + acc * kAccCols + lane_off;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= out.N) break;               // uniform: depends on the tile only
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
        if (row < out.M) store_chunk(out, row, col0, r);
      }
      epilogue_release(ps, acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  pipe_teardown(tmem);
}

std::mutex g_attr_mutex;
bool g_attr_set[64];

template <bool kAMN, bool kBMN, int kTileN, int kStageK>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(det_gemm_kernel<kAMN, kBMN, kTileN, kStageK>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PairRingT<kTileN / 2, kStageK>::kSmemBytes);
}

cudaError_t ensure_attrs(int dev) {
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev]) {
    cudaError_t e = set_attr<false, true, 256, 64>();
    if (e == cudaSuccess) e = set_attr<false, false, 256, 64>();
    if (e == cudaSuccess) e = set_attr<true, true, 256, 64>();
    if (e == cudaSuccess) e = set_attr<false, true, 128, 128>();
    if (e == cudaSuccess) e = set_attr<false, false, 128, 128>();
    if (e == cudaSuccess) e = set_attr<true, true, 128, 128>();
    if (e == cudaSuccess) e = set_attr<false, false, kMidTileN, 128>();
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(det_gemm_fwd_db_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(det_gemm_fwd_db_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_set[dev] = true;
  }
  return cudaSuccess;
}

// Tiling, from the output's extents, the reduction length, the right operand's
// majorness and the number of CTA pairs only.  Wide tiles are 256 x 256 with
// 64-element stages; narrow ones 256 x 128 and, for a K-major right operand
// (dA, the linear forward), 256 x 224 tiles, both with 128-element stages.  Times
// per tile relative to a wide one, measured on GB300: narrow 0.69 (uniform
// narrow tiles at 4096^3: 105 us against 86.7 us; 134 us with 64-element
// stages), 224-wide 0.89 - 0.93 (0.99 with 64-element stages).  The plan with
// the fewest wide-tile times per pair wins:
//  * narrow tiles throughout when all wide tiles fit in half a wave (1000^3:
//    15.0 - 16.0 vs 15.0 - 17.1 us with 64-element stages);
//  * for a last, partial wave that would fill at most half the pairs, when the
//    reduction is long: its wide blocks computed as two narrow halves each in a
//    second launch, which costs a few microseconds of its own (4096^3: 88.7 vs
//    86.7 us; 4096 x 151936 x 4096: 2.80 vs 2.96 - 3.01 ms);
//  * 224-wide tiles where their waves cost less (dA at 4096^3: 19 x 16 = 304
//    tiles fill 4 waves, 80.6 - 82.6 against 86.7 - 87.5 us; at 3072 x 4096 x
//    3072 51.9 against 53.9 us; where they add a wave, 2 - 3% slower: not chosen).
// Every output element runs the same 16-element MMAs in the same order whatever
// the tile, so the bits are the same.
constexpr int64_t kSplitMinReduction = 16384;
constexpr int64_t kHalfTileCost = 70;    // a narrow half tile, in hundredths of a wide tile's time
constexpr int64_t kMidTileCost = 93;     // a 224-wide tile
struct TilePlan {
  bool narrow;     // narrow tiles throughout
  int64_t split;   // wide blocks at the end of the order computed as narrow halves
  int wide_n;      // columns of the other tiles: 256, or 224 (K-major right operand)
};
TilePlan plan_tiles(int64_t out_rows, int64_t out_cols, int64_t red, int64_t clusters,
                    bool b_kmajor) {
  const int64_t rb = ceil_div(out_rows, kPairRows);
  const int64_t wide = rb * ceil_div(out_cols, kBN);
  if (2 * wide <= clusters) return {true, 0, kBN};
  TilePlan plan{false, 0, kBN};
  int64_t best = 100 * ceil_div(wide, clusters);
  const int64_t tail = wide % clusters;
  if (red >= kSplitMinReduction && wide > clusters && 2 * tail <= clusters) {
    plan.split = tail;
    best = 100 * (wide / clusters) + kHalfTileCost;
  }
  if (b_kmajor) {
    const int64_t mid = kMidTileCost * ceil_div(rb * ceil_div(out_cols, kMidTileN), clusters);
    if (100 * mid < 98 * best) plan = TilePlan{false, 0, kMidTileN};   // a 2% margin
  }
  return plan;
}

inline bool dtype_ok(int d) { return d == RLK_BF16 || d == RLK_FP32; }
inline int esize(int d) { return d == RLK_FP32 ? 4 : 2; }
inline bool ptr_aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
constexpr int64_t kDimLimit = int64_t(1) << 31;
constexpr int64_t kLdLimit = int64_t(1) << 36;

// One input operand of a product and how the kernel will read it.
struct Operand {
  const void* ptr;
  int dtype;
  int64_t rows, cols, ld;
  bool staged = false;        // copied / rounded into the workspace first
  int64_t eff_ld = 0;         // pitch the kernel reads
  size_t ws_off = 0, ws_bytes = 0;
};

void plan_operand(Operand& o, size_t& off) {
  o.staged = o.dtype == RLK_FP32 || !tma_ready(o.ptr, o.ld);
  o.eff_ld = o.staged ? staged_ld(o.cols) : o.ld;
  o.ws_off = off;
  o.ws_bytes = o.staged ? align_up((size_t)o.rows * o.eff_ld * 2, 256) : 0;
  off += o.ws_bytes;
}

rlk_status check_operand(const Operand& o, bool allow_fp32) {
  if (!dtype_ok(o.dtype) || (o.dtype == RLK_FP32 && !allow_fp32)) return RLK_ERR_DTYPE;
  if (o.rows < 0 || o.rows >= kMaxExtent || o.cols < 1 || o.cols >= kMaxExtent) return RLK_ERR_SHAPE;
  if (o.ld < o.cols || o.ld >= kLdLimit) return RLK_ERR_SHAPE;
  return RLK_OK;
}

// Stages (if planned) and returns the BF16 pointer the kernel reads.
rlk_status materialise(Operand& o, uint8_t* ws, cudaStream_t s, const void** out) {
  if (!o.staged) {
    *out = o.ptr;
    return RLK_OK;
  }
  uint16_t* dst = reinterpret_cast<uint16_t*>(ws + o.ws_off);
  cudaError_t e = o.dtype == RLK_FP32
                      ? launch_cast_f32_bf16(static_cast<const float*>(o.ptr), o.rows, o.cols, o.ld,
                                             dst, o.eff_ld, s)
                      : launch_stage_bf16(static_cast<const uint16_t*>(o.ptr), o.rows, o.cols, o.ld,
                                          dst, o.eff_ld, s);
  *out = dst;
  return e == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

enum class Kind { kFwd, kDa, kDb };

// Shared driver: x and y are the op's two inputs in argument order; the output
// is out_rows x out_cols, reduced over `red`.  The kind fixes how each operand
// is read: kFwd (x K-major, y MN-major), kDa (both K-major), kDb (both MN-major).
rlk_status run_gemm(Kind kind, Operand x, Operand y, int64_t out_rows, int64_t out_cols,
                    int64_t red, void* C, int c_dtype, int64_t ldc, void* workspace,
                    size_t workspace_bytes, void* stream, bool accum = false) {
  if (!dtype_ok(c_dtype)) return RLK_ERR_DTYPE;
  if (accum && c_dtype != RLK_FP32) return RLK_ERR_DTYPE;
  if (ldc < out_cols || ldc >= kLdLimit) return RLK_ERR_SHAPE;
  // units are numbered in ints (checked for the narrower, more numerous tiles)
  const int64_t num_mb = ceil_div(out_rows, kPairRows);
  if (num_mb * ceil_div(out_cols, kBN / 2) >= kDimLimit) return RLK_ERR_SHAPE;
  size_t off = 0;
  plan_operand(x, off);
  plan_operand(y, off);
  if (out_rows == 0) return RLK_OK;
  if (!C) return RLK_ERR_NULL;
  if (red > 0 && (!x.ptr || !y.ptr)) return RLK_ERR_NULL;
  if (!ptr_aligned(x.ptr, esize(x.dtype)) || !ptr_aligned(y.ptr, esize(y.dtype)) ||
      !ptr_aligned(C, esize(c_dtype)))
    return RLK_ERR_ALIGN;
  if (off > 0 && (!workspace || !ptr_aligned(workspace, 16) || workspace_bytes < off))
    return RLK_ERR_WORKSPACE;
  DeviceInfo dev;
  rlk_status st = device_ready(&dev);
  if (st != RLK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (red == 0 && accum) return RLK_OK;   // C += 0
  if (red == 0) {   // empty reduction (dB with M == 0): the product is all zeros
    const size_t es = esize(c_dtype);
    if (cudaMemset2DAsync(C, ldc * es, 0, out_cols * es, out_rows, s) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    return RLK_OK;
  }
  if (ensure_attrs(dev.device) != cudaSuccess) return RLK_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void *xp, *yp;
  if ((st = materialise(x, ws, s, &xp)) != RLK_OK) return st;
  if ((st = materialise(y, ws, s, &yp)) != RLK_OK) return st;

  const int64_t clusters = dev.sm_count / 2;
  const TilePlan plan = plan_tiles(out_rows, out_cols, red, clusters, kind == Kind::kDa);
  GemmOut o;
  o.M = (int)out_rows;
  o.N = (int)out_cols;
  o.C = C;
  o.ldc = ldc;
  o.fp32 = c_dtype == RLK_FP32;
  o.accum = accum ? 1 : 0;
  o.vec_bytes = store_width(C, ldc, esize(c_dtype));
  GemmSched sc;
  sc.order.rows = (int)num_mb;
  sc.order.cols = (int)ceil_div(out_cols, plan.narrow ? kBN / 2 : plan.wide_n);
  sc.order.band = band_rows(num_mb, red, kPairRows);
  sc.order_n = plan.narrow ? kBN / 2 : plan.wide_n;
  sc.counter = nullptr;
  sc.nkb64 = (int)ceil_div(red, kBK);

  // Tensor maps per tile width: {contiguous extent, row count}, pitch, box (per
  // CTA: 128 left-operand rows, tile_n / 2 right-operand rows or columns; an
  // MN-major box spans one stage of the reduction).  Both are encoded before
  // anything launches, so a failure leaves the output untouched.
  auto encode = [&](bool narrow, CUtensorMap* ta, CUtensorMap* tb) -> bool {
    const int tile_n = narrow ? kBN / 2 : plan.wide_n;
    const int stage_k = narrow || plan.wide_n == kMidTileN ? 128 : 64;
    switch (kind) {
      case Kind::kFwd:   // A [M,K] K-major; B [K,N] MN-major
        return encode_bf16_2d(ta, xp, x.cols, x.rows, x.eff_ld, kBK, kHalfRows) &&
               encode_bf16_2d(tb, yp, y.cols, y.rows, y.eff_ld, 64, stage_k);
      case Kind::kDa:    // dC [M,N] K-major; B [K,N] K-major (N reduced)
        return encode_bf16_2d(ta, xp, x.cols, x.rows, x.eff_ld, kBK, kHalfRows) &&
               encode_bf16_2d(tb, yp, y.cols, y.rows, y.eff_ld, kBK, tile_n / 2);
      case Kind::kDb:    // A [M,K] MN-major; dC [M,N] MN-major (M reduced)
        return encode_bf16_2d(ta, xp, x.cols, x.rows, x.eff_ld, 64, stage_k) &&
               encode_bf16_2d(tb, yp, y.cols, y.rows, y.eff_ld, 64, stage_k);
    }
    return false;
  };
  CUtensorMap ta_w, tb_w, ta_n, tb_n;
  const bool need_wide = !plan.narrow, need_narrow = plan.narrow || plan.split > 0;
  if ((need_wide && !encode(false, &ta_w, &tb_w)) || (need_narrow && !encode(true, &ta_n, &tb_n)))
    return RLK_ERR_CUDA;

  // One launch over units [first, first + units) of the order (halves: two narrow
  // units per wide block).
  auto launch = [&](int64_t first, int64_t units, bool narrow, bool halves) -> rlk_status {
    const CUtensorMap& ta = narrow ? ta_n : ta_w;
    const CUtensorMap& tb = narrow ? tb_n : tb_w;
    GemmSched part = sc;
    part.nkb = (int)ceil_div(red, narrow || plan.wide_n == kMidTileN ? 128 : 64);
    part.first = (int)first;
    part.units = (int)units;
    part.halves = halves ? 1 : 0;
    const int grid = 2 * (int)(units < clusters ? units : clusters);
    constexpr int kWideSmem = PairRingT<kHalfRows, 64>::kSmemBytes;
    constexpr int kNarrowSmem = PairRingT<kHalfRows / 2, 128>::kSmemBytes;
    cudaError_t e = cudaErrorInvalidValue;
    switch (kind) {
      case Kind::kFwd:
        e = narrow ? launch_overlapped(det_gemm_kernel<false, true, 128, 128>, grid, kThreads,
                                       kNarrowSmem, s, ta, tb, part, o)
                   : launch_overlapped(det_gemm_kernel<false, true, 256, 64>, grid, kThreads,
                                       kWideSmem, s, ta, tb, part, o);
        break;
      case Kind::kDa:
        e = narrow ? launch_overlapped(det_gemm_kernel<false, false, 128, 128>, grid, kThreads,
                                       kNarrowSmem, s, ta, tb, part, o)
            : plan.wide_n == kMidTileN
                ? launch_overlapped(det_gemm_kernel<false, false, kMidTileN, 128>, grid, kThreads,
                                    PairRingT<kMidTileN / 2, 128>::kSmemBytes, s, ta, tb, part, o)
                : launch_overlapped(det_gemm_kernel<false, false, 256, 64>, grid, kThreads,
                                    kWideSmem, s, ta, tb, part, o);
        break;
      case Kind::kDb:
        e = narrow ? launch_overlapped(det_gemm_kernel<true, true, 128, 128>, grid, kThreads,
                                       kNarrowSmem, s, ta, tb, part, o)
                   : launch_overlapped(det_gemm_kernel<true, true, 256, 64>, grid, kThreads,
                                       kWideSmem, s, ta, tb, part, o);
        break;
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    return RLK_OK;
  };
  const int64_t blocks = num_mb * sc.order.cols;
  if (plan.narrow) return launch(0, blocks, true, false);
  if ((st = launch(0, blocks - plan.split, false, false)) != RLK_OK) return st;
  return plan.split > 0 ? launch(blocks - plan.split, 2 * plan.split, true, true) : RLK_OK;
}

// Checks an output of a product before anything launches (the checks run_gemm
// makes on it), so that a two-product call fails closed.
rlk_status check_output(int64_t rows, int64_t cols, const void* C, int c_dtype, int64_t ldc) {
  if (!dtype_ok(c_dtype)) return RLK_ERR_DTYPE;
  if (ldc < cols || ldc >= kLdLimit) return RLK_ERR_SHAPE;
  if (ceil_div(rows, kPairRows) * ceil_div(cols, kBN / 2) >= kDimLimit) return RLK_ERR_SHAPE;
  if (rows > 0 && !C) return RLK_ERR_NULL;
  if (!ptr_aligned(C, esize(c_dtype))) return RLK_ERR_ALIGN;
  return RLK_OK;
}

// Both products of a backward from one gradient g [M, N]: out1 = g . r1 (kind k1)
// and out2 = (the kDb product of) x2 and g, with g staged (an FP32 g rounded to
// BF16, or a misaligned BF16 g copied) once into the workspace and shared.
// Workspace: [g staged][r1 staged][x2 staged][unit counter], each 256-byte aligned.
struct TwoProducts {
  Operand g, r1, x2;
  size_t off_ctr = 0, total = 0;
};

rlk_status plan_two(TwoProducts& t) {
  rlk_status st;
  if ((st = check_operand(t.g, true)) != RLK_OK || (st = check_operand(t.r1, false)) != RLK_OK ||
      (st = check_operand(t.x2, false)) != RLK_OK)
    return st;
  size_t off = 0;
  plan_operand(t.g, off);
  plan_operand(t.r1, off);
  plan_operand(t.x2, off);
  t.off_ctr = align_up(off, 256);
  t.total = t.off_ctr + 256;
  return RLK_OK;
}

// Runs out1 = kind1(g, r1) [rows1 x cols1, reduced over red1] and
// out2 = kDb(x2, g) [rows2 x cols2, reduced over M] after validating everything.
rlk_status run_two(TwoProducts t, Kind kind1, int64_t rows1, int64_t cols1, int64_t red1,
                   void* out1, int dt1, int64_t ld1, bool db_x2_is_left, int64_t rows2,
                   int64_t cols2, void* out2, int dt2, int64_t ld2, void* workspace,
                   size_t workspace_bytes, void* stream) {
  rlk_status st;
  if (out1 && (st = check_output(rows1, cols1, out1, dt1, ld1)) != RLK_OK) return st;
  if (out2 && (st = check_output(rows2, cols2, out2, dt2, ld2)) != RLK_OK) return st;
  if (!out1 && !out2) return RLK_OK;
  const int64_t M = t.g.rows;
  if (M > 0 && (!t.g.ptr || (out1 && !t.r1.ptr) || (out2 && !t.x2.ptr))) return RLK_ERR_NULL;
  if (!ptr_aligned(t.g.ptr, esize(t.g.dtype)) || !ptr_aligned(t.r1.ptr, 2) ||
      !ptr_aligned(t.x2.ptr, 2))
    return RLK_ERR_ALIGN;
  if (!workspace || !ptr_aligned(workspace, 16) || workspace_bytes < t.total)
    return RLK_ERR_WORKSPACE;
  DeviceInfo dev;
  if ((st = device_ready(&dev)) != RLK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {   // out1 has no rows; out2 is the empty sum
    if (out2 && cudaMemset2DAsync(out2, ld2 * esize(dt2), 0, cols2 * esize(dt2), rows2, s) !=
                    cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    return RLK_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // Stage each operand that a product will read at most once (g once for both);
  // the products then read BF16, TMA-ready copies and need no workspace.
  const bool use[3] = {true, out1 != nullptr, out2 != nullptr};
  Operand ops[3] = {t.g, t.r1, t.x2};
  for (int i = 0; i < 3; ++i) {
    if (!use[i]) continue;
    const void* p = ops[i].ptr;
    if ((st = materialise(ops[i], ws, s, &p)) != RLK_OK) return st;
    const int64_t ld = ops[i].staged ? ops[i].eff_ld : ops[i].ld;
    ops[i] = Operand{p, RLK_BF16, ops[i].rows, ops[i].cols, ld};
  }
  // Both products wanted, each filling at least one wave of SM pairs with 256 x 256
  // tiles, reductions within a factor of two: one launch over both tile lists, so
  // the tiles of the second product fill the pairs the first one's last wave leaves
  // idle (same bits; measured at 4096^3: 157 vs 167 us with a BF16 gradient; with
  // fewer tiles, or very unequal reductions, two launches were as fast or faster).
  const int64_t pairs = dev.sm_count / 2;
  const int64_t tiles1 = ceil_div(rows1, kPairRows) * ceil_div(cols1, kBN);
  const int64_t tiles2 = ceil_div(rows2, kPairRows) * ceil_div(cols2, kBN);
  const int64_t red_lo = red1 < M ? red1 : M, red_hi = red1 < M ? M : red1;
  if (out1 && out2 && tiles1 >= pairs && tiles2 >= pairs && red_hi <= 2 * red_lo) {
    TwoProductArgs p;
    p.a1 = ops[0].ptr;
    p.lda1 = ops[0].ld;
    p.b1 = ops[1].ptr;
    p.ldb1 = ops[1].ld;
    p.b1_mn = kind1 == Kind::kFwd;
    p.rows1 = rows1;
    p.cols1 = cols1;
    p.red1 = red1;
    const Operand& left2 = db_x2_is_left ? ops[2] : ops[0];
    const Operand& right2 = db_x2_is_left ? ops[0] : ops[2];
    p.a2 = left2.ptr;
    p.lda2 = left2.ld;
    p.b2 = right2.ptr;
    p.ldb2 = right2.ld;
    p.rows2 = rows2;
    p.cols2 = cols2;
    p.red2 = M;
    p.out1 = out1;
    p.dt1 = dt1;
    p.ld1 = ld1;
    p.out2 = out2;
    p.dt2 = dt2;
    p.ld2 = ld2;
    return launch_two_products(p, reinterpret_cast<int*>(ws + t.off_ctr), s);
  }
  if (out1) {
    st = run_gemm(kind1, ops[0], ops[1], rows1, cols1, red1, out1, dt1, ld1, nullptr, 0, stream);
    if (st != RLK_OK) return st;
  }
  if (out2) {
    st = db_x2_is_left
             ? run_gemm(Kind::kDb, ops[2], ops[0], rows2, cols2, M, out2, dt2, ld2, nullptr, 0,
                        stream)
             : run_gemm(Kind::kDb, ops[0], ops[2], rows2, cols2, M, out2, dt2, ld2, nullptr, 0,
                        stream);
    if (st != RLK_OK) return st;
  }
  return RLK_OK;
}

}  // namespace

rlk_status launch_two_products(const TwoProductArgs& p, int* counter, cudaStream_t s) {
  DeviceInfo dev;
  rlk_status st = device_ready(&dev);
  if (st != RLK_OK) return st;
  if (ensure_attrs(dev.device) != cudaSuccess) return RLK_ERR_CUDA;
  CUtensorMap ta1, tb1, ta2, tb2;
  // product 1: [rows1, cols1] = A1 [rows1, red1] (K-major) . B1 ([red1, cols1] MN-major,
  // or [cols1, red1] K-major); product 2: [rows2, cols2] = A2^T . B2 with A2 [red2, rows2]
  // and B2 [red2, cols2], both MN-major
  const bool b1_ok = p.b1_mn ? encode_bf16_2d(&tb1, p.b1, p.cols1, p.red1, p.ldb1, 64, kBK)
                             : encode_bf16_2d(&tb1, p.b1, p.red1, p.cols1, p.ldb1, kBK, kHalfRows);
  if (!encode_bf16_2d(&ta1, p.a1, p.red1, p.rows1, p.lda1, kBK, kHalfRows) || !b1_ok ||
      !encode_bf16_2d(&ta2, p.a2, p.rows2, p.red2, p.lda2, 64, kBK) ||
      !encode_bf16_2d(&tb2, p.b2, p.cols2, p.red2, p.ldb2, 64, kBK))
    return RLK_ERR_CUDA;
  DualSched sc;
  sc.order1.rows = (int)ceil_div(p.rows1, kPairRows);
  sc.order1.cols = (int)ceil_div(p.cols1, kBN);
  sc.order1.band = band_rows(sc.order1.rows, p.red1, kPairRows);
  sc.order2.rows = (int)ceil_div(p.rows2, kPairRows);
  sc.order2.cols = (int)ceil_div(p.cols2, kBN);
  sc.order2.band = band_rows(sc.order2.rows, p.red2, kPairRows);
  sc.nkb1 = (int)ceil_div(p.red1, kBK);
  sc.nkb2 = (int)ceil_div(p.red2, kBK);
  sc.two_first = sc.nkb2 > sc.nkb1 ? 1 : 0;
  sc.counter = counter;
  auto make_out = [](int64_t M, int64_t Ncols, void* C, int dt, int64_t ld) {
    GemmOut o;
    o.M = (int)M;
    o.N = (int)Ncols;
    o.C = C;
    o.ldc = ld;
    o.fp32 = dt == RLK_FP32;
    o.accum = 0;
    o.vec_bytes = store_width(C, ld, esize(dt));
    return o;
  };
  const GemmOut o1 = make_out(p.rows1, p.cols1, p.out1, p.dt1, p.ld1);
  const GemmOut o2 = make_out(p.rows2, p.cols2, p.out2, p.dt2, p.ld2);
  const int64_t units = (int64_t)sc.order1.rows * sc.order1.cols + (int64_t)sc.order2.rows * sc.order2.cols;
  const int64_t clusters = dev.sm_count / 2;
  const int grid = 2 * (int)(units < clusters ? units : clusters);
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(int), s);
  if (e == cudaSuccess)
    e = p.b1_mn ? launch_overlapped(det_gemm_fwd_db_kernel<true>, grid, kThreads, kSmemBytes, s,
                                    ta1, tb1, ta2, tb2, sc, o1, o2)
                : launch_overlapped(det_gemm_fwd_db_kernel<false>, grid, kThreads, kSmemBytes, s,
                                    ta1, tb1, ta2, tb2, sc, o1, o2);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  return RLK_OK;
}

rlk_status launch_fwd_and_db(const void* G, int64_t N, int64_t V, int64_t ldG, const void* W,
                             int64_t H, int64_t ldw, void* out1, int dt1, int64_t ld1,
                             const void* hidden, int64_t ldh, void* out2, int dt2, int64_t ld2,
                             int* counter, cudaStream_t s) {
  // [N, H] = G [N, V] . W [V, H] and [V, H] = G^T . hidden [N, H]
  TwoProductArgs p;
  p.a1 = G; p.lda1 = ldG; p.b1 = W; p.ldb1 = ldw; p.b1_mn = true;
  p.rows1 = N; p.cols1 = H; p.red1 = V;
  p.a2 = G; p.lda2 = ldG; p.b2 = hidden; p.ldb2 = ldh;
  p.rows2 = V; p.cols2 = H; p.red2 = N;
  p.out1 = out1; p.dt1 = dt1; p.ld1 = ld1; p.out2 = out2; p.dt2 = dt2; p.ld2 = ld2;
  return launch_two_products(p, counter, s);
}

uint32_t take_error_det_gemm() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_det_gemm, sizeof v) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaMemcpyToSymbol(g_err_det_gemm, &zero, sizeof zero);
  cudaGetLastError();
  return v;
}

}  // namespace rlk

using namespace rlk;

extern "C" {

rlk_status rlk_det_gemm_tile_plan(int op, int64_t out_rows, int64_t out_cols, int64_t red,
                                  int32_t sm_count, int32_t* tile_cols, int64_t* split_blocks,
                                  int32_t* launches) {
  if (!tile_cols || !split_blocks || !launches) return RLK_ERR_NULL;
  if (op < RLK_GEMM_FWD || op > RLK_GEMM_FWD_ACCUM) return RLK_ERR_SHAPE;
  if (out_rows < 1 || out_rows >= kMaxExtent || out_cols < 1 || out_cols >= kMaxExtent ||
      red < 1 || red >= kMaxExtent || sm_count < 2)
    return RLK_ERR_SHAPE;
  // the products whose right operand is read K-major: dA and the linear forward
  const bool b_kmajor = op == RLK_GEMM_DA || op == RLK_GEMM_LINEAR_FWD;
  const TilePlan plan = plan_tiles(out_rows, out_cols, red, sm_count / 2, b_kmajor);
  *tile_cols = plan.narrow ? kBN / 2 : plan.wide_n;
  *split_blocks = plan.split;
  *launches = plan.split > 0 ? 2 : 1;
  return RLK_OK;
}

size_t rlk_det_gemm_workspace_size(int op, const void* x, int x_dtype, int64_t x_rows,
                                   int64_t x_cols, int64_t ldx, const void* y, int y_dtype,
                                   int64_t y_rows, int64_t y_cols, int64_t ldy) {
  Operand a{x, x_dtype, x_rows, x_cols, ldx};
  Operand b{y, y_dtype, y_rows, y_cols, ldy};
  // which input may be an FP32 gradient (rounded to BF16 in the workspace)
  const bool fp32_x = op == RLK_GEMM_DA || op == RLK_GEMM_LINEAR_DX || op == RLK_GEMM_LINEAR_DW;
  const bool fp32_y = op == RLK_GEMM_DB;
  if (op < RLK_GEMM_FWD || op > RLK_GEMM_FWD_ACCUM) return 0;
  if (check_operand(a, fp32_x) != RLK_OK || check_operand(b, fp32_y) != RLK_OK) return 0;
  size_t off = 0;
  plan_operand(a, off);
  plan_operand(b, off);
  return off;
}

rlk_status rlk_det_gemm_fwd(const void* A, int64_t M, int64_t K, int64_t lda, const void* B,
                            int64_t N, int64_t ldb, void* C, int c_dtype, int64_t ldc,
                            void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  Operand a{A, RLK_BF16, M, K, lda};
  Operand b{B, RLK_BF16, K, N, ldb};
  rlk_status st;
  if ((st = check_operand(a, false)) != RLK_OK || (st = check_operand(b, false)) != RLK_OK) return st;
  if (K < 1) return RLK_ERR_SHAPE;
  return run_gemm(Kind::kFwd, a, b, M, N, K, C, c_dtype, ldc, workspace, workspace_bytes, stream);
}

rlk_status rlk_det_gemm_da(const void* dC, int dc_dtype, int64_t M, int64_t N, int64_t lddc,
                           const void* B, int64_t K, int64_t ldb, void* dA, int out_dtype,
                           int64_t ldda, void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  Operand a{dC, dc_dtype, M, N, lddc};
  Operand b{B, RLK_BF16, K, N, ldb};
  rlk_status st;
  if ((st = check_operand(a, true)) != RLK_OK || (st = check_operand(b, false)) != RLK_OK) return st;
  if (K < 1) return RLK_ERR_SHAPE;
  return run_gemm(Kind::kDa, a, b, M, K, N, dA, out_dtype, ldda, workspace, workspace_bytes,
                  stream);
}

rlk_status rlk_det_gemm_db(const void* A, int64_t M, int64_t K, int64_t lda, const void* dC,
                           int dc_dtype, int64_t N, int64_t lddc, void* dB, int out_dtype,
                           int64_t lddb, void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  Operand a{A, RLK_BF16, M, K, lda};
  Operand b{dC, dc_dtype, M, N, lddc};
  rlk_status st;
  if ((st = check_operand(a, false)) != RLK_OK || (st = check_operand(b, true)) != RLK_OK) return st;
  return run_gemm(Kind::kDb, a, b, K, N, M, dB, out_dtype, lddb, workspace, workspace_bytes,
                  stream);
}

rlk_status rlk_det_gemm_fwd_accum_fp32(const void* A, int64_t M, int64_t K, int64_t lda,
                                      const void* B, int64_t N, int64_t ldb, float* C,
                                      int64_t ldc, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  RLK_CALL_RANGE();
  Operand a{A, RLK_BF16, M, K, lda};
  Operand b{B, RLK_BF16, K, N, ldb};
  rlk_status st;
  if ((st = check_operand(a, false)) != RLK_OK || (st = check_operand(b, false)) != RLK_OK) return st;
  return run_gemm(Kind::kFwd, a, b, M, N, K, C, RLK_FP32, ldc, workspace, workspace_bytes, stream,
                  /*accum=*/true);
}

rlk_status rlk_det_linear_fwd(const void* X, int64_t M, int64_t K, int64_t ldx, const void* W,
                              int64_t N, int64_t ldw, void* Y, int y_dtype, int64_t ldy,
                              void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  Operand a{X, RLK_BF16, M, K, ldx};
  Operand b{W, RLK_BF16, N, K, ldw};
  rlk_status st;
  if ((st = check_operand(a, false)) != RLK_OK || (st = check_operand(b, false)) != RLK_OK) return st;
  // X [M,K] and W [N,K] are both reduction-contiguous: the dA configuration.
  return run_gemm(Kind::kDa, a, b, M, N, K, Y, y_dtype, ldy, workspace, workspace_bytes, stream);
}

rlk_status rlk_det_linear_dx(const void* dY, int dy_dtype, int64_t M, int64_t N, int64_t lddy,
                             const void* W, int64_t K, int64_t ldw, void* dX, int out_dtype,
                             int64_t lddx, void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  Operand a{dY, dy_dtype, M, N, lddy};
  Operand b{W, RLK_BF16, N, K, ldw};
  rlk_status st;
  if ((st = check_operand(a, true)) != RLK_OK || (st = check_operand(b, false)) != RLK_OK) return st;
  // dX [M,K] = dY [M,N] . W [N,K]: the forward configuration with W as the right operand.
  return run_gemm(Kind::kFwd, a, b, M, K, N, dX, out_dtype, lddx, workspace, workspace_bytes,
                  stream);
}

rlk_status rlk_det_linear_dw(const void* dY, int dy_dtype, int64_t M, int64_t N, int64_t lddy,
                             const void* X, int64_t K, int64_t ldx, void* dW, int out_dtype,
                             int64_t lddw, void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  Operand a{dY, dy_dtype, M, N, lddy};
  Operand b{X, RLK_BF16, M, K, ldx};
  rlk_status st;
  if ((st = check_operand(a, true)) != RLK_OK || (st = check_operand(b, false)) != RLK_OK) return st;
  // dW [N,K] = dY^T . X: the dB configuration with the gradient as the left operand.
  return run_gemm(Kind::kDb, a, b, N, K, M, dW, out_dtype, lddw, workspace, workspace_bytes,
                  stream);
}

size_t rlk_det_gemm_backward_workspace_size(const void* dC, int dc_dtype, int64_t M, int64_t N,
                                            int64_t lddc, const void* A, int64_t K, int64_t lda,
                                            const void* B, int64_t ldb) {
  TwoProducts t{{dC, dc_dtype, M, N, lddc}, {B, RLK_BF16, K, N, ldb}, {A, RLK_BF16, M, K, lda}};
  if (K < 1 || plan_two(t) != RLK_OK) return 0;
  return t.total;
}

rlk_status rlk_det_gemm_backward(const void* dC, int dc_dtype, int64_t M, int64_t N,
                                 int64_t lddc, const void* A, int64_t K, int64_t lda,
                                 const void* B, int64_t ldb, void* dA, int da_dtype, int64_t ldda,
                                 void* dB, int db_dtype, int64_t lddb, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  TwoProducts t{{dC, dc_dtype, M, N, lddc}, {B, RLK_BF16, K, N, ldb}, {A, RLK_BF16, M, K, lda}};
  if (K < 1) return RLK_ERR_SHAPE;
  rlk_status st = plan_two(t);
  if (st != RLK_OK) return st;
  // dA [M, K] = dC . B^T (the dA configuration); dB [K, N] = A^T . dC
  return run_two(t, Kind::kDa, M, K, N, dA, da_dtype, ldda, /*db_x2_is_left=*/true, K, N, dB,
                 db_dtype, lddb, workspace, workspace_bytes, stream);
}

size_t rlk_det_linear_backward_workspace_size(const void* dY, int dy_dtype, int64_t M,
                                             int64_t N, int64_t lddy, const void* X, int64_t K,
                                             int64_t ldx, const void* W, int64_t ldw) {
  TwoProducts t{{dY, dy_dtype, M, N, lddy}, {W, RLK_BF16, N, K, ldw}, {X, RLK_BF16, M, K, ldx}};
  if (K < 1 || plan_two(t) != RLK_OK) return 0;
  return t.total;
}

rlk_status rlk_det_linear_backward(const void* dY, int dy_dtype, int64_t M, int64_t N,
                                   int64_t lddy, const void* X, int64_t K, int64_t ldx,
                                   const void* W, int64_t ldw, void* dX, int dx_dtype,
                                   int64_t lddx, void* dW, int dw_dtype, int64_t lddw,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  TwoProducts t{{dY, dy_dtype, M, N, lddy}, {W, RLK_BF16, N, K, ldw}, {X, RLK_BF16, M, K, ldx}};
  if (K < 1) return RLK_ERR_SHAPE;
  rlk_status st = plan_two(t);
  if (st != RLK_OK) return st;
  // dX [M, K] = dY . W (the forward configuration); dW [N, K] = dY^T . X (dY on the left)
  return run_two(t, Kind::kFwd, M, K, N, dX, dx_dtype, lddx, /*db_x2_is_left=*/false, N, K, dW,
                 dw_dtype, lddw, workspace, workspace_bytes, stream);
}

rlk_status rlk_sum_partials_ordered(const float* partials, int64_t num_parts, int64_t rows,
                                    int64_t cols, int64_t ld_partial, int64_t part_stride,
                                    void* out, int out_dtype, int64_t ld_out, void* stream) {
  RLK_CALL_RANGE();
  if (!dtype_ok(out_dtype)) return RLK_ERR_DTYPE;
  if (num_parts < 1 || num_parts >= kDimLimit || rows < 0 || rows >= kMaxExtent || cols < 1 ||
      cols >= kMaxExtent || ld_partial < cols || ld_partial >= kLdLimit || ld_out < cols ||
      ld_out >= kLdLimit || part_stride < 0 || (num_parts > 1 && part_stride < rows * ld_partial))
    return RLK_ERR_SHAPE;
  if (rows == 0) return RLK_OK;
  if (!partials || !out) return RLK_ERR_NULL;
  if (!ptr_aligned(partials, 4) || !ptr_aligned(out, esize(out_dtype))) return RLK_ERR_ALIGN;
  DeviceInfo dev;
  rlk_status st = device_ready(&dev);
  if (st != RLK_OK) return st;
  // 256 threads per block: column blocks to cover a row once (at most 64), row
  // blocks up to about 8 blocks per SM in all (at most 65535)
  int64_t gx = ceil_div(cols, 256);
  gx = gx > 64 ? 64 : gx;
  int64_t gy = ceil_div(8 * (int64_t)dev.sm_count, gx);
  gy = gy > rows ? rows : gy;
  gy = gy < 1 ? 1 : (gy > 65535 ? 65535 : gy);
  const dim3 grid((unsigned)gx, (unsigned)gy, 1);
  if (launch_overlapped(ordered_sum_kernel, grid, 256, 0, static_cast<cudaStream_t>(stream),
                        partials, num_parts, rows, cols, ld_partial, part_stride, out,
                        out_dtype == RLK_FP32 ? 1 : 0, ld_out) != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  return RLK_OK;
}

}  // extern "C"
