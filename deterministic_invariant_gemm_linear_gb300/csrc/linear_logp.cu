// Fused linear log-probability on sm_103a.
//
// Operator ("feat(linear-logp): add batch-invariant fused SM90 operator",
// Walkthrough and PR body): for each row r, z[r, v] = hidden[r] . W[v] (+ bias[v]);
// lse[r] = log sum_v exp z[r, v]; logp[r] = z[r, target[r]] - lse[r]; the [N, V]
// logits are never written to memory.
//
// Stage 1 (linear_logp_partials_kernel): the 2-SM tcgen05 main loop (a cluster
// of two CTAs, M=256 x N=256 per MMA) computes 256 x 256 FP32 logit tiles, each
// CTA holding its 128 rows in TMEM; calls of at most 128 rows run instead on
// the one-CTA loop (linear_logp_solo_kernel, M=128 x N=256 per MMA, one unit
// per CTA), which gives the same bits.  The epilogue keeps, per row and per vocabulary split,
// an online maximum m and sum of exponentials s over the split's tiles in
// ascending vocabulary order, and captures the target logit.  Work unit =
// (vocabulary split j, 256-row block) — 128-row on the one-CTA loop — dealt in
// L2-sized bands of row blocks so that the clusters running at the same time
// share hidden and W tiles in L2.
//
// Stage 2 (linear_logp_combine_kernel): one warp per row merges the row's S
// partials in a fixed order (lane l takes splits l, l+32, ... ascending, then a
// fixed xor butterfly) and writes lse and logp.
//
// The split (S, tiles per split) comes from V alone (the page's author notes:
// V -> split count -> contiguous ranges -> ordered merge; N, the row block and
// the SM count never enter), so each row's arithmetic is the same whatever N,
// its position and its neighbours are.
#include <math.h>

#include <mutex>

#include "rlk.h"
#include "rlk_internal.h"
#include "rlk_pipeline.cuh"
#include "rlk_solo.cuh"

namespace rlk {

__device__ unsigned int g_err_linear_logp = 0;

namespace {

struct LogpSched {
  Banded order;    // rows = 256-row blocks, cols = this call's vocabulary splits
  int* counter;    // zeroed unit counter in the workspace (units in order), or null (round-robin)
  int S;           // vocabulary splits in this call (all S, or a shard's run of them)
  int vps;         // 256-id tiles per split
  int vtiles;      // 256-id tiles of the weight rows this call reads
  int tile0;       // global index of the first of those tiles (0 unless a vocabulary shard)
  int nkb;         // reduction stages over H (64 or 128 wide)
  int nkb64;       // 64-wide blocks of H
  __device__ __forceinline__ int num_units() const { return order.count(); }
  __device__ __forceinline__ int split_of(int u) const {
    int rb, j;
    order.unit(u, rb, j);
    return j;
  }
  __device__ __forceinline__ int rb_of(int u) const {
    int rb, j;
    order.unit(u, rb, j);
    return rb;
  }
  __device__ __forceinline__ int first_tile(int u) const { return split_of(u) * vps; }
  __device__ __forceinline__ int unit_tiles(int u) const {
    const int t0 = first_tile(u);
    return min(vps, vtiles - t0);
  }
  int rows_per_unit;   // 256 (a CTA pair's rows) or 128 (one CTA's, the one-CTA loop)
  __device__ __forceinline__ void tile_coords(int u, int i, int& a0, int& b0) const {
    a0 = rb_of(u) * rows_per_unit;
    b0 = (first_tile(u) + i) * kBN;
  }
};

struct LogpArgs {
  int N, V;                   // V: the whole vocabulary (ids past it are masked)
  int v_off;                  // first vocabulary id of the weight rows read (shard start, or 0)
  int64_t tstride;
  const float* bias;          // [weight rows read] (bias[v - v_off]) or null
  bool bias_vec4;             // bias is 16-byte aligned: a lane reads its 8 floats as 2 vectors
  const int64_t* target;
  float2* ws_ms;              // [N][ld_ms]: (m, s) per row and split of this call
  int64_t ld_ms;
  float* ws_zt;               // [N]: target logit (rows whose target lies in this call's ids)
};

// One 32-column chunk (chunk c of its tile) of a row: bias, vocabulary-tail mask,
// target capture and the online (m, s) update.  z values are natural-unit logits;
// each exponential is 2^((z - m) * log2(e)) with z - m formed first, so the
// running maximum's own term is exactly 2^0 = 1: s >= 1 always, hence lse >= max
// logit and logp <= 0 hold exactly in FP32.  Column i's bias comes from the
// warp's BiasTile (a shuffle: every lane of the warp takes part).
__device__ __forceinline__ void logp_chunk(const uint32_t (&r)[32], int vbase, int V,
                                           bool has_bias, const BiasTile& bias, int c,
                                           int64_t tgt, float& m, float& s, bool& have_zt,
                                           float& zt) {
  float z[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(r[i]);
  if (has_bias) {
    if (vbase + 32 <= V) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        z[i] = __fadd_rn(z[i], bias_tile_at(bias, c, i));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float b = bias_tile_at(bias, c, i);
        if (vbase + i < V) z[i] = __fadd_rn(z[i], b);
      }
    }
  }
  if (vbase + 32 > V) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (vbase + i >= V) z[i] = -INFINITY;
  }
  const int64_t d = tgt - vbase;
  if (d >= 0 && d < 32) {
    // z[d] through a fixed 5-level select tree (keeps z in registers)
    const int di = (int)d;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = (di & 16) ? z[i + 16] : z[i];
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = (di & w) ? t[i + w] : t[i];
    zt = t[0];
    have_zt = true;
  }
  // chunk maximum (fixed pairwise tree)
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = fmaxf(z[2 * i], z[2 * i + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
  const float mn = fmaxf(m, t[0]);            // finite: vbase < V so z[0] is a real logit
  const float scale = ex2_approx(__fmul_rn(__fsub_rn(m, mn), kLog2e));   // m = -inf -> 0
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; ++i)
    a[i & 3] = __fadd_rn(a[i & 3], ex2_approx(__fmul_rn(__fsub_rn(z[i], mn), kLog2e)));
  const float cs = __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
  s = __fadd_rn(__fmul_rn(s, scale), cs);
  m = mn;
}

// Epilogue warps (2..5) of both loops: each thread owns one row (TMEM lane) of
// the CTA's 128 accumulator rows; for every 256-id tile of the unit's split, in
// ascending order, it folds the tile's logits into (m, s) 32 columns at a time,
// then writes the split's partial.  kSolo: the one-CTA loop (128-row blocks,
// round-robin units, local release); else the 2-SM loop (256-row blocks over
// the pair, units from the ring, release on rank 0's barrier).  The arithmetic
// is the same code either way.
template <bool kSolo>
__device__ __forceinline__ void logp_epilogue(const LogpSched& sc, const LogpArgs& args,
                                              const PipeSmem& ps, uint32_t tmem) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = warp & 3;
  const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool run = true;
  long long c_wait = 0, c_work = 0;                         // debug-build counters
  for (int k = 0; run; ++k) {
    const int u = kSolo ? solo_unit(sc, k) : warp_unit_take(sc, ps, k, &g_err_linear_logp);
    if (u < 0) break;
    const int j = sc.split_of(u);
    const int row = sc.rb_of(u) * sc.rows_per_unit + (kSolo ? 0 : (int)ps.rank * kHalfRows) +
                    q * 32 + lane;
    const bool valid = row < args.N;
    const int64_t tgt = valid ? __ldg(args.target + (int64_t)row * args.tstride) : -1;
    float m = -INFINITY, s = 0.f, zt = 0.f;
    bool have_zt = false;
    const int t0 = sc.first_tile(u), nt = sc.unit_tiles(u);
    const bool has_bias = args.bias != nullptr;
    for (int i = 0; i < nt; ++i) {
      const int v0 = (sc.tile0 + t0 + i) * kBN;   // global vocabulary id of the tile
      BiasTile bias;
      if (has_bias)
        load_bias_tile(args.bias + (v0 - args.v_off), args.V - v0, args.bias_vec4, lane, bias);
      const long long c0 = RLK_CYCLES();
      if (!epilogue_acquire(ps, acc, acc_phase, &g_err_linear_logp)) {
        run = false;
        break;
      }
      const long long c1 = RLK_CYCLES();
      c_wait += c1 - c0;
      if (threadIdx.x == 64) RLK_TRACE(3);     // an accumulator is complete
      const uint32_t taddr = tmem + acc * kAccCols + lane_off;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        const int vbase = v0 + c * 32;
        if (vbase >= args.V) break;          // uniform: depends on the tile only
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
        logp_chunk(r, vbase, args.V, has_bias, bias, c, tgt, m, s, have_zt, zt);
      }
      c_work += RLK_CYCLES() - c1;
      if (kSolo)
        solo_release(ps, acc);
      else
        epilogue_release(ps, acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!run) break;
    if (valid) {
      if (RLK_STORE_OK(row >= 0 && row < args.N && j >= 0 && j < args.ld_ms, &g_err_linear_logp))
        args.ws_ms[(int64_t)row * args.ld_ms + j] = make_float2(m, s);
      if (have_zt && RLK_STORE_OK(row >= 0 && row < args.N, &g_err_linear_logp))
        args.ws_zt[row] = zt;
    }
    if (threadIdx.x == 64) RLK_TRACE(4);       // the unit's partials are written
  }
  if (threadIdx.x == 64) {
    RLK_TRACE_SET(kTraceEpiAccWait, c_wait);
    RLK_TRACE_SET(kTraceEpiWork, c_work);
  }
}

// A cluster of two CTAs computes a unit = (split j, 256-row block) on the 2-SM
// tcgen05 loop; the CTA of rank r owns rows [256 * block + 128 r, +128).  kK:
// reduction elements per pipeline stage (64 or 128; see kWideStageRows).
template <int kK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    linear_logp_partials_kernel(const __grid_constant__ CUtensorMap tm_hidden,
                                     const __grid_constant__ CUtensorMap tm_weight, LogpSched sc,
                                     LogpArgs args) {
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) {
    RLK_TRACE(0);
    RLK_TRACE_CYCLES(6);
  }
  const PipeSmem ps = pipe_smem(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_hidden);
    tma_prefetch_desc(&tm_weight);
  }
  const uint32_t tmem = pipe_setup(ps);
  if (threadIdx.x == 0) RLK_TRACE(1);
  using THalf = OperandTile<false, kHalfRows, kK>;
  using R = PairRingT<kHalfRows, kK>;

  if (warp == 0) {
    if (lane == 0)
      producer_role<THalf, THalf, LogpSched, R>(&tm_hidden, &tm_weight, sc, ps, &g_err_linear_logp);
    if (lane == 1 && ps.rank == 0) scheduler_role(sc, ps, &g_err_linear_logp);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && ps.rank == 0)
      mma_role<THalf, THalf, LogpSched, R>(sc, ps, tmem, idesc_bf16_f32(kPairRows, kBN, false, false),
                                           &g_err_linear_logp);
    __syncwarp();
  } else {
    logp_epilogue<false>(sc, args, ps, tmem);
  }
  pipe_teardown(tmem);
  if (threadIdx.x == 0) {
    RLK_TRACE_CYCLES(7);
    RLK_TRACE(5);
  }
}

// One CTA per unit = (split j, 128-row block) on the one-CTA loop, for calls of
// at most 128 rows (a single row block).  R: SoloThin when N <= 32, else
// SoloFull.
template <class R>
__global__ void __launch_bounds__(kThreads, 1)
    linear_logp_solo_kernel(const __grid_constant__ CUtensorMap tm_hidden,
                            const __grid_constant__ CUtensorMap tm_weight, LogpSched sc,
                            LogpArgs args) {
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) {
    RLK_TRACE(0);
    RLK_TRACE_CYCLES(6);
  }
  const PipeSmem ps = pipe_smem(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_hidden);
    tma_prefetch_desc(&tm_weight);
  }
  const uint32_t tmem = solo_setup(ps);
  if (threadIdx.x == 0) RLK_TRACE(1);
  using TA = OperandTile<false, R::kARows>;
  using TB = OperandTile<false, kBN>;

  if (warp == 0) {
    if (lane == 0) solo_producer<TA, TB, R>(&tm_hidden, &tm_weight, sc, ps, &g_err_linear_logp);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0)
      solo_mma<TA, TB, R>(sc, ps, tmem, idesc_bf16_f32(kHalfRows, kBN, false, false),
                          &g_err_linear_logp);
    __syncwarp();
  } else {
    logp_epilogue<true>(sc, args, ps, tmem);
  }
  solo_teardown(tmem);
  if (threadIdx.x == 0) {
    RLK_TRACE_CYCLES(7);
    RLK_TRACE(5);
  }
}

// (m, s) pair merge with explicit roundings, so merge(a, b) == merge(b, a) bitwise.
__device__ __forceinline__ void merge_ms(float& M, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (M == -INFINITY) {
    M = m2;
    s = s2;
    return;
  }
  const float Mn = fmaxf(M, m2);
  const float e1 = ex2_approx(__fmul_rn(__fsub_rn(M, Mn), kLog2e));
  const float e2 = ex2_approx(__fmul_rn(__fsub_rn(m2, Mn), kLog2e));
  s = __fadd_rn(__fmul_rn(s, e1), __fmul_rn(s2, e2));
  M = Mn;
}

// Where the merge reads a row's S partials and its target logit.
// One [N][S] block of (m, s) partials and one [N] array of target logits (one GPU).
struct ContiguousPartials {
  const float2* ms;
  const float* zt;
  int S;
  __device__ __forceinline__ float2 at(int row, int j) const { return ms[(int64_t)row * S + j]; }
  __device__ __forceinline__ float target_logit(int row, int64_t) const { return zt[row]; }
};

// Partials gathered from vocabulary shards: shard q holds splits [off[q], off[q+1])
// as an [N][ld] block at ms + q * shard_stride, and target logits at
// zt + q * zt_stride for the rows whose target lies in its ids.
constexpr int kMaxShards = 64;
struct ShardedPartials {
  const float2* ms;
  int64_t ld, shard_stride;
  const float* zt;
  int64_t zt_stride;
  int vps;
  int off[kMaxShards + 1];
  __device__ __forceinline__ int shard_of(int j) const {   // j < off[last] = S
    int q = 0;
    while (j >= off[q + 1]) ++q;
    return q;
  }
  __device__ __forceinline__ float2 at(int row, int j) const {
    const int q = shard_of(j);
    return ms[q * shard_stride + (int64_t)row * ld + (j - off[q])];
  }
  __device__ __forceinline__ float target_logit(int row, int64_t t) const {
    const int q = shard_of((int)(t / kBN) / vps);
    return zt[q * zt_stride + row];
  }
};

// One warp per row: the same fixed order whatever the source of the partials,
// so a row's bits depend only on its partial values.
template <class Src>
__global__ void __launch_bounds__(256)
    linear_logp_combine_kernel(Src src, const int64_t* __restrict__ target, int64_t tstride, int N,
                               int S, int V, float* __restrict__ logp, float* __restrict__ lse,
                               float* __restrict__ zt_out) {
  griddep_wait();   // the partials kernel has finished and its writes are visible
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= N) return;
  float M = -INFINITY, s = 0.f;
  for (int j = lane; j < S; j += 32) {
    const float2 v = src.at(row, j);
    merge_ms(M, s, v.x, v.y);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    merge_ms(M, s, m2, s2);
  }
  if (lane == 0 && RLK_STORE_OK(row >= 0 && row < N, &g_err_linear_logp)) {
    const float L = __fadd_rn(M, logf(s));
    const int64_t t = __ldg(target + (int64_t)row * tstride);
    const float z = (t >= 0 && t < V) ? src.target_logit(row, t) : __int_as_float(0x7fc00000);
    lse[row] = L;
    logp[row] = __fsub_rn(z, L);
    if (zt_out) zt_out[row] = z;
  }
}

std::mutex g_attr_mutex;
bool g_attr_set[64];

cudaError_t ensure_attrs(int dev) {
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(linear_logp_partials_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairRingT<kHalfRows, 64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(linear_logp_partials_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairRingT<kHalfRows, 128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(linear_logp_solo_kernel<SoloFull>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SoloFull::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(linear_logp_solo_kernel<SoloThin>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SoloThin::kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_set[dev] = true;
  }
  return cudaSuccess;
}

// Workspace plan: [partials N*S float2][target logits N float][unit counter][staged hidden][staged W].
struct LogpPlan {
  int64_t S = 0, vps = 0, vtiles = 0;
  bool stage_h = false, stage_w = false;
  int64_t ldh = 0, ldw = 0;        // pitches the kernel reads
  size_t off_zt = 0, off_ctr = 0, off_h = 0, off_w = 0, total = 0;
};

rlk_status check_shapes(int64_t N, int64_t H, int64_t ldh, int64_t V, int64_t ldw) {
  if (N < 0 || N >= kMaxExtent) return RLK_ERR_SHAPE;
  if (H < 1 || H >= (int64_t(1) << 20)) return RLK_ERR_SHAPE;
  if (V < 1 || V >= kMaxExtent) return RLK_ERR_SHAPE;
  if (ldh < H || ldw < H) return RLK_ERR_SHAPE;
  if (ldh >= (int64_t(1) << 36) || ldw >= (int64_t(1) << 36)) return RLK_ERR_SHAPE;
  return RLK_OK;
}

// Contiguous equal splits of the vocabulary tiles: splits_req = 0 takes the
// V-only policy (rlk_vocab_split_policy); otherwise the tiles are cut into
// ceil(vtiles / ceil(vtiles / splits_req)) splits (splits_req clamped to
// [1, vtiles]).
rlk_status split_plan(int64_t V, int64_t splits_req, int64_t* S, int64_t* vps, int64_t* vtiles) {
  rlk_status st = rlk_vocab_split_policy(V, S, vps, vtiles);
  if (st != RLK_OK || splits_req == 0) return st;
  if (splits_req < 0) return RLK_ERR_SHAPE;
  const int64_t want = splits_req < *vtiles ? splits_req : *vtiles;
  *vps = ceil_div(*vtiles, want);
  *S = ceil_div(*vtiles, *vps);
  return RLK_OK;
}

rlk_status plan(const void* hidden, int64_t N, int64_t H, int64_t ldh, const void* weight,
                int64_t V, int64_t ldw, int64_t splits_req, LogpPlan* p) {
  rlk_status st = check_shapes(N, H, ldh, V, ldw);
  if (st != RLK_OK) return st;
  st = split_plan(V, splits_req, &p->S, &p->vps, &p->vtiles);
  if (st != RLK_OK) return st;
  // (split, row block) units are numbered in an int
  if (ceil_div(N, kPairRows) * p->S >= (int64_t(1) << 31)) return RLK_ERR_SHAPE;
  p->stage_h = !tma_ready(hidden, ldh);
  p->stage_w = !tma_ready(weight, ldw);
  p->ldh = p->stage_h ? staged_ld(H) : ldh;
  p->ldw = p->stage_w ? staged_ld(H) : ldw;
  size_t off = align_up((size_t)N * p->S * sizeof(float2), 256);
  p->off_zt = off;
  off = align_up(off + (size_t)N * sizeof(float), 256);
  p->off_ctr = off;
  off += 256;
  p->off_h = off;
  if (p->stage_h) off = align_up(off + (size_t)N * p->ldh * 2, 256);
  p->off_w = off;
  if (p->stage_w) off = align_up(off + (size_t)V * p->ldw * 2, 256);
  p->total = off;
  return RLK_OK;
}

}  // namespace

static_assert(kTraceFields == RLK_TRACE_FIELDS && kTraceCtas == RLK_TRACE_MAX_CTAS,
              "the trace table matches its description in rlk.h");

rlk_status read_trace(uint64_t* out, int64_t max_ctas, int64_t* n_ctas) {
#ifdef RLK_DEBUG
  if (!out || !n_ctas) return RLK_ERR_NULL;
  if (max_ctas < 0) return RLK_ERR_SHAPE;
  DeviceInfo dev;
  rlk_status st = device_ready(&dev);
  if (st != RLK_OK) return st;
  const int64_t n = max_ctas < kTraceCtas ? max_ctas : kTraceCtas;
  static unsigned long long zeros[kTraceCtas * kTraceFields];
  if (cudaDeviceSynchronize() != cudaSuccess ||
      (n > 0 && cudaMemcpyFromSymbol(out, g_trace, n * kTraceFields * sizeof(uint64_t)) !=
                    cudaSuccess) ||
      cudaMemcpyToSymbol(g_trace, zeros, sizeof zeros) != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  *n_ctas = n;
  return RLK_OK;
#else
  (void)out;
  (void)max_ctas;
  (void)n_ctas;
  return RLK_ERR_NOT_DEBUG_BUILD;
#endif
}

uint32_t take_error_linear_logp() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_linear_logp, sizeof v) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaMemcpyToSymbol(g_err_linear_logp, &zero, sizeof zero);
  cudaGetLastError();
  return v;
}

}  // namespace rlk

using namespace rlk;

namespace rlk {
namespace {

// One launch of the partials kernel over the weight rows of splits [j0, j1) of
// the vocabulary policy: the whole vocabulary (j0 = 0, j1 = S) or a shard of it.
// The caller has validated every argument; this stages misaligned operands,
// encodes the tensor maps and launches.
struct PartialsLaunch {
  const void* hidden;
  int64_t N, H, ld_hidden;
  bool stage_h;
  int64_t ldh;                 // pitch the kernel reads
  uint16_t* h_stage;           // padded copy of hidden (when stage_h)
  const void* weight;          // rows: vocabulary ids [v_off, v_off + w_rows)
  int64_t w_rows, ld_weight;
  bool stage_w;
  int64_t ldw;
  uint16_t* w_stage;
  int64_t V, vps, j0, j1, v_off;
  const float* bias;           // [w_rows] or null
  const int64_t* target;
  int64_t tstride;
  float2* ms;                  // [N][ld_ms]
  int64_t ld_ms;
  float* zt;                   // [N]
  int* counter;                // 256-byte slot for the unit counter
};

rlk_status launch_partials(const PartialsLaunch& L, const DeviceInfo& dev, cudaStream_t s) {
  if (ensure_attrs(dev.device) != cudaSuccess) return RLK_ERR_CUDA;
  const void* h_src = L.hidden;
  const void* w_src = L.weight;
  if (L.stage_h) {
    if (launch_stage_bf16(static_cast<const uint16_t*>(L.hidden), L.N, L.H, L.ld_hidden, L.h_stage,
                          L.ldh, s) != cudaSuccess)
      return RLK_ERR_CUDA;
    h_src = L.h_stage;
  }
  if (L.stage_w) {
    if (launch_stage_bf16(static_cast<const uint16_t*>(L.weight), L.w_rows, L.H, L.ld_weight,
                          L.w_stage, L.ldw, s) != cudaSuccess)
      return RLK_ERR_CUDA;
    w_src = L.w_stage;
  }
  // At most 128 rows (one 128-row block): the one-CTA loop, one unit per CTA;
  // otherwise the 2-SM loop over 256-row blocks.  At most 32 rows: the thin
  // rings (only 32 hidden rows staged per stage).
  const bool solo = L.N <= kHalfRows;
  const bool thin = L.N <= 32;
  const int kRowsPerUnit = solo ? kHalfRows : kPairRows;
  CUtensorMap tm_h, tm_w;
  if (!encode_bf16_2d(&tm_h, h_src, L.H, L.N, L.ldh, kBK, thin ? 32 : kHalfRows) ||
      !encode_bf16_2d(&tm_w, w_src, L.H, L.w_rows, L.ldw, kBK, solo ? kBN : kHalfRows))
    return RLK_ERR_CUDA;

  LogpSched sc;
  const int64_t splits = L.j1 - L.j0;
  sc.order.rows = (int)ceil_div(L.N, kRowsPerUnit);
  sc.order.cols = (int)splits;
  sc.order.band = band_rows(sc.order.rows, L.H, kRowsPerUnit);
  sc.rows_per_unit = kRowsPerUnit;
  sc.S = (int)splits;
  sc.vps = (int)L.vps;
  sc.vtiles = (int)ceil_div(L.w_rows, kBN);
  sc.tile0 = (int)(L.j0 * L.vps);
  // Calls of more than one 256-row block stage 128 reduction columns at a time on
  // the 2-SM loop (see kWideStageRows); the others 64.
  const int stage_k = !solo && L.N > kWideStageRows ? 128 : 64;
  sc.nkb = (int)ceil_div(L.H, stage_k);
  sc.nkb64 = (int)ceil_div(L.H, kBK);
  LogpArgs a;
  a.N = (int)L.N;
  a.V = (int)L.V;
  a.v_off = (int)L.v_off;
  a.ld_ms = L.ld_ms;
  a.tstride = L.tstride;
  a.bias = L.bias;
  a.bias_vec4 = (reinterpret_cast<uintptr_t>(L.bias) & 15u) == 0;
  a.target = L.target;
  a.ws_ms = L.ms;
  a.ws_zt = L.zt;
  const int64_t units = (int64_t)sc.order.rows * sc.S;   // < 2^31: checked by the caller
  if (solo) {
    sc.counter = nullptr;      // round-robin: at most ceil(1024 / #SMs) rounds
    const int grid = (int)(units < dev.sm_count ? units : dev.sm_count);
    const cudaError_t e =
        thin ? launch_overlapped(linear_logp_solo_kernel<SoloThin>, grid, kThreads,
                                 SoloThin::kSmemBytes, s, tm_h, tm_w, sc, a)
             : launch_overlapped(linear_logp_solo_kernel<SoloFull>, grid, kThreads,
                                 SoloFull::kSmemBytes, s, tm_h, tm_w, sc, a);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    return RLK_OK;
  }
  // One cluster of two CTAs per pair of SMs, persistent over the units.
  const int64_t clusters = dev.sm_count / 2;
  const int grid = 2 * (int)(units < clusters ? units : clusters);
  sc.counter = nullptr;
  if (ordered_units(units, clusters)) {
    sc.counter = L.counter;
    if (cudaMemsetAsync(sc.counter, 0, sizeof(int), s) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
  }
  const cudaError_t e =
      stage_k == 128
          ? launch_overlapped(linear_logp_partials_kernel<128>, grid, kThreads,
                              PairRingT<kHalfRows, 128>::kSmemBytes, s, tm_h, tm_w, sc, a)
          : launch_overlapped(linear_logp_partials_kernel<64>, grid, kThreads,
                              PairRingT<kHalfRows, 64>::kSmemBytes, s, tm_h, tm_w, sc, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  return RLK_OK;
}

rlk_status partials_impl(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                         const void* weight, int64_t V, int64_t ld_weight, const float* bias,
                         const int64_t* target, int64_t target_stride, int64_t splits_req,
                         void* workspace, size_t workspace_bytes, void* stream) {
  LogpPlan p;
  rlk_status st = plan(hidden, N, H, ld_hidden, weight, V, ld_weight, splits_req, &p);
  if (st != RLK_OK) return st;
  if (target_stride < 0) return RLK_ERR_SHAPE;
  if (N == 0) return RLK_OK;
  if (!hidden || !weight || !target) return RLK_ERR_NULL;
  if (!workspace) return RLK_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(hidden) & 1u) || (reinterpret_cast<uintptr_t>(weight) & 1u) ||
      (reinterpret_cast<uintptr_t>(target) & 7u) || (reinterpret_cast<uintptr_t>(bias) & 3u))
    return RLK_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) || workspace_bytes < p.total)
    return RLK_ERR_WORKSPACE;
  DeviceInfo dev;
  st = device_ready(&dev);
  if (st != RLK_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PartialsLaunch L;
  L.hidden = hidden;
  L.N = N;
  L.H = H;
  L.ld_hidden = ld_hidden;
  L.stage_h = p.stage_h;
  L.ldh = p.ldh;
  L.h_stage = reinterpret_cast<uint16_t*>(ws + p.off_h);
  L.weight = weight;
  L.w_rows = V;
  L.ld_weight = ld_weight;
  L.stage_w = p.stage_w;
  L.ldw = p.ldw;
  L.w_stage = reinterpret_cast<uint16_t*>(ws + p.off_w);
  L.V = V;
  L.vps = p.vps;
  L.j0 = 0;
  L.j1 = p.S;
  L.v_off = 0;
  L.bias = bias;
  L.target = target;
  L.tstride = target_stride;
  L.ms = reinterpret_cast<float2*>(ws);
  L.ld_ms = p.S;
  L.zt = reinterpret_cast<float*>(ws + p.off_zt);
  L.counter = reinterpret_cast<int*>(ws + p.off_ctr);
  return launch_partials(L, dev, static_cast<cudaStream_t>(stream));
}

rlk_status combine_impl(int64_t N, int64_t V, const int64_t* target, int64_t target_stride,
                        float* logp, float* lse, float* target_logit, int64_t splits_req,
                        const void* workspace, size_t workspace_bytes, void* stream) {
  if (N < 0 || N >= kMaxExtent || V < 1 || V >= kMaxExtent || target_stride < 0)
    return RLK_ERR_SHAPE;
  if (N == 0) return RLK_OK;
  if (!target || !logp || !lse) return RLK_ERR_NULL;
  if (!workspace) return RLK_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(target) & 7u) || (reinterpret_cast<uintptr_t>(logp) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(target_logit) & 3u))
    return RLK_ERR_ALIGN;
  int64_t S, vps, vt;
  rlk_status st = split_plan(V, splits_req, &S, &vps, &vt);
  if (st != RLK_OK) return st;
  const size_t off_zt = align_up((size_t)N * S * sizeof(float2), 256);
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) ||
      workspace_bytes < off_zt + (size_t)N * sizeof(float))
    return RLK_ERR_WORKSPACE;
  DeviceInfo dev;
  st = device_ready(&dev);
  if (st != RLK_OK) return st;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const int rows_per_block = 256 / 32;
  const int grid = (int)ceil_div(N, rows_per_block);
  ContiguousPartials src;
  src.ms = reinterpret_cast<const float2*>(ws);
  src.zt = reinterpret_cast<const float*>(ws + off_zt);
  src.S = (int)S;
  const cudaError_t e = launch_overlapped(
      linear_logp_combine_kernel<ContiguousPartials>, grid, 256, 0,
      static_cast<cudaStream_t>(stream), src, target, target_stride, (int)N, (int)S, (int)V, logp,
      lse, target_logit);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  return RLK_OK;
}

// ---- vocabulary shards ("feat(linear-logp)...", author notes: V -> split count
// -> contiguous ranges -> ordered merge).  A shard is a contiguous run of whole
// splits [j0, j1) of the V-only policy, i.e. the weight rows of vocabulary ids
// [v_begin, v_end); its partials are the ones the whole-vocabulary call computes
// for those splits, bit for bit, because every split is computed from the same
// tiles in the same order.
struct ShardPlan {
  int64_t S = 0, vps = 0, vtiles = 0;
  int64_t v_begin = 0, v_end = 0;
  bool stage_h = false, stage_w = false;
  int64_t ldh = 0, ldw = 0;
  size_t off_h = 0, off_w = 0, total = 0;     // [counter 256][staged hidden][staged W]
};

rlk_status shard_plan(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                      const void* weight, int64_t V, int64_t j0, int64_t j1, int64_t ld_weight,
                      ShardPlan* p) {
  rlk_status st = rlk_vocab_split_policy(V, &p->S, &p->vps, &p->vtiles);
  if (st != RLK_OK) return st;
  if (j0 < 0 || j1 < j0 || j1 > p->S) return RLK_ERR_SHAPE;
  p->v_begin = j0 * p->vps * kVocabTile;
  p->v_end = j1 * p->vps * kVocabTile < V ? j1 * p->vps * kVocabTile : V;
  const int64_t rows = p->v_end - p->v_begin;
  st = check_shapes(N, H, ld_hidden, rows > 0 ? rows : 1, ld_weight);
  if (st != RLK_OK) return st;
  if (ceil_div(N, kPairRows) * (j1 - j0) >= (int64_t(1) << 31)) return RLK_ERR_SHAPE;
  const bool work = N > 0 && rows > 0;
  p->stage_h = work && !tma_ready(hidden, ld_hidden);
  p->stage_w = work && !tma_ready(weight, ld_weight);
  p->ldh = p->stage_h ? staged_ld(H) : ld_hidden;
  p->ldw = p->stage_w ? staged_ld(H) : ld_weight;
  size_t off = 256;
  p->off_h = off;
  if (p->stage_h) off = align_up(off + (size_t)N * p->ldh * 2, 256);
  p->off_w = off;
  if (p->stage_w) off = align_up(off + (size_t)rows * p->ldw * 2, 256);
  p->total = off;
  return RLK_OK;
}

rlk_status shard_partials_impl(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                               const void* weight, int64_t V, int64_t j0, int64_t j1,
                               int64_t ld_weight, const float* bias, const int64_t* target,
                               int64_t target_stride, float* partials, int64_t ld_partials,
                               float* target_logit, void* workspace, size_t workspace_bytes,
                               void* stream) {
  ShardPlan p;
  rlk_status st = shard_plan(hidden, N, H, ld_hidden, weight, V, j0, j1, ld_weight, &p);
  if (st != RLK_OK) return st;
  if (target_stride < 0 || ld_partials < j1 - j0 || ld_partials >= (int64_t(1) << 31))
    return RLK_ERR_SHAPE;
  if (N == 0 || j0 == j1) return RLK_OK;
  if (!hidden || !weight || !target || !partials || !target_logit) return RLK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(hidden) & 1u) || (reinterpret_cast<uintptr_t>(weight) & 1u) ||
      (reinterpret_cast<uintptr_t>(target) & 7u) || (reinterpret_cast<uintptr_t>(bias) & 3u) ||
      (reinterpret_cast<uintptr_t>(partials) & 7u) ||
      (reinterpret_cast<uintptr_t>(target_logit) & 3u))
    return RLK_ERR_ALIGN;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) || workspace_bytes < p.total)
    return RLK_ERR_WORKSPACE;
  DeviceInfo dev;
  st = device_ready(&dev);
  if (st != RLK_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PartialsLaunch L;
  L.hidden = hidden;
  L.N = N;
  L.H = H;
  L.ld_hidden = ld_hidden;
  L.stage_h = p.stage_h;
  L.ldh = p.ldh;
  L.h_stage = reinterpret_cast<uint16_t*>(ws + p.off_h);
  L.weight = weight;
  L.w_rows = p.v_end - p.v_begin;
  L.ld_weight = ld_weight;
  L.stage_w = p.stage_w;
  L.ldw = p.ldw;
  L.w_stage = reinterpret_cast<uint16_t*>(ws + p.off_w);
  L.V = V;
  L.vps = p.vps;
  L.j0 = j0;
  L.j1 = j1;
  L.v_off = p.v_begin;
  L.bias = bias;
  L.target = target;
  L.tstride = target_stride;
  L.ms = reinterpret_cast<float2*>(partials);
  L.ld_ms = ld_partials;
  L.zt = target_logit;
  L.counter = reinterpret_cast<int*>(ws);
  return launch_partials(L, dev, static_cast<cudaStream_t>(stream));
}

rlk_status combine_shards_impl(int64_t N, int64_t V, const int64_t* target, int64_t target_stride,
                               int64_t num_shards, const int64_t* split_offsets,
                               const float* partials, int64_t ld_partials, int64_t shard_stride,
                               const float* target_logits, int64_t zt_stride, float* logp,
                               float* lse, float* target_logit, void* stream) {
  int64_t S, vps, vt;
  rlk_status st = rlk_vocab_split_policy(V, &S, &vps, &vt);
  if (st != RLK_OK) return st;
  if (N < 0 || N >= kMaxExtent || target_stride < 0 || num_shards < 1 ||
      num_shards > kMaxShards)
    return RLK_ERR_SHAPE;
  if (!split_offsets) return RLK_ERR_NULL;
  ShardedPartials src;
  if (split_offsets[0] != 0 || split_offsets[num_shards] != S) return RLK_ERR_SHAPE;
  int64_t widest = 0;
  for (int64_t q = 0; q < num_shards; ++q) {
    const int64_t n = split_offsets[q + 1] - split_offsets[q];
    if (n < 0) return RLK_ERR_SHAPE;
    widest = n > widest ? n : widest;
  }
  for (int64_t q = 0; q <= num_shards; ++q) src.off[q] = (int)split_offsets[q];
  // Unused slots repeat S, so a search for the shard of a split stops in range.
  for (int64_t q = num_shards + 1; q <= kMaxShards; ++q) src.off[q] = (int)S;
  if (ld_partials < widest || ld_partials >= (int64_t(1) << 31)) return RLK_ERR_SHAPE;
  if (N > 0 && (num_shards > 1 && (shard_stride < N * ld_partials || zt_stride < N)))
    return RLK_ERR_SHAPE;
  if (shard_stride < 0 || zt_stride < 0) return RLK_ERR_SHAPE;
  if (N == 0) return RLK_OK;
  if (!target || !partials || !target_logits || !logp || !lse) return RLK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(target) & 7u) || (reinterpret_cast<uintptr_t>(partials) & 7u) ||
      (reinterpret_cast<uintptr_t>(target_logits) & 3u) ||
      (reinterpret_cast<uintptr_t>(logp) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(target_logit) & 3u))
    return RLK_ERR_ALIGN;
  DeviceInfo dev;
  st = device_ready(&dev);
  if (st != RLK_OK) return st;
  src.ms = reinterpret_cast<const float2*>(partials);
  src.ld = ld_partials;
  src.shard_stride = shard_stride;
  src.zt = target_logits;
  src.zt_stride = zt_stride;
  src.vps = (int)vps;
  const int grid = (int)ceil_div(N, 256 / 32);
  const cudaError_t e = launch_overlapped(
      linear_logp_combine_kernel<ShardedPartials>, grid, 256, 0, static_cast<cudaStream_t>(stream),
      src, target, target_stride, (int)N, (int)S, (int)V, logp, lse, target_logit);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  return RLK_OK;
}

rlk_status linear_logp_impl(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                            const void* weight, int64_t V, int64_t ld_weight, const float* bias,
                            const int64_t* target, int64_t target_stride, float* logp, float* lse,
                            float* target_logit, int64_t splits_req, void* workspace,
                            size_t workspace_bytes, void* stream) {
  // Validate everything the second stage needs before the first one launches.
  if (N > 0 && (!logp || !lse)) return RLK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(logp) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(target_logit) & 3u))
    return RLK_ERR_ALIGN;
  rlk_status st = partials_impl(hidden, N, H, ld_hidden, weight, V, ld_weight, bias, target,
                                target_stride, splits_req, workspace, workspace_bytes, stream);
  if (st != RLK_OK) return st;
  return combine_impl(N, V, target, target_stride, logp, lse, target_logit, splits_req, workspace,
                      workspace_bytes, stream);
}

}  // namespace
}  // namespace rlk

extern "C" {

size_t rlk_linear_logp_workspace_size(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                                      const void* weight, int64_t V, int64_t ld_weight) {
  LogpPlan p;
  if (plan(hidden, N, H, ld_hidden, weight, V, ld_weight, 0, &p) != RLK_OK) return 0;
  return p.total;
}

rlk_status rlk_linear_logp_partials(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                                    const void* weight, int64_t V, int64_t ld_weight,
                                    const float* bias, const int64_t* target,
                                    int64_t target_stride, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  return partials_impl(hidden, N, H, ld_hidden, weight, V, ld_weight, bias, target, target_stride,
                       0, workspace, workspace_bytes, stream);
}

rlk_status rlk_linear_logp_combine(int64_t N, int64_t V, const int64_t* target,
                                   int64_t target_stride, float* logp, float* lse,
                                   float* target_logit, const void* workspace,
                                   size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  return combine_impl(N, V, target, target_stride, logp, lse, target_logit, 0, workspace,
                      workspace_bytes, stream);
}

rlk_status rlk_linear_logp(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                           const void* weight, int64_t V, int64_t ld_weight, const float* bias,
                           const int64_t* target, int64_t target_stride, float* logp, float* lse,
                           float* target_logit, void* workspace, size_t workspace_bytes,
                           void* stream) {
  RLK_CALL_RANGE();
  return linear_logp_impl(hidden, N, H, ld_hidden, weight, V, ld_weight, bias, target,
                          target_stride, logp, lse, target_logit, 0, workspace, workspace_bytes,
                          stream);
}

rlk_status rlk_debug_trace_read(uint64_t* out, int64_t max_ctas, int64_t* n_ctas) {
  return read_trace(out, max_ctas, n_ctas);
}

rlk_status rlk_throughput_split_count(int64_t N, int64_t V, int32_t sm_count,
                                      int64_t* num_splits) {
  if (!num_splits) return RLK_ERR_NULL;
  if (N < 1 || N >= kMaxExtent || V < 1 || V >= kMaxExtent || sm_count < 0)
    return RLK_ERR_SHAPE;
  if (sm_count == 0) {
    DeviceInfo dev;
    const rlk_status st = device_ready(&dev);
    if (st != RLK_OK) return st;
    sm_count = dev.sm_count;
  }
  const int64_t vtiles = ceil_div(V, kVocabTile);
  const int64_t row_blocks = ceil_div(N, 256);
  const int64_t pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
  const int64_t want = ceil_div(kOrderedMinRounds * pairs, row_blocks);
  *num_splits = want < vtiles ? want : vtiles;
  return RLK_OK;
}

rlk_status rlk_vocab_shard_range(int64_t V, int64_t num_shards, int64_t shard,
                                 int64_t* split_begin, int64_t* split_end, int64_t* v_begin,
                                 int64_t* v_end) {
  if (!split_begin || !split_end || !v_begin || !v_end) return RLK_ERR_NULL;
  int64_t S, vps, vt;
  const rlk_status st = rlk_vocab_split_policy(V, &S, &vps, &vt);
  if (st != RLK_OK) return st;
  if (num_shards < 1 || num_shards > kMaxShards || shard < 0 || shard >= num_shards)
    return RLK_ERR_SHAPE;
  const int64_t j0 = shard * S / num_shards, j1 = (shard + 1) * S / num_shards;
  const int64_t span = vps * kVocabTile;
  *split_begin = j0;
  *split_end = j1;
  *v_begin = j0 * span < V ? j0 * span : V;
  *v_end = j1 * span < V ? j1 * span : V;
  return RLK_OK;
}

size_t rlk_linear_logp_shard_workspace_size(const void* hidden, int64_t N, int64_t H,
                                            int64_t ld_hidden, const void* weight_shard,
                                            int64_t V, int64_t split_begin, int64_t split_end,
                                            int64_t ld_weight) {
  ShardPlan p;
  if (shard_plan(hidden, N, H, ld_hidden, weight_shard, V, split_begin, split_end, ld_weight,
                 &p) != RLK_OK)
    return 0;
  return p.total;
}

rlk_status rlk_linear_logp_shard_partials(const void* hidden, int64_t N, int64_t H,
                                          int64_t ld_hidden, const void* weight_shard, int64_t V,
                                          int64_t split_begin, int64_t split_end,
                                          int64_t ld_weight, const float* bias_shard,
                                          const int64_t* target, int64_t target_stride,
                                          float* partials, int64_t ld_partials,
                                          float* target_logit, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  return shard_partials_impl(hidden, N, H, ld_hidden, weight_shard, V, split_begin, split_end,
                             ld_weight, bias_shard, target, target_stride, partials, ld_partials,
                             target_logit, workspace, workspace_bytes, stream);
}

rlk_status rlk_linear_logp_combine_shards(int64_t N, int64_t V, const int64_t* target,
                                          int64_t target_stride, int64_t num_shards,
                                          const int64_t* split_offsets, const float* partials,
                                          int64_t ld_partials, int64_t shard_stride,
                                          const float* target_logits, int64_t zt_stride,
                                          float* logp, float* lse, float* target_logit,
                                          void* stream) {
  RLK_CALL_RANGE();
  return combine_shards_impl(N, V, target, target_stride, num_shards, split_offsets, partials,
                             ld_partials, shard_stride, target_logits, zt_stride, logp, lse,
                             target_logit, stream);
}

size_t rlk_linear_logp_splits_workspace_size(const void* hidden, int64_t N, int64_t H,
                                             int64_t ld_hidden, const void* weight, int64_t V,
                                             int64_t ld_weight, int64_t num_splits) {
  LogpPlan p;
  if (plan(hidden, N, H, ld_hidden, weight, V, ld_weight, num_splits, &p) != RLK_OK) return 0;
  return p.total;
}

rlk_status rlk_linear_logp_splits(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                                  const void* weight, int64_t V, int64_t ld_weight,
                                  const float* bias, const int64_t* target, int64_t target_stride,
                                  float* logp, float* lse, float* target_logit,
                                  int64_t num_splits, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  RLK_CALL_RANGE();
  return linear_logp_impl(hidden, N, H, ld_hidden, weight, V, ld_weight, bias, target,
                          target_stride, logp, lse, target_logit, num_splits, workspace,
                          workspace_bytes, stream);
}

}  // extern "C"

// ======================================================================
// Linear-logp without any caller-provided or library-allocated workspace.
//
// Some callers cannot allocate device memory at the point where they need this
// operator: a plugin running inside a host framework that owns the device
// allocator and offers no way to request scratch buffers, code under a device
// memory budget fixed in advance, or a latency-critical loop that must not call
// cudaMalloc / cudaFree because those calls can synchronise the device.  For
// them the partials live in one fixed, file-scope device array that is part of
// the library image: every GPU that loads this library holds these 32 MiB
// until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  Nothing in it has to start at zero: each call overwrites
// every partial it later reads, and a target logit is read only for rows whose
// target was written in the same call.  Calls whose GPU work overlaps (for
// example on two streams without ordering between them) use the same array and
// race; order them on one stream or with events.
namespace rlk {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;

// The cached device address of g_noalloc_scratch, per device, tagged with the
// unique id of the CUDA context it was looked up in: after cudaDeviceReset (or
// any release and re-creation of the primary context) the library's module is
// loaded again at a new address, so an address is reused only while the context
// that produced it is still the current one.
struct NoAllocSlot {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_noalloc_mutex;
NoAllocSlot g_noalloc_slot[kNoAllocMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Id of the context current on this thread (called with g_noalloc_mutex held).
rlk_status current_context_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return RLK_ERR_CUDA;
  if (ctx == nullptr) {
    // No context is current on this thread yet: the symbol lookup below makes
    // the device's primary context current (it allocates nothing).
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return RLK_ERR_CUDA;
  }
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? RLK_OK : RLK_ERR_CUDA;
}

// Host code cannot use g_noalloc_scratch's name as an address (on the host it
// names a stand-in object); the device address is looked up with the device
// current and cached until the current context changes.
rlk_status noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return RLK_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  unsigned long long id = 0;
  rlk_status st = current_context_id(&id);
  if (st != RLK_OK) return st;
  NoAllocSlot& slot = g_noalloc_slot[dev];
  if (slot.ptr == nullptr || slot.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    slot.ptr = p;
    slot.ctx_id = id;
  }
  *out = slot.ptr;
  return RLK_OK;
}

}  // namespace
}  // namespace rlk

extern "C" rlk_status rlk_linear_logp_noalloc(const void* hidden, int64_t N, int64_t H,
                                              int64_t ld_hidden, const void* weight, int64_t V,
                                              int64_t ld_weight, const float* bias,
                                              const int64_t* target, int64_t target_stride,
                                              float* logp, float* lse, float* target_logit,
                                              void* stream) {
  RLK_CALL_RANGE();
  const size_t need = rlk_linear_logp_workspace_size(hidden, N, H, ld_hidden, weight, V, ld_weight);
  if (need > rlk::kNoAllocScratchBytes) return RLK_ERR_WORKSPACE;
  if (N == 0 || need == 0)   // empty call, or arguments the regular entry point rejects
    return rlk_linear_logp(hidden, N, H, ld_hidden, weight, V, ld_weight, bias, target,
                           target_stride, logp, lse, target_logit, nullptr, 0, stream);
  rlk::DeviceInfo dev;
  rlk_status st = rlk::device_ready(&dev);
  if (st != RLK_OK) return st;
  void* scratch = nullptr;
  if ((st = rlk::noalloc_scratch(dev.device, &scratch)) != RLK_OK) return st;
  return rlk_linear_logp(hidden, N, H, ld_hidden, weight, V, ld_weight, bias, target,
                         target_stride, logp, lse, target_logit, scratch,
                         rlk::kNoAllocScratchBytes, stream);
}
