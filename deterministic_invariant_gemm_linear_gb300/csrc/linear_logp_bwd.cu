// Backward of the fused linear log-probability on sm_103a.
//
// Forward ("feat(linear-logp): add batch-invariant fused SM90 operator",
// Walkthrough): logp[r] = z[r, t_r] - lse[r], z = hidden . W^T (+ bias).  That
// page fails closed on backward ("outside the first contract"); this is the
// next step of the same path.  With an upstream gradient g[r] = dL/dlogp[r]:
//   G[r, v]        = dL/dz[r, v] = g[r] * ([v == t_r] - exp(z[r, v] - lse[r]))
//   grad_hidden    = G . W           (reduction over V in ascending order)
//   grad_weight    = G^T . hidden    (reduction over the N rows in ascending order)
//   grad_bias[v]   = sum_r G[r, v]   (ascending r)
//
// Stage 1 (linear_logp_grad_kernel): the same 2-SM tcgen05 loop as the forward
// recomputes each 256 x 256 logit tile (128 rows per CTA of the pair); the epilogue forms G in FP32 from the
// forward's lse and rounds it to BF16 (nearest even) into the workspace.  Rows
// are independent, so a row's G (hence its grad_hidden row) does not depend on
// the other rows in the call.
// Stage 2: grad_hidden and grad_weight are the deterministic GEMMs
// (rlk_det_gemm_fwd and rlk_det_gemm_db) on that BF16 G; grad_bias is a
// column sum of G in ascending row order.
#include <math.h>

#include <mutex>

#include <cuda_bf16.h>

#include "rlk.h"
#include "rlk_internal.h"
#include "rlk_pipeline.cuh"

namespace rlk {

__device__ unsigned int g_err_linear_logp_bwd = 0;

namespace {

struct GradSched {
  Banded order;    // rows = 256-row blocks (one per CTA pair), cols = 256-id vocabulary tiles
  int* counter;    // zeroed unit counter in the workspace (units in order), or null (round-robin)
  int nkb;         // reduction stages over H (64 or 128 wide)
  int nkb64;       // 64-wide blocks of H
  __device__ __forceinline__ int num_units() const { return order.count(); }
  __device__ __forceinline__ int unit_tiles(int) const { return 1; }
  __device__ __forceinline__ void tile_coords(int u, int, int& a0, int& b0) const {
    int rb, vt;
    order.unit(u, rb, vt);
    a0 = rb * kPairRows;
    b0 = vt * kBN;
  }
};

struct GradArgs {
  int N, V;
  int64_t tstride;
  const float* bias;
  bool bias_vec4;       // bias is 16-byte aligned: a lane reads its 8 floats as 2 vectors
  const int64_t* target;
  const float* lse;
  const float* grad;
  uint16_t* G;          // [N, ldG] BF16
  int64_t ldG;          // multiple of 8 elements
};

// kK: reduction elements per pipeline stage (64 or 128; see kWideStageRows).
template <int kK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    linear_logp_grad_kernel(const __grid_constant__ CUtensorMap tm_hidden,
                            const __grid_constant__ CUtensorMap tm_weight, GradSched sc,
                            GradArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const PipeSmem ps = pipe_smem(smem_raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_hidden);
    tma_prefetch_desc(&tm_weight);
  }
  const uint32_t tmem = pipe_setup(ps);
  using THalf = OperandTile<false, kHalfRows, kK>;
  using R = PairRingT<kHalfRows, kK>;

  if (warp == 0) {
    if (lane == 0)
      producer_role<THalf, THalf, GradSched, R>(&tm_hidden, &tm_weight, sc, ps,
                                                &g_err_linear_logp_bwd);
    if (lane == 1 && ps.rank == 0) scheduler_role(sc, ps, &g_err_linear_logp_bwd);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && ps.rank == 0)
      mma_role<THalf, THalf, GradSched, R>(sc, ps, tmem, idesc_bf16_f32(kPairRows, kBN, false, false),
                              &g_err_linear_logp_bwd);
    __syncwarp();
  } else {
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int k = 0;; ++k) {
      const int u = warp_unit_take(sc, ps, k, &g_err_linear_logp_bwd);
      if (u < 0) break;
      int r0, v0;
      sc.tile_coords(u, 0, r0, v0);
      const int row = r0 + (int)ps.rank * kHalfRows + q * 32 + lane;
      const bool valid = row < a.N;
      // the row's inputs and the tile's bias are read before the accumulator is
      // waited for, so their latency hides behind the MMAs
      int64_t t = -1;
      float g = 0.f, L = 0.f;
      if (valid) {
        t = __ldg(a.target + (int64_t)row * a.tstride);
        g = __ldg(a.grad + row);
        L = __ldg(a.lse + row);
      }
      const bool has_bias = a.bias != nullptr;
      BiasTile bias;
      if (has_bias) load_bias_tile(a.bias + v0, a.V - v0, a.bias_vec4, lane, bias);
      if (!epilogue_acquire(ps, acc, acc_phase, &g_err_linear_logp_bwd)) break;
      // A row whose target is outside [0, V) has no log-probability: zero gradient.
      const bool live = valid && t >= 0 && t < a.V;
      const uint32_t taddr = tmem + acc * kAccCols + lane_off;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        const int vbase = v0 + c * 32;
        if (vbase >= a.V) break;                 // uniform: depends on the tile only
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
        float G[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int v = vbase + i;
          float z = __uint_as_float(r[i]);
          if (has_bias) {
            const float b = bias_tile_at(bias, c, i);
            if (v < a.V) z = __fadd_rn(z, b);
          }
          const float p = ex2_approx(__fmul_rn(__fsub_rn(z, L), kLog2e));
          const float onehot = (int64_t)v == t ? 1.f : 0.f;
          G[i] = (live && v < a.V) ? __fmul_rn(g, __fsub_rn(onehot, p)) : 0.f;
        }
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(G[2 * i], G[2 * i + 1]);
            pk[i] = *reinterpret_cast<uint32_t*>(&b);
          }
          uint4* dst = reinterpret_cast<uint4*>(a.G + (int64_t)row * a.ldG + vbase);
#pragma unroll
          for (int k = 0; k < 4; ++k)   // 8 columns per store; groups past V stay within ldG
            if (vbase + 8 * k < a.V &&
                RLK_STORE_OK(row >= 0 && row < a.N && vbase + 8 * k + 8 <= a.ldG,
                             &g_err_linear_logp_bwd))
              dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      epilogue_release(ps, acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  pipe_teardown(tmem);
}

// grad_bias[v] = sum over rows r = 0..N-1 (ascending) of G[r, v], two columns per thread.
// The row loop is unrolled 64 deep so that many rows' loads are issued before their
// (still ascending) adds: 0.74 of HBM at the mid shape against 0.54 at depth 8.
__global__ void __launch_bounds__(256)
    column_sum_bf16_kernel(const uint16_t* __restrict__ G, int N, int V, int64_t ldG,
                           float* __restrict__ out) {
  griddep_wait();   // G is complete (the gradient kernels before this one have finished)
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int v = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (v >= V) return;
  float s0 = 0.f, s1 = 0.f;
  const uint32_t* p = reinterpret_cast<const uint32_t*>(G + v);
  const int64_t step = ldG / 2;
#pragma unroll 64
  for (int r = 0; r < N; ++r) {
    const uint32_t w = __ldg(p + (int64_t)r * step);
    s0 = __fadd_rn(s0, __uint_as_float(w << 16));
    s1 = __fadd_rn(s1, __uint_as_float(w & 0xffff0000u));
  }
  if (RLK_STORE_OK(v >= 0 && v < V, &g_err_linear_logp_bwd)) out[v] = s0;
  if (v + 1 < V && RLK_STORE_OK(v + 1 < V, &g_err_linear_logp_bwd)) out[v + 1] = s1;
}

std::mutex g_attr_mutex;
bool g_attr_set[64];

cudaError_t ensure_attrs(int dev) {
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(linear_logp_grad_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairRingT<kHalfRows, 64>::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(linear_logp_grad_kernel<128>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairRingT<kHalfRows, 128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_set[dev] = true;
  }
  return cudaSuccess;
}

inline int64_t grad_ld(int64_t V) { return ceil_div(V, 8) * 8; }

constexpr int64_t kLdLimit = int64_t(1) << 36;
constexpr int64_t kUnitLimit = int64_t(1) << 31;

// Workspace plan of the backward (each region 256-byte aligned):
// [G: N x ldG BF16][unit counter][padded copy of hidden][padded copy of W].
// hidden / W are copied (zero padded) only when TMA cannot read them in place;
// the copies hold the same values, so the results are bitwise the same.
struct BwdPlan {
  int64_t ldG = 0;
  bool stage_h = false, stage_w = false;
  int64_t ldh = 0, ldw = 0;      // pitches the kernels read
  size_t off_ctr = 0, off_h = 0, off_w = 0, total = 0;
};

rlk_status bwd_plan(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                    const void* weight, int64_t V, int64_t ld_weight, BwdPlan* p) {
  if (N < 0 || N >= kMaxExtent || H < 1 || H >= (int64_t(1) << 20) || V < 1 ||
      V >= kMaxExtent || ld_hidden < H || ld_weight < H || ld_hidden >= kLdLimit ||
      ld_weight >= kLdLimit)
    return RLK_ERR_SHAPE;
  // work-unit counts of the G kernel and of the two products, numbered in ints
  // (the products are checked for their narrower, 128-column tiles)
  const int64_t rb = ceil_div(N, kPairRows), vt = ceil_div(V, kBN), hb = ceil_div(H, kBN / 2);
  if (rb * vt >= kUnitLimit || rb * hb >= kUnitLimit || vt * hb >= kUnitLimit)
    return RLK_ERR_SHAPE;
  p->ldG = grad_ld(V);
  p->stage_h = N > 0 && !tma_ready(hidden, ld_hidden);
  p->stage_w = N > 0 && !tma_ready(weight, ld_weight);
  p->ldh = p->stage_h ? staged_ld(H) : ld_hidden;
  p->ldw = p->stage_w ? staged_ld(H) : ld_weight;
  size_t off = align_up((size_t)N * p->ldG * 2, 256);
  p->off_ctr = off;
  off += 256;
  p->off_h = off;
  if (p->stage_h) off = align_up(off + (size_t)N * p->ldh * 2, 256);
  p->off_w = off;
  if (p->stage_w) off = align_up(off + (size_t)V * p->ldw * 2, 256);
  p->total = off;
  return RLK_OK;
}

inline bool aligned_to(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace

uint32_t take_error_linear_logp_bwd() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_linear_logp_bwd, sizeof v) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaMemcpyToSymbol(g_err_linear_logp_bwd, &zero, sizeof zero);
  cudaGetLastError();
  return v;
}

}  // namespace rlk

using namespace rlk;

extern "C" {

size_t rlk_linear_logp_backward_workspace_size(int64_t N, int64_t V) {
  if (N < 0 || N >= kMaxExtent || V < 1 || V >= kMaxExtent) return 0;
  return align_up((size_t)N * grad_ld(V) * 2, 256) + 256;   // G, then the unit counter
}

size_t rlk_linear_logp_backward_workspace_size_for(const void* hidden, int64_t N, int64_t H,
                                                   int64_t ld_hidden, const void* weight,
                                                   int64_t V, int64_t ld_weight) {
  BwdPlan p;
  if (bwd_plan(hidden, N, H, ld_hidden, weight, V, ld_weight, &p) != RLK_OK) return 0;
  return p.total;
}

rlk_status rlk_linear_logp_backward(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                                    const void* weight, int64_t V, int64_t ld_weight,
                                    const float* bias, const int64_t* target,
                                    int64_t target_stride, const float* lse, const float* grad_logp,
                                    void* grad_hidden, int grad_hidden_dtype,
                                    int64_t ld_grad_hidden, void* grad_weight,
                                    int grad_weight_dtype, int64_t ld_grad_weight, float* grad_bias,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  RLK_CALL_RANGE();
  // ---- every check, including those of the products below, before the first launch
  BwdPlan p;
  rlk_status st = bwd_plan(hidden, N, H, ld_hidden, weight, V, ld_weight, &p);
  if (st != RLK_OK) return st;
  if (target_stride < 0) return RLK_ERR_SHAPE;
  if (grad_hidden && (ld_grad_hidden < H || ld_grad_hidden >= kLdLimit)) return RLK_ERR_SHAPE;
  if (grad_weight && (ld_grad_weight < H || ld_grad_weight >= kLdLimit)) return RLK_ERR_SHAPE;
  if ((grad_hidden && grad_hidden_dtype != RLK_BF16 && grad_hidden_dtype != RLK_FP32) ||
      (grad_weight && grad_weight_dtype != RLK_BF16 && grad_weight_dtype != RLK_FP32))
    return RLK_ERR_DTYPE;
  const size_t es_h = grad_hidden_dtype == RLK_FP32 ? 4 : 2;
  const size_t es_w = grad_weight_dtype == RLK_FP32 ? 4 : 2;
  if ((grad_hidden && !aligned_to(grad_hidden, es_h)) ||
      (grad_weight && !aligned_to(grad_weight, es_w)) || !aligned_to(grad_bias, 4))
    return RLK_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // No rows: grad_hidden is empty; grad_weight and grad_bias are the empty sums.
    if (!grad_weight && !grad_bias) return RLK_OK;
    DeviceInfo dev;
    st = device_ready(&dev);
    if (st != RLK_OK) return st;
    if (grad_weight &&
        cudaMemset2DAsync(grad_weight, ld_grad_weight * es_w, 0, H * es_w, V, s) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    if (grad_bias && cudaMemsetAsync(grad_bias, 0, V * sizeof(float), s) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
    return RLK_OK;
  }
  if (!hidden || !weight || !target || !lse || !grad_logp) return RLK_ERR_NULL;
  if (!aligned_to(hidden, 2) || !aligned_to(weight, 2) || !aligned_to(target, 8) ||
      !aligned_to(lse, 4) || !aligned_to(grad_logp, 4) || !aligned_to(bias, 4))
    return RLK_ERR_ALIGN;
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < p.total)
    return RLK_ERR_WORKSPACE;
  DeviceInfo dev;
  st = device_ready(&dev);
  if (st != RLK_OK) return st;
  if (ensure_attrs(dev.device) != cudaSuccess) return RLK_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const void* h_src = hidden;
  const void* w_src = weight;
  CUtensorMap tm_h, tm_w;
  // The tensor maps only describe addresses; encoding them launches nothing.
  if (p.stage_h) h_src = ws + p.off_h;
  if (p.stage_w) w_src = ws + p.off_w;
  if (!encode_bf16_2d(&tm_h, h_src, H, N, p.ldh, kBK, kHalfRows) ||
      !encode_bf16_2d(&tm_w, w_src, H, V, p.ldw, kBK, kHalfRows))
    return RLK_ERR_CUDA;
  if (p.stage_h &&
      launch_stage_bf16(static_cast<const uint16_t*>(hidden), N, H, ld_hidden,
                        reinterpret_cast<uint16_t*>(ws + p.off_h), p.ldh, s) != cudaSuccess)
    return RLK_ERR_CUDA;
  if (p.stage_w &&
      launch_stage_bf16(static_cast<const uint16_t*>(weight), V, H, ld_weight,
                        reinterpret_cast<uint16_t*>(ws + p.off_w), p.ldw, s) != cudaSuccess)
    return RLK_ERR_CUDA;

  GradSched sc;
  sc.order.rows = (int)ceil_div(N, kPairRows);
  sc.order.cols = (int)ceil_div(V, kBN);
  sc.order.band = band_rows(sc.order.rows, H, kPairRows);
  const int stage_k = N > kWideStageRows ? 128 : 64;   // as the forward's 2-SM loop
  sc.nkb = (int)ceil_div(H, stage_k);
  sc.nkb64 = (int)ceil_div(H, kBK);
  GradArgs a;
  a.N = (int)N;
  a.V = (int)V;
  a.tstride = target_stride;
  a.bias = bias;
  a.bias_vec4 = aligned_to(bias, 16);
  a.target = target;
  a.lse = lse;
  a.grad = grad_logp;
  a.G = reinterpret_cast<uint16_t*>(ws);
  a.ldG = p.ldG;
  const int64_t units = (int64_t)sc.order.rows * sc.order.cols;
  const int64_t clusters = dev.sm_count / 2;
  const int grid = 2 * (int)(units < clusters ? units : clusters);
  sc.counter = nullptr;
  if (ordered_units(units, clusters)) {
    sc.counter = reinterpret_cast<int*>(ws + p.off_ctr);
    if (cudaMemsetAsync(sc.counter, 0, sizeof(int), s) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
  }
  if ((stage_k == 128
           ? launch_overlapped(linear_logp_grad_kernel<128>, grid, kThreads,
                               PairRingT<kHalfRows, 128>::kSmemBytes, s, tm_h, tm_w, sc, a)
           : launch_overlapped(linear_logp_grad_kernel<64>, grid, kThreads,
                               PairRingT<kHalfRows, 64>::kSmemBytes, s, tm_h, tm_w, sc, a)) !=
      cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }

  // The products read G and the (possibly staged) operands, all TMA-ready, so
  // they need no workspace and every argument they check was checked above.
  // Both requested and the longer-reduction product's 256 x 256 tiles fill at
  // most half of the SM pairs: one launch over both products' tiles, so the
  // short tiles use the pairs the long ones leave idle (same bits as two
  // launches).  Measured on GB300 at H = 4096, V = 151,936: N = 512 1.37 vs
  // 1.67 ms; with a wave or more of long tiles the two products running side by
  // side were 3 - 4% slower (N = 1024, 2048) or level (N = 4096), so there they
  // stay apart.
  const int64_t long_tiles = ceil_div(V >= N ? N : V, kPairRows) * ceil_div(H, kBN);
  const bool one_launch = 2 * long_tiles <= dev.sm_count / 2;
  if (grad_hidden && grad_weight && one_launch) {
    st = launch_fwd_and_db(a.G, N, V, a.ldG, w_src, H, p.ldw, grad_hidden, grad_hidden_dtype,
                           ld_grad_hidden, h_src, p.ldh, grad_weight, grad_weight_dtype,
                           ld_grad_weight, reinterpret_cast<int*>(ws + p.off_ctr), s);
    if (st != RLK_OK) return st;
  } else {
    if (grad_hidden) {   // [N, H] = G [N, V] . W [V, H]
      st = rlk_det_gemm_fwd(a.G, N, V, a.ldG, w_src, H, p.ldw, grad_hidden, grad_hidden_dtype,
                            ld_grad_hidden, nullptr, 0, stream);
      if (st != RLK_OK) return st;
    }
    if (grad_weight) {   // [V, H] = G^T . hidden
      st = rlk_det_gemm_db(a.G, N, V, a.ldG, h_src, RLK_BF16, H, p.ldh, grad_weight,
                           grad_weight_dtype, ld_grad_weight, nullptr, 0, stream);
      if (st != RLK_OK) return st;
    }
  }
  if (grad_bias) {
    const int threads = 256;
    const int grid_b = (int)ceil_div(ceil_div(V, 2), threads);
    if (launch_overlapped(column_sum_bf16_kernel, grid_b, threads, 0, s, a.G, (int)N, (int)V,
                          a.ldG, grad_bias) != cudaSuccess) {
      cudaGetLastError();
      return RLK_ERR_CUDA;
    }
  }
  return RLK_OK;
}

}  // extern "C"
