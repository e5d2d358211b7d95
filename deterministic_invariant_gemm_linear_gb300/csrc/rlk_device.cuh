// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (TMEM allocation, BF16 MMA, commit, loads)
// and the shared-memory / instruction descriptors the MMA consumes.
//
// Everything here is inline PTX written against the PTX ISA's tcgen05,
// cp.async.bulk.tensor and mbarrier sections.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rlk {

// ---------------------------------------------------------------- tile shape
// A pair of CTAs (a cluster of two, one per SM) owns one 256 x 256 FP32
// accumulator tile per MMA chain, 128 rows in each CTA's TMEM; the reduction
// advances in blocks of 64 BF16 (128 bytes = one 128B-swizzle row).
constexpr int kHalfRows = 128;     // accumulator rows (TMEM lanes) per CTA; operand rows per CTA
constexpr int kPairRows = 2 * kHalfRows;      // accumulator rows per CTA pair (MMA M)
constexpr int kBN = 256;           // accumulator columns (TMEM columns, MMA N)
constexpr int kBK = 64;            // reduction elements per TMA box row (one swizzle atom); a stage holds 64 or 128
constexpr int kUmmaK = 16;         // reduction per tcgen05.mma (kind::f16)
constexpr int kAccCols = kBN;      // FP32 accumulator columns per buffer
constexpr int kTmemCols = 2 * kAccCols;       // double-buffered accumulator: 512 columns
constexpr int kThreads = 192;      // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpilogueThreads = 128;

// Bounded waits: a wait that has not completed after this long gives up,
// raises the device error word and makes the CTA wind down.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s
constexpr uint32_t kDevErrTimeout = 0x1u;
constexpr uint32_t kDevErrBounds = 0x2u;

// Store checks of the debug build (-DRLK_DEBUG): every global store first tests
// its index against the extent of the buffer it writes; a store outside raises
// kDevErrBounds in the error word and is skipped (nothing traps).  Release builds
// compile the test away.
#ifdef RLK_DEBUG
__device__ __forceinline__ bool store_in_bounds(bool ok, unsigned int* err) {
  if (!ok) atomicOr(err, kDevErrBounds);
  return ok;
}
#define RLK_STORE_OK(cond, err) (::rlk::store_in_bounds((cond), (err)))
#else
#define RLK_STORE_OK(cond, err) true
#endif

__device__ __forceinline__ uint64_t globaltimer_ns();

// Phase timestamps of the debug build: field f of this CTA's record takes the
// current %globaltimer (a later mark of the same field overwrites it).  Each
// translation unit has its own table; the linear-logp one is read back by
// rlk_debug_trace_read.  Release builds compile the marks away.
// Fields 6 and 7 hold the SM's cycle counter (clock64) at entry and exit, so that
// cycles / elapsed ns gives the clock the CTA actually ran at.  Fields 8 - 15 are
// the roles' cycle counters (kTraceMma... below), each written once when its role
// finishes.  RLK_CYCLES() reads the cycle counter in the debug build and is the
// constant 0 in release builds, where the counter arithmetic folds away.
constexpr int kTraceFields = 16;
constexpr int kTraceCtas = 1024;
constexpr int kTraceMmaOperandWait = 8;    // MMA issuer: cycles waiting for operand stages
constexpr int kTraceMmaAccWait = 9;        // MMA issuer: cycles waiting for a free accumulator
constexpr int kTraceMmaCycles = 10;        // MMA issuer: cycles from its first unit to its last MMA
constexpr int kTraceMmaTiles = 11;         // MMA issuer: accumulator tiles issued
constexpr int kTraceLoadSlotWait = 12;     // producer: cycles waiting for free ring slots
constexpr int kTraceLoadCycles = 13;       // producer: cycles from its first unit to its last copy
constexpr int kTraceEpiAccWait = 14;       // epilogue thread 64: cycles waiting for accumulators
constexpr int kTraceEpiWork = 15;          // epilogue thread 64: cycles reading and folding them
#ifdef RLK_DEBUG
static __device__ unsigned long long g_trace[kTraceCtas * kTraceFields];
__device__ __forceinline__ void trace_mark(int field) {
  if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x * kTraceFields + field] = globaltimer_ns();
}
__device__ __forceinline__ void trace_cycles(int field) {
  if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x * kTraceFields + field] = clock64();
}
__device__ __forceinline__ void trace_set(int field, long long v) {
  if (blockIdx.x < kTraceCtas) g_trace[blockIdx.x * kTraceFields + field] = (unsigned long long)v;
}
#define RLK_TRACE(field) ::rlk::trace_mark(field)
#define RLK_TRACE_CYCLES(field) ::rlk::trace_cycles(field)
#define RLK_TRACE_SET(field, v) ::rlk::trace_set((field), (v))
#define RLK_CYCLES() ((long long)clock64())
#else
#define RLK_TRACE(field) ((void)0)
#define RLK_TRACE_CYCLES(field) ((void)0)
#define RLK_TRACE_SET(field, v) ((void)(v))
#define RLK_CYCLES() 0ll
#endif

// The bias values of one 256-id vocabulary tile spread over a warp: lane l holds
// entries 8 l .. 8 l + 7 of the tile (0 past its n valid entries).  An epilogue
// warp loads a tile's values once, before it waits for the tile's accumulator, so
// the loads' latency hides behind the MMAs instead of stalling every 32-column
// chunk; each column's value then comes from its lane by shuffle.  vec4: the tile
// start is 16-byte aligned (a lane reads its 8 values as two vectors).
struct BiasTile {
  float q[8];
};

__device__ __forceinline__ void load_bias_tile(const float* tile, int n, bool vec4, int lane,
                                               BiasTile& b) {
  const int e = 8 * lane;
  if (vec4 && e + 8 <= n) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(tile + e));
    const float4 y = __ldg(reinterpret_cast<const float4*>(tile + e) + 1);
    b.q[0] = x.x;
    b.q[1] = x.y;
    b.q[2] = x.z;
    b.q[3] = x.w;
    b.q[4] = y.x;
    b.q[5] = y.y;
    b.q[6] = y.z;
    b.q[7] = y.w;
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      b.q[k] = 0.f;
      if (e + k < n) b.q[k] = __ldg(tile + e + k);
    }
  }
}

// Entry 32 c + i of the tile (i a compile-time index in an unrolled loop); every
// lane of the warp must take part.
__device__ __forceinline__ float bias_tile_at(const BiasTile& b, int c, int i) {
  return __shfl_sync(0xffffffffu, b.q[i & 7], 4 * c + (i >> 3));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Programmatic dependent launch.  griddep_wait blocks until the kernel before
// this one in the stream has completed and its memory is visible (it returns at
// once for an ordinary launch); griddep_launch_dependents lets the next kernel,
// if launched with programmatic serialisation, start its own prologue.  Every
// library kernel runs its prologue (barriers, TMEM, descriptor prefetch) and
// waits before it reads or writes global memory; the tensor-core kernels signal
// once their producer has run out of work, the short kernels right away.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of parity `parity` to complete.  Returns false when the
// CTA is winding down (abort flag set by another role) or when this wait ran
// past timeout_ns (kWaitTimeoutNs unless given); in the latter case it sets the abort flag and ORs
// kDevErrTimeout into *err.  Every wait ends: either the phase completes, the
// abort flag is seen, or the time limit passes (with a hard cap on polls as a
// second bound).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err,
                                          uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns || n > (1u << 30)) {
        *abort_flag = 1;
        atomicOr(err, kDevErrTimeout);
        return false;
      }
    }
  }
}

// A wait used only while winding down: bounded by the same limit, ignores the
// abort flag (its purpose is to let in-flight asynchronous work land).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned int* err) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 31u && (globaltimer_ns() - t0 > kWaitTimeoutNs || n > (1u << 30))) {
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, BF16 inputs, FP32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive FP32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- work order
// Grouped order of a 2-D grid of work units (rows x cols): units are dealt in
// bands of `band` consecutive row blocks; inside a band the row block varies
// fastest, then the column.  CTAs that run at the same time then share a band's
// row operands and a few columns' operands in L2.  The order decides only which
// CTA computes a unit, never how.
struct Banded {
  int rows;    // row blocks
  int cols;    // column blocks (vocabulary splits / tiles, output column blocks)
  int band;    // row blocks per band (>= 1)
  __device__ __forceinline__ int count() const { return rows * cols; }
  __device__ __forceinline__ void unit(int u, int& row, int& col) const {
    const int full = band * cols;
    const int b = u / full;
    const int r0 = b * band;
    const int n = min(band, rows - r0);
    const int rem = u - b * full;
    col = rem / n;
    row = r0 + (rem - col * n);
  }
};

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bit 46, and the
// 128-byte swizzle layout (value 2) in bits 61..63.  Base offset 0: every
// swizzle atom used here starts on a 1024-byte boundary.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16: FP32 accumulator (bits 4-5 = 1), BF16
// A and B (bits 7-9 and 10-12 = 1), operand majorness (bit 15 for A, bit 16
// for B: 0 = K-major, 1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Operand staging for one pipeline stage.
//  K-major operand (rows x 64 reduction elements): one TMA box {64, rows},
//    rows 128 bytes apart, 8-row swizzle atoms 1024 bytes apart (SBO); the MMA's
//    16-element reduction step advances the start address by 32 bytes inside
//    the swizzle atom.
//  MN-major operand (64 reduction rows x rows contiguous elements): boxes of
//    {64 contiguous, 64 reduction}, each 8 KiB, placed one after another along
//    the MN extent (LBO = 8 KiB between 64-element MN atoms); reduction rows are
//    128 bytes apart with 8-row groups 1024 bytes apart (SBO); the 16-element
//    reduction step advances the start address by 2 groups = 2048 bytes.
// 2-D tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of a cluster pair (`cta_group::2`).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t mbar,
                                                 int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar), "r"(c0), "r"(c1)
      : "memory");
}

// kStageK: reduction elements per stage, 64 (one 128-byte swizzle atom per row)
// or 128.  A 128-deep K-major stage is two 64-wide boxes side by side (each row
// of a box is one 128-byte swizzle row), the MMA descriptors stepping into the
// second box after four 16-element steps; an MN-major stage's 64-element chunks
// are 64 x kStageK x 2 bytes apart.  The stage depth changes only how the same
// 16-element MMAs are grouped, never which run or their order.
template <bool kMN, int kRows, int kStageK = kBK>
struct OperandTile {
  static_assert(kStageK == 64 || kStageK == 128, "stages of 64 or 128 reduction elements");
  static constexpr int kK = kStageK;
  static constexpr uint32_t kBytes = kRows * kStageK * 2;
  // kPair: the copies complete on a barrier that may live in the pair's other CTA.
  template <bool kPair = false>
  static __device__ __forceinline__ void load(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int32_t row0, int32_t k0) {
    if constexpr (!kMN) {
#pragma unroll
      for (int i = 0; i < kStageK / 64; ++i) {
        if constexpr (kPair) tma_load_2d_pair(dst + i * (kRows * 128), map, bar, k0 + 64 * i, row0);
        else tma_load_2d(dst + i * (kRows * 128), map, bar, k0 + 64 * i, row0);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRows / 64; ++i) {
        if constexpr (kPair) tma_load_2d_pair(dst + i * (64 * kStageK * 2), map, bar, row0 + 64 * i, k0);
        else tma_load_2d(dst + i * (64 * kStageK * 2), map, bar, row0 + 64 * i, k0);
      }
    }
  }
  static __device__ __forceinline__ uint64_t desc(uint32_t base, int kstep) {
    if constexpr (!kMN) {
      return sdesc_sw128(base + static_cast<uint32_t>(kstep / 4) * (kRows * 128u) +
                             32u * static_cast<uint32_t>(kstep % 4),
                         16u, 1024u);
    } else {
      return sdesc_sw128(base + 2048u * kstep, 64u * kStageK * 2u, 1024u);
    }
  }
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace rlk
