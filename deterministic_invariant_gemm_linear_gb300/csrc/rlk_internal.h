// Host-side helpers shared by the rlk translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "rlk.h"

namespace rlk {

// Names a C-ABI call in profiler timelines: an NVTX range around the call (the
// kernels it launches fall inside it; `ncu --nvtx --nvtx-include "<name>/"`
// selects them).  Without an attached tool NVTX calls return at once.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define RLK_CALL_RANGE() ::rlk::CallRange rlk_call_range_(__func__)

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
};

// Checks that a CUDA device is current and is sm_103 (cached per device).
rlk_status device_ready(DeviceInfo* info);

// 2-D BF16 tensor map with 128-byte swizzle; zero fill outside the tensor.
// inner = contiguous extent (elements), outer = row count, ld = row pitch
// (elements).  Returns false when the CUDA driver rejects the description.
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t ld, uint32_t box_inner, uint32_t box_outer);

// Launches `kernel` with programmatic stream serialisation: it may begin while
// the previous kernel in the stream is finishing, and must call griddep_wait()
// (rlk_device.cuh) before it touches global memory that kernel may use.
template <class... KArgs, class... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Largest accepted row / column / vocabulary extent (exclusive): kernels index
// rows and ids in 32-bit ints, and the last index of a 256-wide block (and a
// 32-wide chunk's end) must stay below 2^31.
constexpr int64_t kMaxExtent = (int64_t(1) << 31) - 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// A BF16 operand can be read by TMA in place when its base is 16-byte aligned
// and its row pitch is a multiple of 16 bytes.
inline bool tma_ready(const void* p, int64_t ld) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (ld % 8) == 0;
}
// Padded pitch of a staged copy: the column count rounded up to 8 elements.
inline int64_t staged_ld(int64_t cols) { return ceil_div(cols, 8) * 8; }

// Copies rows x cols BF16 from src (pitch ld_src) to dst (pitch ld_dst),
// writing zeros into columns [cols, ld_dst).
cudaError_t launch_stage_bf16(const uint16_t* src, int64_t rows, int64_t cols, int64_t ld_src,
                              uint16_t* dst, int64_t ld_dst, cudaStream_t stream);

// Rounds rows x cols FP32 to BF16 (nearest even) into dst (pitch ld_dst),
// zero-filling columns [cols, ld_dst).
cudaError_t launch_cast_f32_bf16(const float* src, int64_t rows, int64_t cols, int64_t ld_src,
                                 uint16_t* dst, int64_t ld_dst, cudaStream_t stream);

// Row blocks per band of the work order: as many 128-row blocks of a
// K-element BF16 row operand as fit in 32 MiB of L2 (at least 1, at most rows).
inline int band_rows(int64_t rows, int64_t K, int64_t rows_per_block = 128) {
  const int64_t per = rows_per_block * K * 2;
  int64_t b = (int64_t(32) << 20) / (per > 0 ? per : 1);
  if (b < 1) b = 1;
  if (b > rows) b = rows;
  return (int)(b > 0 ? b : 1);
}

// Whether a persistent launch hands its units out in order from a counter in
// the workspace (zeroed before the launch) or deals them round-robin.  Over
// many rounds round-robin clusters drift apart and their operand tiles stop
// sharing L2; a launch of a few rounds cannot drift far, and skips the zeroing.
// Either way only which cluster computes a unit changes, never its arithmetic.
constexpr int64_t kOrderedMinRounds = 8;
inline bool ordered_units(int64_t units, int64_t clusters) {
  return units > kOrderedMinRounds * clusters;
}

// Vocabulary split policy (function of V only).
constexpr int64_t kVocabTile = 256;
constexpr int64_t kMaxVocabSplits = 1024;

// grad_hidden-style and grad_weight-style products of one BF16 G in one launch
// (det_gemm.cu): out1 [N, H] = G [N, V] . W [V, H] and out2 [V, H] = G^T . hidden
// [N, H], with every tile computed as by rlk_det_gemm_fwd / rlk_det_gemm_db (same
// bits).  All operands TMA-ready and all arguments validated by the caller;
// `counter` is a 4-byte slot of device memory the launch zeroes and uses.
rlk_status launch_fwd_and_db(const void* G, int64_t N, int64_t V, int64_t ldG, const void* W,
                             int64_t H, int64_t ldw, void* out1, int dt1, int64_t ld1,
                             const void* hidden, int64_t ldh, void* out2, int dt2, int64_t ld2,
                             int* counter, cudaStream_t s);

// The general form: out1 [rows1, cols1] = A1 [rows1, red1] (K-major) . B1, with B1
// [red1, cols1] row-major (b1_mn: the forward configuration) or [cols1, red1]
// row-major (the dA configuration); out2 [rows2, cols2] = A2^T . B2 with A2
// [red2, rows2] and B2 [red2, cols2] row-major (the dB configuration).  Each
// product's tiles are computed exactly as by its own det_gemm launch.
struct TwoProductArgs {
  const void* a1 = nullptr;
  int64_t lda1 = 0;
  const void* b1 = nullptr;
  int64_t ldb1 = 0;
  bool b1_mn = true;
  int64_t rows1 = 0, cols1 = 0, red1 = 0;
  const void* a2 = nullptr;
  int64_t lda2 = 0;
  const void* b2 = nullptr;
  int64_t ldb2 = 0;
  int64_t rows2 = 0, cols2 = 0, red2 = 0;
  void* out1 = nullptr;
  int dt1 = 0;
  int64_t ld1 = 0;
  void* out2 = nullptr;
  int dt2 = 0;
  int64_t ld2 = 0;
};
rlk_status launch_two_products(const TwoProductArgs& p, int* counter, cudaStream_t s);

// Per-translation-unit device error words: read-and-clear after a stream sync.
uint32_t take_error_linear_logp();
uint32_t take_error_det_gemm();
uint32_t take_error_common();
uint32_t take_error_linear_logp_bwd();

}  // namespace rlk
