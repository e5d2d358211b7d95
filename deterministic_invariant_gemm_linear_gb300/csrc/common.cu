// Shared host logic of the rlk library: status strings, the device check,
// TMA descriptor encoding, the vocabulary split policy, operand staging
// kernels and the device error word.
#include <mutex>

#include <cuda_bf16.h>

#include "rlk.h"
#include "rlk_device.cuh"
#include "rlk_internal.h"

namespace rlk {

__device__ unsigned int g_err_common = 0;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mutex;
EncodeTiledFn g_encode = nullptr;
constexpr int kMaxDevices = 64;
int g_dev_state[kMaxDevices];      // 0 unknown, 1 ready, -1 unsupported
int g_dev_sms[kMaxDevices];

EncodeTiledFn get_encode() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

}  // namespace

rlk_status device_ready(DeviceInfo* info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return RLK_ERR_UNSUPPORTED_DEVICE;
  }
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev_state[dev] == 0) {
      int major = 0, minor = 0, sms = 0;
      bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ==
                    cudaSuccess &&
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) ==
                    cudaSuccess &&
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
      cudaGetLastError();
      // the 2-SM kernels need at least one pair of SMs (and divide work by pairs)
      g_dev_state[dev] = (ok && major == 10 && minor == 3 && sms >= 2) ? 1 : -1;
      g_dev_sms[dev] = sms;
    }
    if (g_dev_state[dev] != 1) return RLK_ERR_UNSUPPORTED_DEVICE;
    info->device = dev;
    info->sm_count = g_dev_sms[dev];
  }
  if (!get_encode()) return RLK_ERR_CUDA;
  return RLK_OK;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- staging kernels
namespace {

// Rows are dealt to blocks (blockIdx.y, then in steps of gridDim.y) and each row's
// columns to consecutive threads, so loads and stores are coalesced and no index
// is divided.  Columns [cols, ld_dst) of dst are zero.
__global__ void stage_bf16_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                                  int64_t ld_src, uint16_t* __restrict__ dst, int64_t ld_dst) {
  const int64_t c0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t cstep = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const uint16_t* s = src + r * ld_src;
    uint16_t* d = dst + r * ld_dst;
    for (int64_t c = c0; c < ld_dst; c += cstep)
      if (RLK_STORE_OK(r * ld_dst + c < rows * ld_dst, &g_err_common))
        d[c] = c < cols ? s[c] : (uint16_t)0;
  }
}

__global__ void cast_f32_bf16_kernel(const float* __restrict__ src, int64_t rows, int64_t cols,
                                     int64_t ld_src, uint16_t* __restrict__ dst, int64_t ld_dst) {
  const int64_t c0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t cstep = (int64_t)gridDim.x * blockDim.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const float* s = src + r * ld_src;
    uint16_t* d = dst + r * ld_dst;
    for (int64_t c = c0; c < ld_dst; c += cstep) {
      uint16_t v = 0;
      if (c < cols) {
        __nv_bfloat16 b = __float2bfloat16_rn(s[c]);
        v = *reinterpret_cast<uint16_t*>(&b);
      }
      if (RLK_STORE_OK(r * ld_dst + c < rows * ld_dst, &g_err_common)) d[c] = v;
    }
  }
}

// The same copies, 8 columns per thread: dst rows are 16-byte aligned (a pitch of
// a multiple of 8 elements from a 16-byte aligned base, as every staged operand's
// is), so each thread writes one 16-byte vector; it reads its 8 source elements
// as independent loads (two 16-byte vectors for an aligned FP32 source), so a
// warp keeps several times more bytes in flight than one element per thread.
__device__ __forceinline__ uint32_t pack2(uint16_t lo, uint16_t hi) {
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__global__ void stage_bf16_vec8_kernel(const uint16_t* __restrict__ src, int64_t rows,
                                       int64_t cols, int64_t ld_src, uint16_t* __restrict__ dst,
                                       int64_t ld_dst) {
  const int64_t c0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 8;
  const int64_t cstep = (int64_t)gridDim.x * blockDim.x * 8;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const uint16_t* s = src + r * ld_src;
    uint16_t* d = dst + r * ld_dst;
    for (int64_t c = c0; c < ld_dst; c += cstep) {
      uint16_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[k] = 0;
        if (c + k < cols) v[k] = s[c + k];
      }
      if (RLK_STORE_OK(r * ld_dst + c + 8 <= rows * ld_dst, &g_err_common))
        *reinterpret_cast<uint4*>(d + c) =
            make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    }
  }
}

__global__ void cast_f32_bf16_vec8_kernel(const float* __restrict__ src, int64_t rows,
                                          int64_t cols, int64_t ld_src, int src_vec4,
                                          uint16_t* __restrict__ dst, int64_t ld_dst) {
  const int64_t c0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 8;
  const int64_t cstep = (int64_t)gridDim.x * blockDim.x * 8;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const float* s = src + r * ld_src;
    uint16_t* d = dst + r * ld_dst;
    for (int64_t c = c0; c < ld_dst; c += cstep) {
      float f[8];
      if (src_vec4 && c + 8 <= cols) {
        const float4 x = *reinterpret_cast<const float4*>(s + c);
        const float4 y = *reinterpret_cast<const float4*>(s + c + 4);
        f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
        f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          f[k] = 0.f;
          if (c + k < cols) f[k] = s[c + k];
        }
      }
      uint16_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        __nv_bfloat16 b = __float2bfloat16_rn(f[k]);
        v[k] = c + k < cols ? *reinterpret_cast<uint16_t*>(&b) : (uint16_t)0;
      }
      if (RLK_STORE_OK(r * ld_dst + c + 8 <= rows * ld_dst, &g_err_common))
        *reinterpret_cast<uint4*>(d + c) =
            make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    }
  }
}

bool dst_vec8(const uint16_t* dst, int64_t ld_dst) {
  return (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 && ld_dst % 8 == 0;
}

// Blocks of 256 threads: enough column blocks to cover a row's `units` (elements,
// or groups of 8) once (at most 64), and row blocks so that about 4096 blocks run
// (at most 65535, the y limit).
dim3 stage_grid(int64_t rows, int64_t units) {
  int64_t gx = ceil_div(units, 256);
  gx = gx < 1 ? 1 : (gx > 64 ? 64 : gx);
  int64_t gy = ceil_div(4096, gx);
  gy = gy > rows ? rows : gy;
  gy = gy < 1 ? 1 : (gy > 65535 ? 65535 : gy);
  return dim3((unsigned)gx, (unsigned)gy, 1);
}

}  // namespace

cudaError_t launch_stage_bf16(const uint16_t* src, int64_t rows, int64_t cols, int64_t ld_src,
                              uint16_t* dst, int64_t ld_dst, cudaStream_t stream) {
  if (dst_vec8(dst, ld_dst))
    stage_bf16_vec8_kernel<<<stage_grid(rows, ceil_div(ld_dst, 8)), 256, 0, stream>>>(
        src, rows, cols, ld_src, dst, ld_dst);
  else
    stage_bf16_kernel<<<stage_grid(rows, ld_dst), 256, 0, stream>>>(src, rows, cols, ld_src, dst,
                                                                    ld_dst);
  return cudaGetLastError();
}

cudaError_t launch_cast_f32_bf16(const float* src, int64_t rows, int64_t cols, int64_t ld_src,
                                 uint16_t* dst, int64_t ld_dst, cudaStream_t stream) {
  if (dst_vec8(dst, ld_dst)) {
    const int src_vec4 = (reinterpret_cast<uintptr_t>(src) & 15u) == 0 && ld_src % 4 == 0;
    cast_f32_bf16_vec8_kernel<<<stage_grid(rows, ceil_div(ld_dst, 8)), 256, 0, stream>>>(
        src, rows, cols, ld_src, src_vec4, dst, ld_dst);
  } else {
    cast_f32_bf16_kernel<<<stage_grid(rows, ld_dst), 256, 0, stream>>>(src, rows, cols, ld_src,
                                                                       dst, ld_dst);
  }
  return cudaGetLastError();
}

// One thread waits on a shared-memory mbarrier that nothing ever arrives on,
// through the same bounded wait the tensor-core kernels use: the wait gives up
// after timeout_ns, raises the error word and the kernel returns.
__global__ void selftest_wait_kernel(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
    (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_err_common, timeout_ns);
  }
}

// Debug builds only: one thread declares a store outside its buffer through the
// debug store check, which records kDevErrBounds and skips the store (no memory
// is written at all).
__global__ void selftest_store_check_kernel(unsigned int* never_written) {
  if (threadIdx.x == 0 && RLK_STORE_OK(false, &g_err_common)) *never_written = 1u;
}

uint32_t take_error_common() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_common, sizeof v) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaMemcpyToSymbol(g_err_common, &zero, sizeof zero);
  cudaGetLastError();
  return v;
}

}  // namespace rlk

// ====================================================================== C ABI
extern "C" {

const char* rlk_status_string(int status) {
  switch (status) {
    case RLK_OK: return "RLK_OK";
    case RLK_ERR_NULL: return "RLK_ERR_NULL: a required pointer is NULL";
    case RLK_ERR_SHAPE: return "RLK_ERR_SHAPE: a size or leading dimension is out of range";
    case RLK_ERR_DTYPE: return "RLK_ERR_DTYPE: unsupported dtype";
    case RLK_ERR_ALIGN: return "RLK_ERR_ALIGN: pointer not aligned to its element size";
    case RLK_ERR_WORKSPACE: return "RLK_ERR_WORKSPACE: workspace missing or too small";
    case RLK_ERR_UNSUPPORTED_DEVICE:
      return "RLK_ERR_UNSUPPORTED_DEVICE: no CUDA device, or the device is not sm_103";
    case RLK_ERR_CUDA: return "RLK_ERR_CUDA: the CUDA runtime rejected a call";
    case RLK_ERR_TIMEOUT: return "RLK_ERR_TIMEOUT: a kernel wait expired";
    case RLK_ERR_BOUNDS:
      return "RLK_ERR_BOUNDS: a debug-build kernel skipped a store outside its buffer";
    case RLK_ERR_NOT_DEBUG_BUILD:
      return "RLK_ERR_NOT_DEBUG_BUILD: the call needs the debug build of the library";
    default: return "RLK_ERR_UNKNOWN";
  }
}

int rlk_numerics_version(void) { return RLK_NUMERICS_VERSION; }

rlk_status rlk_device_check(void) {
  rlk::DeviceInfo info;
  return rlk::device_ready(&info);
}

rlk_status rlk_get_device_error(void* stream, uint32_t* flags) {
  if (!flags) return RLK_ERR_NULL;
  *flags = 0;
  rlk::DeviceInfo info;
  rlk_status st = rlk::device_ready(&info);
  if (st != RLK_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return RLK_ERR_CUDA;
  }
  *flags = rlk::take_error_linear_logp() | rlk::take_error_det_gemm() | rlk::take_error_common() |
           rlk::take_error_linear_logp_bwd();
  if (*flags & RLK_DEVERR_TIMEOUT) return RLK_ERR_TIMEOUT;
  return *flags ? RLK_ERR_BOUNDS : RLK_OK;
}

rlk_status rlk_selftest_bounded_wait(uint32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 2000000u) return RLK_ERR_SHAPE;
  rlk::DeviceInfo info;
  rlk_status st = rlk::device_ready(&info);
  if (st != RLK_OK) return st;
  rlk::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      (uint64_t)timeout_us * 1000u);
  return cudaGetLastError() == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

int rlk_is_debug_build(void) {
#ifdef RLK_DEBUG
  return 1;
#else
  return 0;
#endif
}

rlk_status rlk_selftest_store_check(void* stream) {
#ifdef RLK_DEBUG
  rlk::DeviceInfo info;
  rlk_status st = rlk::device_ready(&info);
  if (st != RLK_OK) return st;
  rlk::selftest_store_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(nullptr);
  return cudaGetLastError() == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
#else
  (void)stream;
  return RLK_ERR_NOT_DEBUG_BUILD;
#endif
}

rlk_status rlk_vocab_split_policy(int64_t V, int64_t* num_splits, int64_t* vtiles_per_split,
                                  int64_t* num_vtiles) {
  if (!num_splits || !vtiles_per_split || !num_vtiles) return RLK_ERR_NULL;
  if (V < 1 || V >= rlk::kMaxExtent) return RLK_ERR_SHAPE;
  const int64_t vt = rlk::ceil_div(V, rlk::kVocabTile);
  const int64_t vps = rlk::ceil_div(vt, rlk::kMaxVocabSplits);
  *num_vtiles = vt;
  *vtiles_per_split = vps;
  *num_splits = rlk::ceil_div(vt, vps);
  return RLK_OK;
}

}  // extern "C"
