// Host-side helpers shared by the library's runtimes (MoE layer, attention
// block): the thread's last error message, CUDA error checks, the current-device
// guard, TMA descriptor encoding and the persistent CTA-pair grid size.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "moe_layer.h"

namespace moe_host {

// Detail of the last failed call on this thread (moe_last_error_message).
inline thread_local std::string g_last_error;

inline moe_status_t fail(moe_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

inline moe_status_t ok() {
  g_last_error.clear();
  return MOE_OK;
}

#define MOE_CUDA_TRY(call)                                                                              \
  do {                                                                                                  \
    cudaError_t e_ = (call);                                                                            \
    if (e_ != cudaSuccess) return moe_host::fail(MOE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait inside a kernel

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched through the runtime (no libcuda link).
inline EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

constexpr uint32_t kTmapBoxInner = 64;  // bf16 boxes are 64 elements (128 bytes) wide

// Row-major 2-D tensor [rows, inner] of bf16, box [box_rows, 64], 128-byte swizzle;
// reads outside the tensor return zeros.
inline moe_status_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                                   uint32_t box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {kTmapBoxInner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

// Row-major 2-D tensor [rows, inner] of esize-byte elements, box [box_rows, box_inner],
// no swizzle (rows land in shared memory as they are in global memory).
inline moe_status_t make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base,
                                 uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (%u-byte elements) failed (%d)", esize, (int)r);
  return MOE_OK;
}

// CTAs of a persistent cluster launch of `kernel` (clusters of 2): twice the
// clusters that can be resident at once, at most one CTA per SM.
inline moe_status_t cluster_pair_grid(int num_sms, const void* kernel, int threads, size_t smem, int* grid) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2 * (num_sms / 2), 1, 1);
  lc.blockDim = dim3(threads, 1, 1);
  lc.dynamicSmemBytes = smem;
  int clusters = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &lc);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
  if (clusters < 1) return fail(MOE_ERR_UNSUPPORTED, "no CTA pair of the grouped GEMM fits on this device");
  *grid = 2 * std::min(clusters, num_sms / 2);
  return MOE_OK;
}

}  // namespace moe_host
