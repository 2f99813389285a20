// Host-side helpers shared by the entry points: argument checks, the device guard, cached
// device attributes and TMA tensor-map encoding. Nothing here allocates device memory.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <utility>

#include "mot.h"

namespace mot {

constexpr int kMaxDevices = 64;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device that owns `stream` (the current device for the legacy default stream).
inline int stream_device(cudaStream_t s, int* dev) {
  if (s == nullptr) return cudaGetDevice(dev) == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
  return cudaStreamGetDevice(s, dev) == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

// A pointer is usable only if it is device (or managed) memory of `dev`.
inline int check_ptr(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return MOT_ERR_DEVICE;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return MOT_ERR_DEVICE;
  if (a.device != dev) return MOT_ERR_DEVICE;
  return MOT_OK;
}

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 ok, 2 wrong arch
  std::atomic<int> sms{0};
};

inline DeviceInfo& device_info(int dev) {
  static DeviceInfo info[kMaxDevices];
  return info[dev];
}

// Compute capability 10.3 is required (tcgen05, TMEM and TMA forms compiled for sm_103a).
inline int check_arch(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return MOT_ERR_DEVICE;
  DeviceInfo& d = device_info(dev);
  int st = d.state.load();
  if (st == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOT_ERR_CUDA;
    d.sms.store(sms);
    st = (major == 10 && minor == 3) ? 1 : 2;
    d.state.store(st);
  }
  return st == 1 ? MOT_OK : MOT_ERR_ARCH;
}

inline int sm_count(int dev) { return device_info(dev).sms.load(); }

// Launches `kernel` so that it may start while the stream's preceding grid is still running
// (programmatic dependent launch; the kernel must call pdl_wait before it reads that grid's
// output).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Makes `dev` current for the lifetime of the guard and restores the previous device.
struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) changed = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

// Resolves the stream's device, checks the architecture and every pointer in `ptrs`
// (NULL entries are skipped: optional arguments are checked for NULL by the caller).
inline int check_device(cudaStream_t s, const void* const* ptrs, int n, int* dev_out) {
  int dev = -1;
  int st = stream_device(s, &dev);
  if (st != MOT_OK) return st;
  st = check_arch(dev);
  if (st != MOT_OK) return st;
  for (int i = 0; i < n; ++i) {
    if (ptrs[i] == nullptr) continue;
    st = check_ptr(ptrs[i], dev);
    if (st != MOT_OK) return st;
  }
  *dev_out = dev;
  return MOT_OK;
}

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry point so that
// the library does not link against the driver library directly.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load();
  if (f == nullptr) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn.store(f);
  }
  return reinterpret_cast<EncodeTiledFn>(f);
}

// 2D bf16 tensor map over a row-major [rows][cols] array with the 128-byte swizzle.
inline bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                           uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Enqueues the routing pre-pass into `ws` (at least plan_bytes(T) bytes) without argument
// checks; used by entry points that have already validated their arguments.
int enqueue_route_plan(const uint8_t* mod, int T, uint8_t* ws, cudaStream_t s);

}  // namespace mot
