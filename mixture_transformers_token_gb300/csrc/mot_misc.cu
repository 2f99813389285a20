// ABI housekeeping, the RoPE table builder, the device status read-back and the one-time
// gate/up weight interleave.

#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {

// fp32 -> bf16 bits, round to nearest even (host side of the table builder)
static uint16_t host_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return uint16_t((u >> 16) | 0x40u);  // NaN
  const uint32_t lsb = (u >> 16) & 1u;
  return uint16_t((u + 0x7FFFu + lsb) >> 16);
}

// w_gu[e][256 b + o][:] = o < 128 ? w_gate[e][128 b + o][:] : w_up[e][128 b + o - 128][:]
__global__ void swiglu_interleave_kernel(const uint4* __restrict__ wg, const uint4* __restrict__ wu, int I, int K8,
                                         uint4* __restrict__ out) {
  const int64_t total = int64_t(2) * 2 * I * K8;  // experts x 2I rows x K/8 vectors
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t k8 = idx % K8;
    const int64_t r = (idx / K8) % (2 * I);
    const int64_t e = idx / (int64_t(K8) * 2 * I);
    const int64_t b = r / 256, o = r % 256;
    const uint4* src = o < 128 ? wg : wu;
    const int64_t srow = 128 * b + (o % 128);
    out[idx] = src[(e * I + srow) * K8 + k8];
  }
}

// Waits on an mbarrier that nothing ever signals, through the same bounded wait as every
// pipeline wait of the library: after the limit the wait gives up, records MOT_DEV_TIMEOUT in
// the error word and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
}

}  // namespace mot

using namespace mot;

extern "C" int mot_abi_version(void) { return MOT_ABI_VERSION; }

extern "C" const char* mot_status_string(int status) {
  switch (status) {
    case MOT_OK: return "ok";
    case MOT_ERR_NULL: return "a required pointer is NULL";
    case MOT_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case MOT_ERR_GEOMETRY: return "unsupported geometry";
    case MOT_ERR_DEVICE: return "a pointer is not device memory of the stream's device";
    case MOT_ERR_WORKSPACE: return "workspace too small";
    case MOT_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case MOT_ERR_CUDA: return "CUDA runtime error";
    case MOT_ERR_ARG: return "invalid argument";
    case MOT_ERR_NOALLOC_LIMIT: return "T exceeds MOT_NOALLOC_MAX_TOKENS, the row limit of the allocation-free entry point";
    default: return "unknown status";
  }
}

extern "C" size_t mot_workspace_bytes(int64_t T) {
  if (T < 1 || T > MOT_MAX_TOKENS) return 0;
  return size_t(plan_bytes(T));
}

// (cos_i, sin_i) of positions 0 .. P-1 in fp32: inv_i = theta^(-2i/D) in fp64 stored fp32,
// angle = fp32(p) * inv_i in fp32, cos and sin in fp64 of that angle, stored fp32.
template <typename Store>
static int rope_table_fill(double theta, int D, int P, Store store) {
  if (D < 2 || D > 1024 || D % 2 != 0 || P < 1 || P > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (!(theta > 1.0) || !std::isfinite(theta)) return MOT_ERR_ARG;
  const int half = D / 2;
  float inv[512];
  for (int i = 0; i < half; ++i) inv[i] = float(std::pow(theta, -2.0 * double(i) / double(D)));
  for (int p = 0; p < P; ++p) {
    const float fp = float(p);
    for (int i = 0; i < half; ++i) {
      const float ang = fp * inv[i];
      store((int64_t(p) * half + i) * 2, float(std::cos(double(ang))), float(std::sin(double(ang))));
    }
  }
  return MOT_OK;
}

extern "C" int mot_rope_table_fill_host(double theta, int D, int P, mot_bf16* host_cs) {
  if (host_cs == nullptr) return MOT_ERR_NULL;
  return rope_table_fill(theta, D, P, [host_cs](int64_t k, float c, float s) {
    host_cs[k] = host_f32_to_bf16(c);
    host_cs[k + 1] = host_f32_to_bf16(s);
  });
}

extern "C" int mot_rope_table_fill_host_fp32(double theta, int D, int P, float* host_cs) {
  if (host_cs == nullptr) return MOT_ERR_NULL;
  return rope_table_fill(theta, D, P, [host_cs](int64_t k, float c, float s) {
    host_cs[k] = c;
    host_cs[k + 1] = s;
  });
}

extern "C" int mot_device_status(const void* ws, uint32_t* flags, void* stream) {
  if (ws == nullptr || flags == nullptr) return MOT_ERR_NULL;
  if (!aligned16(ws)) return MOT_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = -1;
  int st = stream_device(s, &dev);
  if (st != MOT_OK) return st;
  st = check_ptr(ws, dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOT_ERR_CUDA;
  const PlanHeader* hdr = static_cast<const PlanHeader*>(ws);
  if (cudaMemcpy(flags, &hdr->error, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MOT_ERR_CUDA;
  return MOT_OK;
}

extern "C" int mot_swiglu_interleave(const mot_bf16* w_gate, const mot_bf16* w_up, int I, int K, mot_bf16* w_gu,
                                     void* stream) {
  if (!w_gate || !w_up || !w_gu) return MOT_ERR_NULL;
  if (I < 128 || I % 128 != 0 || K < 8 || K % 8 != 0 || int64_t(I) * K > (int64_t(1) << 34)) return MOT_ERR_GEOMETRY;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_gu)) return MOT_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {w_gate, w_up, w_gu};
  int dev = -1;
  int st = check_device(s, ptrs, 3, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const int grid = 4 * sm_count(dev);
  swiglu_interleave_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(w_gate),
                                                 reinterpret_cast<const uint4*>(w_up), I, K / 8,
                                                 reinterpret_cast<uint4*>(w_gu));
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

extern "C" int mot_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr) return MOT_ERR_NULL;
  if (!aligned16(ws)) return MOT_ERR_ALIGN;
  if (ws_bytes < sizeof(PlanHeader)) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {ws};
  int dev = -1;
  int st = check_device(s, ptrs, 1, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(&static_cast<PlanHeader*>(ws)->error);
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
