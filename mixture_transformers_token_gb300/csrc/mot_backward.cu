// Backward of the fused residual-add RMSNorm: the input gradient (dx = dres) and the gradient
// of the per-expert norm weights.
//
// Sources: [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435
// (§3 BAGEL-specific rules: phase A trains the gen weight set, the frozen und operators still
// need dX; §3 Numerical contract: fixed accumulation order, no atomics); [WS1][CUDA][Qwen3-Next]
// MoE route/combine contract ... #503 (gated-norm commit: a dx kernel, and the weight gradient
// as per-row fp32 partials folded in ascending row order; zero-centred RMSNorm commit: the
// fixed 32-wide chunked sum).
//
// Forward: s = bf16(x + res), rstd = 1/sqrt(sum s^2 / H + eps), y = bf16(s * rstd * w[e]).
// Backward, every operation rounded on its own in fp32 (no fused multiply-add):
//   xh = s * rstd, g = dy * w[e], dot = the forward's fixed tree over g * xh, c = dot / H,
//   ds = rstd * (g - xh * c) (+ d_res_out), dx = bf16(ds);
//   dw[e][j] = ((p_r0 + p_r1) + p_r2) + ... over the rows r0 < r1 < ... of weight set e,
//   p_r = dy[r][j] * xh[r][j].
//
// add_rmsnorm_bwd_kernel   one warp per row; lane l holds columns 256 j + 8 l + t (the
//                          forward's tree layout) of s and dy in registers for three passes
//                          (sum of s^2, dot, output), writes dx and the row's rstd.
// rmsnorm_dw_fold_kernel   one CTA per (weight set, 64-column block): its 128 threads stream
//                          the set's rows (ascending, from the routing plan) through a ring of
//                          shared-memory stages with cp.async; 64 of them fold one column each.

#include <cuda_runtime.h>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {
namespace bwd {

struct NormBwdArgs {
  const uint4* dy;
  const uint4* s;
  const uint4* dro;  // may be null
  const uint4* w;    // [2][H/8]
  const uint8_t* mod;
  int T, H;
  float eps;
  uint4* dx;
  float* rstd;
  uint32_t* err;
};

__device__ __forceinline__ float elem(const uint4& v, int t) {
  const uint32_t wd = t < 2 ? v.x : (t < 4 ? v.y : (t < 6 ? v.z : v.w));
  return (t & 1) ? bf_hi(wd) : bf_lo(wd);
}

__device__ __forceinline__ float warp_tree(float p) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off));
  return p;
}

template <int NJ>  // NJ >= H / 256
__global__ void __launch_bounds__(256) add_rmsnorm_bwd_kernel(const NormBwdArgs a) {
  extern __shared__ uint4 sw[];  // both weight sets, [2][H/8]
  const int h8 = a.H / 8, nj = a.H / 256;
  for (int i = threadIdx.x; i < 2 * h8; i += blockDim.x) sw[i] = __ldg(a.w + i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  const float fH = float(a.H);
  for (int64_t row = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < a.T; row += warps) {
    const int e = a.mod[row];
    if (e > 1) {
      if (lane == 0) atomicOr(a.err, MOT_DEV_BAD_MODALITY);
      continue;
    }
    const uint4* srow = a.s + row * h8 + lane;
    const uint4* drow = a.dy + row * h8 + lane;
    // rows wider than 4096 keep only s in registers and read dy again in passes 2 and 3
    constexpr bool kHoldDy = NJ <= 16;
    uint4 sv[NJ], dv[kHoldDy ? NJ : 1];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
        sv[j] = __ldcs(srow + j * 32);
        if constexpr (kHoldDy) dv[j] = __ldcs(drow + j * 32);
      }
    }
    // pass 1: sum of s^2 on the forward's tree
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float v = elem(sv[j], t);
          ss = __fadd_rn(ss, __fmul_rn(v, v));
        }
      }
    }
    ss = warp_tree(ss);
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, fH), a.eps)));
    // pass 2: dot = sum of (dy * w) * (s * rstd) on the same tree
    const uint4* wrow = sw + e * h8 + lane;
    float dot = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
        const uint4 wv = wrow[j * 32];
        uint4 d;
        if constexpr (kHoldDy) d = dv[j]; else d = __ldg(drow + j * 32);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float xh = __fmul_rn(elem(sv[j], t), rstd);
          const float g = __fmul_rn(elem(d, t), elem(wv, t));
          dot = __fadd_rn(dot, __fmul_rn(g, xh));
        }
      }
    }
    dot = warp_tree(dot);
    const float c = __fdiv_rn(dot, fH);
    // pass 3: ds = rstd * (g - xh * c) (+ d_res_out), one cast
    uint4* orow = a.dx + row * h8 + lane;
    const uint4* rrow = a.dro ? a.dro + row * h8 + lane : nullptr;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
        const uint4 wv = wrow[j * 32];
        uint4 d;
        if constexpr (kHoldDy) d = dv[j]; else d = __ldg(drow + j * 32);
        uint4 rv = make_uint4(0u, 0u, 0u, 0u);
        if (rrow) rv = __ldcs(rrow + j * 32);
        float o[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float xh = __fmul_rn(elem(sv[j], t), rstd);
          const float g = __fmul_rn(elem(d, t), elem(wv, t));
          float ds = __fmul_rn(rstd, __fsub_rn(g, __fmul_rn(xh, c)));
          if (rrow) ds = __fadd_rn(ds, elem(rv, t));
          o[t] = ds;
        }
        __stcs(orow + j * 32, make_uint4(pack_bf2(o[0], o[1]), pack_bf2(o[2], o[3]), pack_bf2(o[4], o[5]),
                                         pack_bf2(o[6], o[7])));
      }
    }
    if (lane == 0) a.rstd[row] = rstd;
  }
}

constexpr int kFoldCols = 64, kFoldRows = 32, kFoldStages = 12, kFoldThreads = 128;
constexpr size_t kFoldStageBytes = size_t(2) * kFoldRows * kFoldCols * 2 + kFoldRows * 4;
constexpr size_t kFoldSmem = kFoldStages * kFoldStageBytes;

struct FoldArgs {
  const uint16_t* dy;
  const uint16_t* s;
  const float* rstd;
  const uint8_t* ws;
  int T, H;
  float* dw;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kFoldThreads) rmsnorm_dw_fold_kernel(const FoldArgs a) {
  extern __shared__ __align__(16) uint8_t fsm[];
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(a.ws);
  const int ncb = a.H / kFoldCols;
  const int e = int(blockIdx.x) / ncb, cb = int(blockIdx.x) % ncb;
  const int tid = threadIdx.x;
  if (hdr->magic != kPlanMagic || hdr->T != a.T) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(const_cast<uint32_t*>(&hdr->error), MOT_DEV_PLAN_MISMATCH);
    return;
  }
  if (hdr->count[0] + hdr->count[1] != a.T) return;  // no plan (bad modality): nothing is defined
  const int count = hdr->count[e];
  const int32_t* rows = reinterpret_cast<const int32_t*>(a.ws + perm_offset()) + (e ? hdr->count[0] : 0);
  const int nst = (count + kFoldRows - 1) / kFoldRows;
  const int col0 = cb * kFoldCols;
  auto stage_dy = [&](int slot) { return fsm + size_t(slot) * kFoldStageBytes; };
  auto stage_s = [&](int slot) { return fsm + size_t(slot) * kFoldStageBytes + kFoldRows * kFoldCols * 2; };
  auto stage_r = [&](int slot) { return fsm + size_t(slot) * kFoldStageBytes + 2 * kFoldRows * kFoldCols * 2; };
  auto load_stage = [&](int k, int slot) {
    // 32 rows x 64 columns of dy and of s (8 chunks of 16 B per row), and the rows' rstd
    for (int c = tid; c < 2 * kFoldRows * 8; c += kFoldThreads) {
      const int arr = c / (kFoldRows * 8), rr = (c / 8) % kFoldRows, part = c % 8;
      const int i = k * kFoldRows + rr;
      if (i < count) {
        const int64_t r = rows[i];
        const uint16_t* src = (arr ? a.s : a.dy) + r * a.H + col0 + part * 8;
        uint8_t* dst = (arr ? stage_s(slot) : stage_dy(slot)) + (rr * kFoldCols + part * 8) * 2;
        cp_async16(smem_u32(dst), src);
      }
    }
    if (tid < kFoldRows) {
      const int i = k * kFoldRows + tid;
      if (i < count) cp_async4(smem_u32(stage_r(slot) + tid * 4), a.rstd + rows[i]);
    }
  };
#pragma unroll 1
  for (int k = 0; k < kFoldStages - 1; ++k) {
    if (k < nst) load_stage(k, k);
    cp_async_commit();
  }
  float acc = -0.0f;  // -0 + p = p for every p: the fold starts with the first row's partial
#pragma unroll 1
  for (int k = 0; k < nst; ++k) {
    cp_async_wait<kFoldStages - 2>();
    __syncthreads();  // stage k landed for every thread; stage k - 1 is no longer read
    const int kn = k + kFoldStages - 1;
    if (kn < nst) load_stage(kn, kn % kFoldStages);
    cp_async_commit();
    if (tid < kFoldCols) {
      const int slot = k % kFoldStages;
      const uint16_t* sdy = reinterpret_cast<const uint16_t*>(stage_dy(slot));
      const uint16_t* ssv = reinterpret_cast<const uint16_t*>(stage_s(slot));
      const float* srs = reinterpret_cast<const float*>(stage_r(slot));
      const int n = count - k * kFoldRows < kFoldRows ? count - k * kFoldRows : kFoldRows;
#pragma unroll 4
      for (int rr = 0; rr < n; ++rr) {
        const float xh = __fmul_rn(bf_to_f(ssv[rr * kFoldCols + tid]), srs[rr]);
        acc = __fadd_rn(acc, __fmul_rn(bf_to_f(sdy[rr * kFoldCols + tid]), xh));
      }
    }
  }
  cp_async_wait<0>();
  if (tid < kFoldCols) a.dw[int64_t(e) * a.H + col0 + tid] = count > 0 ? acc : 0.0f;
}

template <int NJ>
static cudaError_t launch_bwd(const NormBwdArgs& a, int dev, cudaStream_t s) {
  const size_t smem = size_t(a.H) * 2 * 2;
  cudaError_t st = cudaFuncSetAttribute(add_rmsnorm_bwd_kernel<NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(smem));
  if (st != cudaSuccess) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, add_rmsnorm_bwd_kernel<NJ>, 256, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int64_t want = (int64_t(a.T) + 7) / 8;
  const int64_t cap = int64_t(per_sm) * sm_count(dev);
  const int grid = int(want < cap ? want : cap);
  add_rmsnorm_bwd_kernel<NJ><<<grid, 256, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace mot

using namespace mot;

extern "C" int mot_add_rmsnorm_backward(const mot_bf16* dy, const mot_bf16* d_res_out, const mot_bf16* s,
                                        const mot_bf16* w, const uint8_t* mod, int64_t T, int H, float eps,
                                        void* ws, size_t ws_bytes, mot_bf16* dx, float* rstd, void* stream) {
  if (!dy || !s || !w || !mod || !ws || !dx || !rstd) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || H < 256 || H > 8192 || H % 256 != 0) return MOT_ERR_GEOMETRY;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return MOT_ERR_ARG;
  if (!aligned16(dy) || (d_res_out && !aligned16(d_res_out)) || !aligned16(s) || !aligned16(w) || !aligned16(ws) ||
      !aligned16(dx) || !aligned16(rstd))
    return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {dy, d_res_out, s, w, mod, ws, dx, rstd};
  int dev = -1;
  int rc = check_device(st, ptrs, 8, &dev);
  if (rc != MOT_OK) return rc;
  DeviceGuard guard(dev);
  bwd::NormBwdArgs a{};
  a.dy = reinterpret_cast<const uint4*>(dy);
  a.s = reinterpret_cast<const uint4*>(s);
  a.dro = reinterpret_cast<const uint4*>(d_res_out);
  a.w = reinterpret_cast<const uint4*>(w);
  a.mod = mod;
  a.T = int(T);
  a.H = H;
  a.eps = eps;
  a.dx = reinterpret_cast<uint4*>(dx);
  a.rstd = rstd;
  a.err = &static_cast<PlanHeader*>(ws)->error;
  const int nj = H / 256;
  cudaError_t e;
  if (nj <= 4)
    e = bwd::launch_bwd<4>(a, dev, st);
  else if (nj <= 8)
    e = bwd::launch_bwd<8>(a, dev, st);
  else if (nj <= 16)
    e = bwd::launch_bwd<16>(a, dev, st);
  else
    e = bwd::launch_bwd<32>(a, dev, st);
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

extern "C" int mot_rmsnorm_dweight(const mot_bf16* dy, const mot_bf16* s, const float* rstd, int64_t T, int H,
                                   void* ws, size_t ws_bytes, float* dw, void* stream) {
  if (!dy || !s || !rstd || !ws || !dw) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || H < 256 || H > 8192 || H % 256 != 0) return MOT_ERR_GEOMETRY;
  if (!aligned16(dy) || !aligned16(s) || !aligned16(rstd) || !aligned16(ws) || !aligned16(dw)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {dy, s, rstd, ws, dw};
  int dev = -1;
  int rc = check_device(st, ptrs, 5, &dev);
  if (rc != MOT_OK) return rc;
  DeviceGuard guard(dev);
  if (cudaFuncSetAttribute(bwd::rmsnorm_dw_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(bwd::kFoldSmem)) != cudaSuccess)
    return MOT_ERR_CUDA;
  bwd::FoldArgs a{};
  a.dy = dy;
  a.s = s;
  a.rstd = rstd;
  a.ws = static_cast<const uint8_t*>(ws);
  a.T = int(T);
  a.H = H;
  a.dw = dw;
  const int grid = 2 * (H / bwd::kFoldCols);
  bwd::rmsnorm_dw_fold_kernel<<<grid, bwd::kFoldThreads, bwd::kFoldSmem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
