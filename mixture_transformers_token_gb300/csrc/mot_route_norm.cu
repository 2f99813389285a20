// Routing pre-pass and fused residual-add RMSNorm.
//
// Routing: [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435,
// §1 Motivation item 1 -- every GEMM and norm picks its weight set per token by a fixed
// index set, with no learned router.
// RMSNorm: [WS1][CUDA][Qwen3-Next] MoE route/combine contract ... #503, zero-centred RMSNorm
// commit (x * rstd * w, weight multiply in fp32, one trailing cast, offset 0) and its "On
// exactness against vLLM" section (a fixed 32-wide chunked sum gives batch invariance).

#include <cuda_runtime.h>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {

// ---------------------------------------------------------------------------
// routing pre-pass: one CTA builds the per-expert row lists and the tile table
// ---------------------------------------------------------------------------
constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) route_plan_kernel(const uint8_t* __restrict__ mod, int T,
                                                                    uint8_t* __restrict__ ws) {
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + perm_offset());
  Tile* tiles = reinterpret_cast<Tile*>(ws + tiles_offset(T));
  __shared__ int warp_incl[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // each thread owns a contiguous segment of rows, so a block-wide scan of the und counts
  // gives every row its slot in the stable ascending lists
  const int seg = (T + kRouteThreads - 1) / kRouteThreads;
  const int begin = min(tid * seg, T), end = min(begin + seg, T);
  int n_und = 0, bad = 0;
  for (int r = begin; r < end; ++r) {
    const int m = mod[r];
    bad |= (m > 1);
    n_und += (m == 0);
  }
  int incl = n_und;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_incl[warp] = incl;
  bad = __syncthreads_or(bad);
  if (warp == 0) {
    int v = warp_incl[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += u;
    }
    warp_incl[lane] = v;
  }
  __syncthreads();
  const int total_und = warp_incl[31];
  if (bad) {
    if (tid == 0) {
      hdr->T = T;
      hdr->count[0] = hdr->count[1] = 0;
      hdr->num_m_tiles = 0;
      hdr->error = MOT_DEV_BAD_MODALITY;
      hdr->magic = kPlanMagic;
    }
    return;
  }
  const int und_before = (warp > 0 ? warp_incl[warp - 1] : 0) + incl - n_und;
  int u = und_before, g = total_und + (begin - und_before);
  for (int r = begin; r < end; ++r) {
    if (mod[r] == 0)
      perm[u++] = r;
    else
      perm[g++] = r;
  }
  __syncthreads();
  const int total_gen = T - total_und;
  const int nt0 = (total_und + kTileRows - 1) / kTileRows;
  const int nt1 = (total_gen + kTileRows - 1) / kTileRows;
  for (int t = tid; t < nt0 + nt1; t += kRouteThreads) {
    const int e = t < nt0 ? 0 : 1;
    const int i = e == 0 ? t : t - nt0;
    const int cnt = e == 0 ? total_und : total_gen;
    Tile tl;
    tl.list_begin = (e == 0 ? 0 : total_und) + kTileRows * i;
    tl.n_rows = min(kTileRows, cnt - kTileRows * i);
    tl.expert = e;
    const int first = perm[tl.list_begin], last = perm[tl.list_begin + tl.n_rows - 1];
    tl.row0 = (last - first == tl.n_rows - 1) ? first : -1;
    tiles[t] = tl;
  }
  if (tid == 0) {
    hdr->T = T;
    hdr->count[0] = total_und;
    hdr->count[1] = total_gen;
    hdr->num_m_tiles = nt0 + nt1;
    hdr->error = 0;
    hdr->magic = kPlanMagic;
  }
}

// ---------------------------------------------------------------------------
// fused residual add + routed RMSNorm: one warp per row
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 128;

template <int NJ>
__global__ void __launch_bounds__(kNormThreads) add_rmsnorm_kernel(
    const uint4* __restrict__ x, const uint4* res, const uint16_t* __restrict__ w,
    const uint8_t* __restrict__ mod, int T, int H, float eps, uint4* __restrict__ y, uint4* res_out,
    uint32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (kNormThreads / 32) + (threadIdx.x >> 5);
  if (row >= T) return;
  const int nj = H >> 8;
  const int64_t base = row * (H >> 3);  // row start in 16-byte units
  // lane l owns columns 256 j + 8 l + t: one 16-byte vector per j
  uint4 xs[NJ], rs[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (j < nj) {
      xs[j] = __ldcs(x + base + 32 * j + lane);
      rs[j] = __ldcs(res + base + 32 * j + lane);
    }
  const int m = mod[row];
  float p = 0.0f;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (j < nj) {
      const uint32_t xv[4] = {xs[j].x, xs[j].y, xs[j].z, xs[j].w};
      const uint32_t rv[4] = {rs[j].x, rs[j].y, rs[j].z, rs[j].w};
      uint32_t sv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sv[k] = pack_bf2(__fadd_rn(bf_lo(xv[k]), bf_lo(rv[k])), __fadd_rn(bf_hi(xv[k]), bf_hi(rv[k])));
        const float s0 = bf_lo(sv[k]), s1 = bf_hi(sv[k]);
        p = __fadd_rn(p, __fmul_rn(s0, s0));  // t = 2k
        p = __fadd_rn(p, __fmul_rn(s1, s1));  // t = 2k + 1
      }
      xs[j] = make_uint4(sv[0], sv[1], sv[2], sv[3]);
      __stcs(res_out + base + 32 * j + lane, xs[j]);
    }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off));
  if (m > 1) {
    if (lane == 0 && err != nullptr) atomicOr(err, MOT_DEV_BAD_MODALITY);
    return;
  }
  const float ms = __fdiv_rn(p, float(H));
  const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
  const uint4* wv = reinterpret_cast<const uint4*>(w + int64_t(m) * H);
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (j < nj) {
      const uint4 ww = __ldg(wv + 32 * j + lane);
      const uint32_t sv[4] = {xs[j].x, xs[j].y, xs[j].z, xs[j].w};
      const uint32_t wq[4] = {ww.x, ww.y, ww.z, ww.w};
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        o[k] = pack_bf2(__fmul_rn(__fmul_rn(bf_lo(sv[k]), rstd), bf_lo(wq[k])),
                        __fmul_rn(__fmul_rn(bf_hi(sv[k]), rstd), bf_hi(wq[k])));
      y[base + 32 * j + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int NJ>
static cudaError_t launch_norm(const mot_bf16* x, const mot_bf16* res, const mot_bf16* w, const uint8_t* mod,
                               int T, int H, float eps, mot_bf16* y, mot_bf16* res_out, uint32_t* err,
                               cudaStream_t s) {
  const int rows_per_block = kNormThreads / 32;
  const unsigned grid = unsigned((T + rows_per_block - 1) / rows_per_block);
  add_rmsnorm_kernel<NJ><<<grid, kNormThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(x), reinterpret_cast<const uint4*>(res), w, mod, T, H, eps,
      reinterpret_cast<uint4*>(y), reinterpret_cast<uint4*>(res_out), err);
  return cudaGetLastError();
}

int enqueue_route_plan(const uint8_t* mod, int T, uint8_t* ws, cudaStream_t s) {
  route_plan_kernel<<<1, kRouteThreads, 0, s>>>(mod, T, ws);
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

}  // namespace mot

using namespace mot;

extern "C" int mot_route_plan(const uint8_t* mod, int64_t T, void* ws, size_t ws_bytes, void* stream) {
  if (mod == nullptr || ws == nullptr) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (!aligned16(ws)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {mod, ws};
  int dev = -1;
  int st = check_device(s, ptrs, 2, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  route_plan_kernel<<<1, kRouteThreads, 0, s>>>(mod, int(T), static_cast<uint8_t*>(ws));
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

extern "C" int mot_fused_add_rmsnorm(const mot_bf16* x, const mot_bf16* res, const mot_bf16* w,
                                     const uint8_t* mod, int64_t T, int H, float eps, mot_bf16* y,
                                     mot_bf16* res_out, void* ws, void* stream) {
  if (!x || !res || !w || !mod || !y || !res_out) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || H < 256 || H > 8192 || H % 256 != 0) return MOT_ERR_GEOMETRY;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return MOT_ERR_ARG;
  if (!aligned16(x) || !aligned16(res) || !aligned16(w) || !aligned16(y) || !aligned16(res_out) ||
      (ws && !aligned16(ws)))
    return MOT_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {x, res, w, mod, y, res_out, ws};
  int dev = -1;
  int st = check_device(s, ptrs, 7, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  uint32_t* err = ws ? &static_cast<PlanHeader*>(ws)->error : nullptr;
  const int nj = H / 256;
  cudaError_t e;
  if (nj <= 4)
    e = launch_norm<4>(x, res, w, mod, int(T), H, eps, y, res_out, err, s);
  else if (nj <= 8)
    e = launch_norm<8>(x, res, w, mod, int(T), H, eps, y, res_out, err, s);
  else if (nj <= 16)
    e = launch_norm<16>(x, res, w, mod, int(T), H, eps, y, res_out, err, s);
  else
    e = launch_norm<32>(x, res, w, mod, int(T), H, eps, y, res_out, err, s);
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
