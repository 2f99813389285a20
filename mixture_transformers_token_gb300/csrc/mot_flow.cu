// Flow-matching sampler pieces: the step schedule, three-branch renormalised CFG and the SDE
// step with its log-probability, per request.
//
// Sources: [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435
// (§1 Motivation items 2 and 3: the policy log-probability is the ODE-to-SDE transition density;
// three-branch renormalised CFG with two scales, a timestep window and a norm-ratio rescale;
// §3 BAGEL-specific rules: schedule built in FP64 and stored in FP32 with the shift s; SDE step
// and logp in FP32 with sigma = t and dt = t_i - t_{i+1} > 0; logp summed over all latent
// elements in a fixed order; CFG window compared on FP32 t; renorm per request; no fast math).
//
// Readings (the pages give no formulas): the rectified-flow path x_t = (1 - t) x_0 + t eps with
// velocity v = eps - x_0; the SDE step mu = x - dt (v + sigma^2 / (2 t) (x + (1 - t) v)),
// std = sigma sqrt(dt); CFG v1 = tu + s_text (c - tu), v2 = iu + s_img (v1 - iu), rescaled by
// clamp(||c|| / ||v2||, min, 1) over the request's elements.
//
// A request's elements are cut into segments of 8192; a CTA of 256 threads takes one segment at
// a time (the CTAs stride over all requests' segments).
// The segment's elements are taken in chunks of 8; thread tau owns the segment's chunks q with
// q % 256 == tau (so a warp's loads are consecutive 16- or 32-byte pieces); a segment sum runs
// sequentially per thread over its chunks in ascending order, then as an xor butterfly (16, 8,
// 4, 2, 1) inside each warp, then over the 8 warps left to right; the request's sum folds its
// segment sums left to right. The order depends only on the request's length, never on the
// batch. Every operation is rounded on its own in fp32 (no fused multiply-add).
//
// CFG reads its inputs twice (once for the sums, once to scale), the second time mostly from
// L2; the SDE step reads them once and a small kernel folds each request's segment sums. The
// fused CFG + SDE step applies the CFG's rescale inside the SDE step's element pass, so the
// guided velocity never goes to memory and back.

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {
namespace flow {

constexpr int THREADS = 256;
constexpr int SEG = 8192;                    // elements per segment
constexpr int CPT = SEG / 8 / THREADS;       // chunks per thread and segment (4)
constexpr int64_t kMaxN = int64_t(1) << 24;  // elements per request
constexpr int kMaxReq = 65535;
constexpr int kCtasPerSm = 4;                // resident CTAs per SM at the launch bounds below
constexpr float kLogSqrt2Pi = 0.918938533204672742f;  // log(2 pi) / 2

__host__ __device__ constexpr int segments(int64_t N) { return int((N + SEG - 1) / SEG); }

// Workspace: the 64-byte header (error word), then 8 bytes per (request, segment): the CFG's
// (sum c c, sum v2 v2), or the SDE step's sum d d; then 4 bytes per (request, segment), where
// the fused CFG + SDE step keeps its sums of d d while the CFG's are still being read.
inline size_t cfg_region_bytes(int n_req, int64_t N) {
  return (size_t(n_req) * size_t(segments(N)) * 8 + 15) & ~size_t(15);
}
inline size_t workspace_bytes(int n_req, int64_t N) {
  return sizeof(PlanHeader) + cfg_region_bytes(n_req, N) + ((size_t(n_req) * size_t(segments(N)) * 4 + 15) & ~size_t(15));
}

// The CTA's sum of the per-thread partials p: butterfly inside each warp, then the warps left
// to right. Every thread returns it.
__device__ __forceinline__ float cta_sum(float p, float* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off));
  __syncthreads();  // every thread has read wsum's previous contents
  if (lane == 0) wsum[warp] = p;
  __syncthreads();
  float acc = wsum[0];
#pragma unroll
  for (int k = 1; k < THREADS / 32; ++k) acc = __fadd_rn(acc, wsum[k]);
  return acc;
}

// Left fold of a request's n segment sums p[0..n): ((p0 + p1) + p2) + ... The lanes of the calling
// warp fetch 32 sums at a time in parallel and the fold takes them in order through shuffles, so
// the chain waits on one L2 round trip per 32 sums instead of one per sum. Every lane returns it.
__device__ __forceinline__ float warp_fold(const float* p, int n) {
  const int lane = threadIdx.x & 31;
  float acc = 0.0f;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const float v = i0 + lane < n ? __ldcg(p + i0 + lane) : 0.0f;
    const int m = n - i0 < 32 ? n - i0 : 32;
    for (int l = 0; l < m; ++l) {
      const float w = __shfl_sync(0xffffffffu, v, l);
      acc = (i0 + l == 0) ? w : __fadd_rn(acc, w);
    }
  }
  return acc;
}

__device__ __forceinline__ float2 warp_fold2(const float2* p, int n) {
  const int lane = threadIdx.x & 31;
  float2 acc = make_float2(0.0f, 0.0f);
  for (int i0 = 0; i0 < n; i0 += 32) {
    const float2 v = i0 + lane < n ? __ldcg(p + i0 + lane) : make_float2(0.0f, 0.0f);
    const int m = n - i0 < 32 ? n - i0 : 32;
    for (int l = 0; l < m; ++l) {
      const float wx = __shfl_sync(0xffffffffu, v.x, l), wy = __shfl_sync(0xffffffffu, v.y, l);
      if (i0 + l == 0) {
        acc = make_float2(wx, wy);
      } else {
        acc.x = __fadd_rn(acc.x, wx);
        acc.y = __fadd_rn(acc.y, wy);
      }
    }
  }
  return acc;
}

// The CFG's ratio from the request's folded sums: sqrt(ss_c) / sqrt(ss_g) (1 when ss_g is 0),
// clamped to [renorm_min, 1].
__device__ __forceinline__ float cfg_ratio(float2 acc, float rmin) {
  const float r = acc.y == 0.0f ? 1.0f : __fdiv_rn(__fsqrt_rn(acc.x), __fsqrt_rn(acc.y));
  return fminf(fmaxf(r, rmin), 1.0f);
}

__device__ __forceinline__ void unpack8_bf16(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf_lo(w[i]);
    v[2 * i + 1] = bf_hi(w[i]);
  }
}

struct F8 {
  float4 a, b;
};

// Eight consecutive floats: one 32-byte load when the array allows it (w32), else two 16-byte ones.
__device__ __forceinline__ F8 load8_f32(const float* p, bool w32) {
  if (w32) {
    F8 f;
    asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(f.a.x), "=f"(f.a.y), "=f"(f.a.z), "=f"(f.a.w), "=f"(f.b.x), "=f"(f.b.y), "=f"(f.b.z),
                   "=f"(f.b.w)
                 : "l"(p));
    return f;
  }
  return F8{__ldg(reinterpret_cast<const float4*>(p)), __ldg(reinterpret_cast<const float4*>(p) + 1)};
}

__device__ __forceinline__ void unpack8_f32(const F8& f, float (&v)[8]) {
  v[0] = f.a.x; v[1] = f.a.y; v[2] = f.a.z; v[3] = f.a.w;
  v[4] = f.b.x; v[5] = f.b.y; v[6] = f.b.z; v[7] = f.b.w;
}

// Eight consecutive floats: one 32-byte store when the array allows it (w32), else two 16-byte ones.
__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8], bool w32) {
  if (w32) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]),
                 "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
    return;
  }
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

struct CfgArgs {
  const uint16_t* c;    // [n_req][N] bf16
  const uint16_t* tu;
  const uint16_t* iu;   // or null: two branches
  const float* policy;  // [n_req][6]: t, s_text, s_img, t_lo, t_hi, renorm_min
  int64_t N;
  int S;                // segments per request
  float2* part;         // [n_req][S]: (sum c c, sum v2 v2) of each segment
  float* out;           // [n_req][N] fp32
  int w32;              // out is 32-byte aligned
};

struct CfgPolicy {
  float t, s_text, s_img, t_lo, t_hi, rmin;
  __device__ bool guided() const { return t_lo <= t && t <= t_hi; }
};

__device__ __forceinline__ CfgPolicy load_policy(const float* p) {
  return CfgPolicy{p[0], p[1], p[2], p[3], p[4], p[5]};
}

// The segment's chunks of this thread, loaded together (CPT loads of each input in flight).
struct CfgChunks {
  uint4 c[CPT], tu[CPT], iu[CPT];
  int n;  // how many of the CPT chunks exist
};

__device__ __forceinline__ void cfg_load(const CfgArgs& a, int64_t base, int nch, CfgChunks& k) {
  k.n = 0;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int q = int(threadIdx.x) + THREADS * j;
    if (q < nch) {
      k.n = j + 1;
      k.c[j] = __ldg(reinterpret_cast<const uint4*>(a.c + base + 8 * q));
      k.tu[j] = __ldg(reinterpret_cast<const uint4*>(a.tu + base + 8 * q));
      if (a.iu) k.iu[j] = __ldg(reinterpret_cast<const uint4*>(a.iu + base + 8 * q));
    }
  }
}

// v1 = tu + s_text (c - tu); v2 = iu + s_img (v1 - iu), or v1 without iu.
__device__ __forceinline__ void cfg_guide(const CfgArgs& a, const CfgPolicy& pol, const CfgChunks& k, int j,
                                          float (&c)[8], float (&v2)[8]) {
  float tu[8];
  unpack8_bf16(k.c[j], c);
  unpack8_bf16(k.tu[j], tu);
#pragma unroll
  for (int i = 0; i < 8; ++i) v2[i] = __fadd_rn(tu[i], __fmul_rn(pol.s_text, __fsub_rn(c[i], tu[i])));
  if (a.iu) {
    float iu[8];
    unpack8_bf16(k.iu[j], iu);
#pragma unroll
    for (int i = 0; i < 8; ++i) v2[i] = __fadd_rn(iu[i], __fmul_rn(pol.s_img, __fsub_rn(v2[i], iu[i])));
  }
}

// Pass 1: each segment's sums of c c and v2 v2; outside the window the segment is copied.
// CTAs stride over the (request, segment) units.
__global__ void __launch_bounds__(THREADS, 4) cfg_partials_kernel(const CfgArgs a, const int64_t units) {
  __shared__ float wsum[2][THREADS / 32];
  pdl_trigger();  // the scale pass may start and load its inputs
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int req = int(u / a.S), seg = int(u % a.S);
    const CfgPolicy pol = load_policy(a.policy + 6 * req);
    const int64_t base = int64_t(req) * a.N + int64_t(seg) * SEG;
    const int nch = int(min(int64_t(SEG), a.N - int64_t(seg) * SEG) / 8);
    if (!pol.guided()) {
      if (a.out == nullptr) continue;  // the fused step reads c itself
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int q = int(threadIdx.x) + THREADS * j;
        if (q < nch) {
          float c[8];
          unpack8_bf16(__ldg(reinterpret_cast<const uint4*>(a.c + base + 8 * q)), c);
          store8_f32(a.out + base + 8 * q, c, a.w32);
        }
      }
      continue;  // uniform across the CTA
    }
    CfgChunks k;
    cfg_load(a, base, nch, k);
    float pc = 0.0f, pg = 0.0f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      if (j < k.n) {
        float c[8], v2[8];
        cfg_guide(a, pol, k, j, c, v2);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pc = __fadd_rn(pc, __fmul_rn(c[i], c[i]));
          pg = __fadd_rn(pg, __fmul_rn(v2[i], v2[i]));
        }
      }
    }
    const float sc = cta_sum(pc, wsum[0]);
    const float sg = cta_sum(pg, wsum[1]);
    if (threadIdx.x == 0) a.part[u] = make_float2(sc, sg);
  }
}

// Pass 2, launched as a dependent of pass 1: a CTA loads its segment's inputs (written before
// pass 1 started), waits for pass 1, folds the request's segment sums (the same order in every
// CTA, so the same r) and writes out = v2 r.
__global__ void __launch_bounds__(THREADS, 4) cfg_scale_kernel(const CfgArgs a, const int64_t units) {
  __shared__ float r_s;
  bool waited = false;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int req = int(u / a.S), seg = int(u % a.S);
    const CfgPolicy pol = load_policy(a.policy + 6 * req);
    if (!pol.guided()) continue;  // pass 1 copied c
    const int64_t base = int64_t(req) * a.N + int64_t(seg) * SEG;
    const int nch = int(min(int64_t(SEG), a.N - int64_t(seg) * SEG) / 8);
    CfgChunks k;
    cfg_load(a, base, nch, k);
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    if (threadIdx.x < 32) {
      const float r = cfg_ratio(warp_fold2(a.part + int64_t(req) * a.S, a.S), pol.rmin);
      if (threadIdx.x == 0) r_s = r;
    }
    __syncthreads();
    const float r = r_s;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      if (j < k.n) {
        const int q = int(threadIdx.x) + THREADS * j;
        float c[8], v2[8];
        cfg_guide(a, pol, k, j, c, v2);
#pragma unroll
        for (int i = 0; i < 8; ++i) v2[i] = __fmul_rn(v2[i], r);
        store8_f32(a.out + base + 8 * q, v2, a.w32);
      }
    }
    __syncthreads();  // r_s is rewritten for the next unit
  }
  if (!waited) pdl_wait();  // this grid completes only after pass 1 has
}

struct SdeArgs {
  const float* x;      // [n_req][N]
  const float* v;
  const float* z;      // or null: x_next is an input
  float* x_next;
  const float* times;  // [n_req][2]: t_i, t_next
  int64_t N;
  int S;
  int n_req;
  float* part;         // [n_req][S]: each segment's sum of d d
  float* logp;         // [n_req]
  uint32_t* err;
  int w32;             // x, v, z and x_next are 32-byte aligned
};

__device__ __forceinline__ bool times_ok(float t, float tn) {
  return __fsub_rn(t, tn) > 0.0f && tn >= 0.0f && t <= 1.0f;
}

__global__ void __launch_bounds__(THREADS, 4) sde_step_kernel(const SdeArgs a, const int64_t units) {
  __shared__ float wsum[THREADS / 32];
  pdl_trigger();  // the logp fold may start
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int req = int(u / a.S), seg = int(u % a.S);
    const float t = a.times[2 * req], tn = a.times[2 * req + 1];
    if (!times_ok(t, tn)) {
      if (threadIdx.x == 0 && seg == 0) atomicOr(a.err, MOT_DEV_BAD_TIME);
      continue;  // uniform across the CTA
    }
    const float dt = __fsub_rn(t, tn);
    const float sigma = t;
    const float kk = __fdiv_rn(__fmul_rn(sigma, sigma), __fmul_rn(2.0f, t));
    const float omt = __fsub_rn(1.0f, t);
    const float sd = __fmul_rn(sigma, __fsqrt_rn(dt));
    const int64_t base = int64_t(req) * a.N + int64_t(seg) * SEG;
    const int nch = int(min(int64_t(SEG), a.N - int64_t(seg) * SEG) / 8);
    const float* third = a.z ? a.z : a.x_next;
    float p = 0.0f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int q = int(threadIdx.x) + THREADS * j;
      if (q < nch) {
        float x[8], v[8], w[8], mu[8], xn[8];
        unpack8_f32(load8_f32(a.x + base + 8 * q, a.w32), x);
        unpack8_f32(load8_f32(a.v + base + 8 * q, a.w32), v);
        unpack8_f32(load8_f32(third + base + 8 * q, a.w32), w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float e = __fadd_rn(x[i], __fmul_rn(omt, v[i]));
          mu[i] = __fsub_rn(x[i], __fmul_rn(dt, __fadd_rn(v[i], __fmul_rn(kk, e))));
          xn[i] = a.z ? __fadd_rn(mu[i], __fmul_rn(sd, w[i])) : w[i];
        }
        if (a.z) store8_f32(a.x_next + base + 8 * q, xn, a.w32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float d = __fsub_rn(xn[i], mu[i]);
          p = __fadd_rn(p, __fmul_rn(d, d));
        }
      }
    }
    const float ss = cta_sum(p, wsum);
    if (threadIdx.x == 0) a.part[u] = ss;
  }
}

// The fused CFG + SDE step, launched as a dependent of the CFG's pass 1 (cfg_partials_kernel
// without a copy): per (request, segment) unit it waits for pass 1 once, folds the request's
// CFG sums (the same order as cfg_scale_kernel, so the same r), then chunk by chunk loads the
// branches, x and z, forms v = v2 r (c outside the window) in registers and runs the SDE
// step's arithmetic on it, exactly as sde_step_kernel would on the v that the two-call chain
// writes. Its sums of d d go to their own region. Nothing is loaded ahead of its chunk: at 63
// registers four CTAs fit on an SM, and their warps keep the loads in flight.
__global__ void __launch_bounds__(THREADS, 4) cfg_sde_kernel(const CfgArgs c, const SdeArgs a, float* v_out,
                                                             const int64_t units) {
  __shared__ float wsum[THREADS / 32];
  __shared__ float r_s;
  bool waited = false;
  pdl_trigger();  // the logp fold may start
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int req = int(u / a.S), seg = int(u % a.S);
    const float t = a.times[2 * req], tn = a.times[2 * req + 1];
    if (!times_ok(t, tn)) {
      if (threadIdx.x == 0 && seg == 0) atomicOr(a.err, MOT_DEV_BAD_TIME);
      continue;  // uniform across the CTA
    }
    const CfgPolicy pol = load_policy(c.policy + 6 * req);
    const bool guided = pol.guided();
    const int64_t base = int64_t(req) * a.N + int64_t(seg) * SEG;
    const int nch = int(min(int64_t(SEG), a.N - int64_t(seg) * SEG) / 8);
    const float* third = a.z ? a.z : a.x_next;
    const int kn = nch / THREADS + (int(threadIdx.x) < nch % THREADS ? 1 : 0);  // this thread's chunks
    float r = 1.0f;
    if (guided) {
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      if (threadIdx.x < 32) {
        const float rr = cfg_ratio(warp_fold2(c.part + int64_t(req) * a.S, a.S), pol.rmin);
        if (threadIdx.x == 0) r_s = rr;
      }
      __syncthreads();
      r = r_s;
    }
    const float dt = __fsub_rn(t, tn);
    const float sigma = t;
    const float kk = __fdiv_rn(__fmul_rn(sigma, sigma), __fmul_rn(2.0f, t));
    const float omt = __fsub_rn(1.0f, t);
    const float sd = __fmul_rn(sigma, __fsqrt_rn(dt));
    float p = 0.0f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      if (j < kn) {
        const int q = int(threadIdx.x) + THREADS * j;
        float v[8], x[8], w[8], mu[8], xn[8];
        if (guided) {
          CfgChunks k;
          k.c[j] = __ldg(reinterpret_cast<const uint4*>(c.c + base + 8 * q));
          k.tu[j] = __ldg(reinterpret_cast<const uint4*>(c.tu + base + 8 * q));
          if (c.iu) k.iu[j] = __ldg(reinterpret_cast<const uint4*>(c.iu + base + 8 * q));
          float cc[8];
          cfg_guide(c, pol, k, j, cc, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], r);
        } else {
          unpack8_bf16(__ldg(reinterpret_cast<const uint4*>(c.c + base + 8 * q)), v);
        }
        if (v_out) store8_f32(v_out + base + 8 * q, v, c.w32);
        unpack8_f32(load8_f32(a.x + base + 8 * q, a.w32), x);
        unpack8_f32(load8_f32(third + base + 8 * q, a.w32), w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float e = __fadd_rn(x[i], __fmul_rn(omt, v[i]));
          mu[i] = __fsub_rn(x[i], __fmul_rn(dt, __fadd_rn(v[i], __fmul_rn(kk, e))));
          xn[i] = a.z ? __fadd_rn(mu[i], __fmul_rn(sd, w[i])) : w[i];
        }
        if (a.z) store8_f32(a.x_next + base + 8 * q, xn, a.w32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float d = __fsub_rn(xn[i], mu[i]);
          p = __fadd_rn(p, __fmul_rn(d, d));
        }
      }
    }
    const float ss = cta_sum(p, wsum);  // its barriers also order r_s's reads before the next write
    if (threadIdx.x == 0) a.part[u] = ss;
  }
  if (!waited) pdl_wait();  // this grid completes only after pass 1 has
}

// logp = -(ss / (2 (std std))) - N (log(std) + log sqrt(2 pi)) with std = t sqrt(t - t_next).
__device__ __forceinline__ float sde_logp(float ss, float t, float tn, int64_t N) {
  const float sd = __fmul_rn(t, __fsqrt_rn(__fsub_rn(t, tn)));
  const float aa = __fdiv_rn(ss, __fmul_rn(2.0f, __fmul_rn(sd, sd)));
  const float lw = __fmul_rn(float(N), __fadd_rn(logf(sd), kLogSqrt2Pi));
  return __fsub_rn(-aa, lw);
}

// Launched as a dependent of the step: one warp per request folds the segment sums left to
// right, then forms logp.
__global__ void __launch_bounds__(128) sde_logp_kernel(const SdeArgs a) {
  const int req = int(blockIdx.x) * 4 + int(threadIdx.x >> 5);
  const bool live = req < a.n_req;
  float t = 0.0f, tn = 0.0f;
  if (live) {
    t = a.times[2 * req];
    tn = a.times[2 * req + 1];
  }
  pdl_wait();
  if (!live || !times_ok(t, tn)) return;  // uniform across the warp
  const float ss = warp_fold(a.part + int64_t(req) * a.S, a.S);
  if ((threadIdx.x & 31) == 0) a.logp[req] = sde_logp(ss, t, tn, a.N);
}

// ---------------------------------------------------------------------------
// Per-sample transition noise: Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011) and the Box-Muller transform
// ---------------------------------------------------------------------------
// Element 4b + m of request r at step k takes word m of the block with counter (b, k, 0, 0) and
// key (seed_r, kNoiseDomain); the top 23 bits give u = ((x >> 41) + 0.5) 2^-23, exact in fp32
// and inside (0, 1); pairs (u_even, u_odd) give sqrt(-2 ln u_even) (cos, sin)(2 pi u_odd).

constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull, kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull, kPhiloxW1 = 0xBB67AE8584CAA73Bull;
constexpr uint64_t kNoiseDomain = 0x4D6F54466C6F77ull;  // "MoTFlow"

__device__ __forceinline__ void philox4x64_10(uint64_t (&x)[4], uint64_t k0, uint64_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t hi0 = __umul64hi(kPhiloxM0, x[0]), lo0 = kPhiloxM0 * x[0];
    const uint64_t hi1 = __umul64hi(kPhiloxM1, x[2]), lo1 = kPhiloxM1 * x[2];
    x[0] = hi1 ^ x[1] ^ k0;
    x[1] = lo1;
    x[2] = hi0 ^ x[3] ^ k1;
    x[3] = lo0;
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
}

__device__ __forceinline__ float noise_uniform(uint64_t x) {
  return __fmul_rn(__fadd_rn(float(uint32_t(x >> 41)), 0.5f), 1.1920928955078125e-7f);  // 2^-23
}

__device__ __forceinline__ void box_muller(float u0, float u1, float& z0, float& z1) {
  const float rad = __fsqrt_rn(__fmul_rn(-2.0f, logf(u0)));
  float sn, cs;
  sincospif(__fmul_rn(2.0f, u1), &sn, &cs);
  z0 = __fmul_rn(rad, cs);
  z1 = __fmul_rn(rad, sn);
}

__global__ void __launch_bounds__(256) flow_noise_kernel(const uint64_t* seeds, uint64_t step, int n_req, int64_t N,
                                                         float* z) {
  const int64_t nb = N / 4;  // four deviates per block
  const int64_t total = int64_t(n_req) * nb;
  for (int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < total; u += int64_t(gridDim.x) * blockDim.x) {
    const int r = int(u / nb);
    const int64_t b = u % nb;
    uint64_t x[4] = {uint64_t(b), step, 0ull, 0ull};
    philox4x64_10(x, seeds[r], kNoiseDomain);
    float4 o;
    box_muller(noise_uniform(x[0]), noise_uniform(x[1]), o.x, o.y);
    box_muller(noise_uniform(x[2]), noise_uniform(x[3]), o.z, o.w);
    reinterpret_cast<float4*>(z + int64_t(r) * N)[b] = o;
  }
}

}  // namespace flow
}  // namespace mot

using namespace mot;

extern "C" size_t mot_flow_workspace_bytes(int n_req, int64_t N) {
  if (n_req < 1 || n_req > flow::kMaxReq || N < 8 || N % 8 != 0 || N > flow::kMaxN) return 0;
  return flow::workspace_bytes(n_req, N);
}

extern "C" int mot_flow_schedule_host(int n, double shift, float* host_t) {
  if (host_t == nullptr) return MOT_ERR_NULL;
  if (n < 2 || n > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (!(shift > 0.0) || !std::isfinite(shift)) return MOT_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    const double u = 1.0 - double(i) / double(n - 1);
    host_t[i] = float(shift * u / (1.0 + (shift - 1.0) * u));
  }
  return MOT_OK;
}

extern "C" int mot_cfg_combine_renorm(const mot_bf16* v_c, const mot_bf16* v_tu, const mot_bf16* v_iu, int n_req,
                                      int64_t N, const float* policy, void* ws, size_t ws_bytes, float* out,
                                      void* stream) {
  if (!v_c || !v_tu || !policy || !ws || !out) return MOT_ERR_NULL;
  if (n_req < 1 || n_req > flow::kMaxReq || N < 8 || N % 8 != 0 || N > flow::kMaxN) return MOT_ERR_GEOMETRY;
  if (!aligned16(v_c) || !aligned16(v_tu) || (v_iu && !aligned16(v_iu)) || !aligned16(policy) || !aligned16(ws) ||
      !aligned16(out))
    return MOT_ERR_ALIGN;
  if (ws_bytes < flow::workspace_bytes(n_req, N)) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {v_c, v_tu, v_iu, policy, ws, out};
  int dev = -1;
  int st = check_device(s, ptrs, 6, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const int S = flow::segments(N);
  flow::CfgArgs a{v_c, v_tu, v_iu, policy, N, S,
                  reinterpret_cast<float2*>(static_cast<char*>(ws) + sizeof(PlanHeader)), out,
                  reinterpret_cast<uintptr_t>(out) % 32 == 0 ? 1 : 0};
  const int64_t units = int64_t(n_req) * S;
  const unsigned grid = unsigned(std::min<int64_t>(units, int64_t(flow::kCtasPerSm) * sm_count(dev)));
  flow::cfg_partials_kernel<<<grid, flow::THREADS, 0, s>>>(a, units);
  if (cudaGetLastError() != cudaSuccess) return MOT_ERR_CUDA;
  if (launch_dependent(flow::cfg_scale_kernel, dim3(grid), dim3(flow::THREADS), 0, s, a, units) != cudaSuccess)
    return MOT_ERR_CUDA;
  return MOT_OK;
}

extern "C" int mot_flow_sde_step(const float* x, const float* v, const float* z, float* x_next, int n_req, int64_t N,
                                 const float* times, void* ws, size_t ws_bytes, float* logp, void* stream) {
  if (!x || !v || !x_next || !times || !ws || !logp) return MOT_ERR_NULL;
  if (n_req < 1 || n_req > flow::kMaxReq || N < 8 || N % 8 != 0 || N > flow::kMaxN) return MOT_ERR_GEOMETRY;
  if (!aligned16(x) || !aligned16(v) || (z && !aligned16(z)) || !aligned16(x_next) || !aligned16(times) ||
      !aligned16(ws) || !aligned16(logp))
    return MOT_ERR_ALIGN;
  if (ws_bytes < flow::workspace_bytes(n_req, N)) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {x, v, z, x_next, times, ws, logp};
  int dev = -1;
  int st = check_device(s, ptrs, 7, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const int S = flow::segments(N);
  const bool w32 = reinterpret_cast<uintptr_t>(x) % 32 == 0 && reinterpret_cast<uintptr_t>(v) % 32 == 0 &&
                   reinterpret_cast<uintptr_t>(z) % 32 == 0 && reinterpret_cast<uintptr_t>(x_next) % 32 == 0;
  flow::SdeArgs a{x, v, z, x_next, times, N, S, n_req,
                  reinterpret_cast<float*>(static_cast<char*>(ws) + sizeof(PlanHeader)), logp,
                  &static_cast<PlanHeader*>(ws)->error, w32 ? 1 : 0};
  const int64_t units = int64_t(n_req) * S;
  const unsigned grid = unsigned(std::min<int64_t>(units, int64_t(flow::kCtasPerSm) * sm_count(dev)));
  flow::sde_step_kernel<<<grid, flow::THREADS, 0, s>>>(a, units);
  if (cudaGetLastError() != cudaSuccess) return MOT_ERR_CUDA;
  if (launch_dependent(flow::sde_logp_kernel, dim3((n_req + 3) / 4), dim3(128), 0, s, a) != cudaSuccess)
    return MOT_ERR_CUDA;
  return MOT_OK;
}

extern "C" int mot_flow_cfg_sde_step(const mot_bf16* v_c, const mot_bf16* v_tu, const mot_bf16* v_iu,
                                     const float* policy, const float* x, const float* z, float* x_next, int n_req,
                                     int64_t N, const float* times, void* ws, size_t ws_bytes, float* v_out,
                                     float* logp, void* stream) {
  if (!v_c || !v_tu || !policy || !x || !x_next || !times || !ws || !logp) return MOT_ERR_NULL;
  if (n_req < 1 || n_req > flow::kMaxReq || N < 8 || N % 8 != 0 || N > flow::kMaxN) return MOT_ERR_GEOMETRY;
  if (!aligned16(v_c) || !aligned16(v_tu) || (v_iu && !aligned16(v_iu)) || !aligned16(policy) || !aligned16(x) ||
      (z && !aligned16(z)) || !aligned16(x_next) || !aligned16(times) || !aligned16(ws) || (v_out && !aligned16(v_out)) ||
      !aligned16(logp))
    return MOT_ERR_ALIGN;
  if (ws_bytes < flow::workspace_bytes(n_req, N)) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {v_c, v_tu, v_iu, policy, x, z, x_next, times, ws, v_out, logp};
  int dev = -1;
  int st = check_device(s, ptrs, 11, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const int S = flow::segments(N);
  char* scratch = static_cast<char*>(ws) + sizeof(PlanHeader);
  flow::CfgArgs ca{v_c, v_tu, v_iu, policy, N, S, reinterpret_cast<float2*>(scratch), nullptr,
                   v_out != nullptr && reinterpret_cast<uintptr_t>(v_out) % 32 == 0 ? 1 : 0};
  const bool w32 = reinterpret_cast<uintptr_t>(x) % 32 == 0 && reinterpret_cast<uintptr_t>(z) % 32 == 0 &&
                   reinterpret_cast<uintptr_t>(x_next) % 32 == 0;
  flow::SdeArgs sa{x, nullptr, z, x_next, times, N, S, n_req,
                   reinterpret_cast<float*>(scratch + flow::cfg_region_bytes(n_req, N)), logp,
                   &static_cast<PlanHeader*>(ws)->error, w32 ? 1 : 0};
  const int64_t units = int64_t(n_req) * S;
  const unsigned grid1 = unsigned(std::min<int64_t>(units, int64_t(flow::kCtasPerSm) * sm_count(dev)));
  const unsigned grid2 = unsigned(std::min<int64_t>(units, int64_t(4) * sm_count(dev)));
  flow::cfg_partials_kernel<<<grid1, flow::THREADS, 0, s>>>(ca, units);
  if (cudaGetLastError() != cudaSuccess) return MOT_ERR_CUDA;
  if (launch_dependent(flow::cfg_sde_kernel, dim3(grid2), dim3(flow::THREADS), 0, s, ca, sa, v_out, units) !=
      cudaSuccess)
    return MOT_ERR_CUDA;
  if (launch_dependent(flow::sde_logp_kernel, dim3((n_req + 3) / 4), dim3(128), 0, s, sa) != cudaSuccess)
    return MOT_ERR_CUDA;
  return MOT_OK;
}

extern "C" int mot_flow_noise(const uint64_t* seeds, uint64_t step, int n_req, int64_t N, float* z, void* stream) {
  if (!seeds || !z) return MOT_ERR_NULL;
  if (n_req < 1 || n_req > flow::kMaxReq || N < 8 || N % 8 != 0 || N > flow::kMaxN) return MOT_ERR_GEOMETRY;
  if (!aligned16(seeds) || !aligned16(z)) return MOT_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {seeds, z};
  int dev = -1;
  int st = check_device(s, ptrs, 2, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const int64_t total = int64_t(n_req) * (N / 4);
  const int64_t grid = std::min<int64_t>((total + 255) / 256, int64_t(8) * sm_count(dev));
  flow::flow_noise_kernel<<<unsigned(grid), 256, 0, s>>>(seeds, step, n_req, N, z);
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
