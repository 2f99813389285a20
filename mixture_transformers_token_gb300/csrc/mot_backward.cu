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
// add_rmsnorm_bwd_kernel   persistent, one CTA per SM, rows in the routing plan's order: a
//                          producer warp bulk-copies whole rows of s, dy (and d_res_out) into
//                          shared-memory slots; one consumer warp per slot runs the three passes
//                          (sum of s^2, dot, output) with lane l on columns 256 j + 8 l + t (the
//                          forward's tree layout), writes dx, the row's rstd and its partials.
// rmsnorm_dw_fold_kernel   one CTA per (folded weight set, 64-column block): the set's partials,
//                          left by the backward kernel as one contiguous run per column block,
//                          stream in by TMA tiles; two warps fold one column per thread over
//                          the set's rows in ascending order. Phase A of the BAGEL training
//                          rules trains the gen set only: the backward kernel then writes the
//                          gen rows' partials alone and the fold runs over the gen set alone.

#include <cuda.h>
#include <cuda_runtime.h>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {
namespace bwd {

struct NormBwdArgs {
  const uint16_t* dy;
  const uint16_t* s;
  const uint16_t* dro;  // may be null
  const uint16_t* w;    // [2][H]
  int T, H;
  float eps;
  uint4* dx;
  float* rstd;
  float* part;          // [H/64][T][64] per-row dweight partials by plan position, or null
  int psets;            // bit e: write the partials of the rows of weight set e
  const uint8_t* ws;    // the routing plan: rows are visited in its order
  uint32_t* err;
  int consumers;        // consumer warps = row slots
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

// Elements 2t and 2t + 1 of eight bf16 values, as fp32.
__device__ __forceinline__ float2 f2_of(const uint4& v, int t) {
  const uint32_t wd = t == 0 ? v.x : (t == 1 ? v.y : (t == 2 ? v.z : v.w));
  return make_float2(bf_lo(wd), bf_hi(wd));
}

// Two IEEE fp32 multiplies per instruction, each rounded as the scalar one would be; used only
// where the products feed further multiplies or scalar additions. The pairs move between
// float2 and the 64-bit register pair by mov.b64.
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  unsigned long long pa, pb, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pa), "l"(pb));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// One CTA per SM, persistent over the plan positions b + k G (b = blockIdx.x), so the
// weight-gradient partials of each weight set come out as one contiguous run. Warp 0 streams
// the whole rows of s, dy (and d_res_out) of those positions into C shared-memory slots with
// 1D bulk copies; consumer warp c owns slot c and takes every C-th position of the CTA. A
// consumer reads s, dy, the weights and d_res_out from shared memory in its three passes
// (independent products two at a time with packed fp32 multiplies, each rounded on its own;
// the sums in the tree's order), writes dx and rstd, and hands the slot back after the last
// pass.
constexpr int kBwdMaxConsumers = 8;
constexpr size_t kBwdSlotBudget = 180 * 1024;

template <int NJ>  // NJ >= H / 256
__global__ void __launch_bounds__(32 * (1 + kBwdMaxConsumers), 1) add_rmsnorm_bwd_kernel(const NormBwdArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int C = a.consumers;
  const uint32_t row_bytes = uint32_t(a.H) * 2;
  const int nrows = a.dro ? 3 : 2;  // rows per slot: s, dy (, d_res_out)
  uint8_t* wbuf = smem;                   // [2][H] norm weights
  uint8_t* slots = smem + 2 * row_bytes;  // C x nrows rows
  uint64_t* full = reinterpret_cast<uint64_t*>(slots + size_t(C) * nrows * row_bytes);
  uint64_t* empty = full + kBwdMaxConsumers;
  uint64_t* wbar = empty + kBwdMaxConsumers;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(wbar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = int(blockIdx.x), G = int(gridDim.x);
  // a programmatic dependent: launched while the preceding grid (the input gradient's GEMM)
  // runs, it reads nothing before that grid has completed
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int c = 0; c < C; ++c) {
      mbar_init(smem_u32(&full[c]), 1);
      mbar_init(smem_u32(&empty[c]), 1);
    }
    mbar_init(smem_u32(wbar), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();

  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(a.ws);
  if (hdr->magic != kPlanMagic || hdr->T != a.T) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.err, MOT_DEV_PLAN_MISMATCH);
    return;  // uniform across the grid
  }
  if (hdr->count[0] + hdr->count[1] != a.T) return;  // no plan (bad modality): nothing is defined
  const int32_t* perm = reinterpret_cast<const int32_t*>(a.ws + perm_offset());
  const int count0 = hdr->count[0];

  if (warp == 0) {
    // ---------------- producer: plan positions b + k G, their rows read 32 ahead ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(wbar), 2 * row_bytes);
      bulk_load(smem_u32(wbuf), a.w, 2 * row_bytes, smem_u32(wbar));
    }
    int issued = 0;
    bool ok = true;
    for (int k0 = 0; ok; k0 += 32) {
      const int64_t mine = int64_t(b) + int64_t(k0 + lane) * G;
      const int my_row = mine < a.T ? perm[mine] : -1;
      for (int q = 0; q < 32; ++q) {
        const int k = k0 + q;
        const int row = __shfl_sync(0xffffffffu, my_row, q);
        if (row < 0) {
          ok = false;
          break;
        }
        const int c = k % C;
        const uint32_t round = uint32_t(k / C);
        if (lane == 0) {
          if (!mbar_wait(smem_u32(&empty[c]), (round & 1u) ^ 1u, abort_flag, a.err)) {
            ok = false;
          } else {
            uint8_t* slot = slots + size_t(c) * nrows * row_bytes;
            const uint32_t fb = smem_u32(&full[c]);
            const int64_t off = int64_t(row) * a.H;  // elements
            mbar_arrive_expect_tx(fb, uint32_t(nrows) * row_bytes);
            bulk_load(smem_u32(slot), a.s + off, row_bytes, fb);
            bulk_load(smem_u32(slot + row_bytes), a.dy + off, row_bytes, fb);
            if (a.dro) bulk_load(smem_u32(slot + 2 * row_bytes), a.dro + off, row_bytes, fb);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        issued = k + 1;
      }
    }
    // no copy may still be landing when the CTA exits: wait for the last fill of every slot
    if (lane == 0) {
      mbar_drain(smem_u32(wbar), 0);
      for (int k = issued - C > 0 ? issued - C : 0; k < issued; ++k)
        mbar_drain(smem_u32(&full[k % C]), uint32_t(k / C) & 1u);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int c = warp - 1;
  if (c >= C) return;
  const int nj = a.H >> 8, h8 = a.H >> 3;
  const float fH = float(a.H);
  const uint4* ss4 = reinterpret_cast<const uint4*>(slots + size_t(c) * nrows * row_bytes);
  const uint4* sd4 = ss4 + h8;
  const uint4* sr4 = ss4 + 2 * h8;
  if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(wbar), 0, abort_flag, a.err))) return;
  for (int k = c;; k += C) {
    const int64_t pos = int64_t(b) + int64_t(k) * G;  // plan position
    if (pos >= a.T) break;
    const int64_t row = perm[pos];
    const int e = pos < count0 ? 0 : 1;
    const bool wpart = a.part != nullptr && ((a.psets >> e) & 1) != 0;  // this row's partials are wanted
    const uint32_t round = uint32_t(k / C);
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[c]), round & 1u, abort_flag, a.err))) break;
    {
      // pass 1: sum of s^2 on the forward's tree (lane l: columns 256 j + 8 l + t, j outer)
      float ss = 0.0f;
#pragma unroll 2
      for (int j = 0; j < nj; ++j) {
        const uint4 s1 = ss4[32 * j + lane];
        float2 sq[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) sq[t] = f2_mul(f2_of(s1, t), f2_of(s1, t));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          ss = __fadd_rn(ss, sq[t].x);
          ss = __fadd_rn(ss, sq[t].y);
        }
      }
      ss = warp_tree(ss);
      const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, fH), a.eps)));
      const float2 rstd2 = make_float2(rstd, rstd);
      // pass 2: dot = sum of (dy * w) * (s * rstd) on the same tree
      const uint4* wrow = reinterpret_cast<const uint4*>(wbuf + size_t(e) * row_bytes);
      float dot = 0.0f;
#pragma unroll 2
      for (int j = 0; j < nj; ++j) {
        const uint4 wv = wrow[32 * j + lane], d = sd4[32 * j + lane], sj = ss4[32 * j + lane];
        float2 pr[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          pr[t] = f2_mul(f2_mul(f2_of(d, t), f2_of(wv, t)), f2_mul(f2_of(sj, t), rstd2));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          dot = __fadd_rn(dot, pr[t].x);
          dot = __fadd_rn(dot, pr[t].y);
        }
      }
      dot = warp_tree(dot);
      const float cc = __fdiv_rn(dot, fH);
      // pass 3: ds = rstd * (g - xh * c) (+ d_res_out), one cast; partials dy * xh
      uint4* orow = a.dx + row * h8 + lane;
#pragma unroll 2
      for (int j = 0; j < nj; ++j) {
        const uint4 wv = wrow[32 * j + lane], d = sd4[32 * j + lane], sj = ss4[32 * j + lane];
        const uint4 rv = a.dro ? sr4[32 * j + lane] : make_uint4(0u, 0u, 0u, 0u);
        uint32_t ow[4];
        float2 pp[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 dd = f2_of(d, t);
          const float2 xh = f2_mul(f2_of(sj, t), rstd2);
          const float2 g = f2_mul(dd, f2_of(wv, t));
          const float2 r = f2_of(rv, t);
          // a product that feeds an addition stays a scalar multiply, so no multiply-add can
          // take its place
          float ds0 = __fmul_rn(rstd, __fsub_rn(g.x, __fmul_rn(xh.x, cc)));
          float ds1 = __fmul_rn(rstd, __fsub_rn(g.y, __fmul_rn(xh.y, cc)));
          if (a.dro) {
            ds0 = __fadd_rn(ds0, r.x);
            ds1 = __fadd_rn(ds1, r.y);
          }
          ow[t] = pack_bf2(ds0, ds1);
          pp[t] = f2_mul(dd, xh);
        }
        if (wpart) {
          // columns 256 j + 8 lane + t: block 4 j + lane / 8, offset 8 (lane % 8) + t
          float4* pd = reinterpret_cast<float4*>(a.part + ((int64_t(4 * j + (lane >> 3)) * a.T + pos) << 6) +
                                                 8 * (lane & 7));
          __stcs(pd, make_float4(pp[0].x, pp[0].y, pp[1].x, pp[1].y));
          __stcs(pd + 1, make_float4(pp[2].x, pp[2].y, pp[3].x, pp[3].y));
        }
        __stcs(orow + 32 * j, make_uint4(ow[0], ow[1], ow[2], ow[3]));
      }
      if (lane == 0) a.rstd[row] = rstd;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[c]));
  }
}

// Weight-gradient fold. The backward kernel leaves the per-row partials p = dy * (s * rstd)
// in fp32 blocks of 64 columns by plan position, part[cb][i][64], so the rows of a weight set
// in a column block are one contiguous run in ascending row order. One CTA per (set, block):
// warp 0 streams 128-row tiles of the run (32 KB) with TMA into a ring of kFoldStages slots
// (larger tiles halve the per-tile barrier handshakes on the fold's critical path); warps 1
// and 2 fold 32 columns each, one column per thread.
constexpr int kFoldCols = 64, kFoldRows = 128, kFoldStages = 4;
constexpr int kFoldThreads = 32 * 3;
constexpr uint32_t kFoldPartBytes = kFoldRows * kFoldCols * 4;  // 32 KB
constexpr size_t kFoldSmem = 128 + kFoldStages * size_t(kFoldPartBytes) + 2 * kFoldStages * 8 + 16;

struct FoldArgs {
  const uint8_t* ws;
  int T, H;
  int set_lo;  // the first weight set folded; the grid covers it and the sets after it
  float* dw;
  uint32_t* err;
};

__device__ __forceinline__ void tma_load_2d_cta(uint32_t dst, const void* tmap, int32_t x, int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__global__ void __launch_bounds__(kFoldThreads) rmsnorm_dw_fold_kernel(const __grid_constant__ CUtensorMap tm_part,
                                                                      const FoldArgs a) {
  extern __shared__ __align__(128) uint8_t fraw[];
  uint8_t* fsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fraw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(fsm + kFoldStages * size_t(kFoldPartBytes));
  uint64_t* empty = full + kFoldStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + kFoldStages);
  pdl_trigger();  // a programmatic dependent: nothing is read before the preceding grid completes
  pdl_wait();
  const int ncb = a.H / kFoldCols;
  const int e = a.set_lo + int(blockIdx.x) / ncb, cb = int(blockIdx.x) % ncb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(a.ws);
  if (hdr->magic != kPlanMagic || hdr->T != a.T) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.err, MOT_DEV_PLAN_MISMATCH);
    return;
  }
  if (hdr->count[0] + hdr->count[1] != a.T) return;  // no plan (bad modality): nothing is defined
  const int start = e == 0 ? 0 : hdr->count[0];
  const int count = hdr->count[e];
  const int nst = (count + kFoldRows - 1) / kFoldRows;
  if (threadIdx.x == 0) {
    for (int sl = 0; sl < kFoldStages; ++sl) {
      mbar_init(smem_u32(&full[sl]), 1);
      mbar_init(smem_u32(&empty[sl]), 2);  // the two fold warps
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int issued = 0;
      for (int k = 0; k < nst; ++k) {
        const int slot = k % kFoldStages;
        const uint32_t round = uint32_t(k / kFoldStages);
        if (!mbar_wait(smem_u32(&empty[slot]), (round & 1u) ^ 1u, abort_flag, a.err)) break;
        const uint32_t fb = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(fb, kFoldPartBytes);
        tma_load_2d_cta(smem_u32(fsm + size_t(slot) * kFoldPartBytes), &tm_part, 0,
                        cb * a.T + start + k * kFoldRows, fb);
        issued = k + 1;
      }
      for (int k = issued - kFoldStages > 0 ? issued - kFoldStages : 0; k < issued; ++k)
        mbar_drain(smem_u32(&full[k % kFoldStages]), uint32_t(k / kFoldStages) & 1u);
    }
    return;
  }
  // ---------------- folds: warp 1 columns 0..31, warp 2 columns 32..63 ----------------
  const int col = (warp - 1) * 32 + lane;
  float acc = -0.0f;  // -0 + p = p for every p: the fold starts with the set's first partial
  bool ok = true;
  for (int k = 0; k < nst; ++k) {
    const int slot = k % kFoldStages;
    const uint32_t round = uint32_t(k / kFoldStages);
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[slot]), round & 1u, abort_flag, a.err));
    if (!ok) break;
    const float* sp = reinterpret_cast<const float*>(fsm + size_t(slot) * kFoldPartBytes);
    const int n = count - k * kFoldRows < kFoldRows ? count - k * kFoldRows : kFoldRows;
    if (n == kFoldRows) {
#pragma unroll
      for (int rr = 0; rr < kFoldRows; ++rr) acc = __fadd_rn(acc, sp[rr * kFoldCols + col]);
    } else {
      for (int rr = 0; rr < n; ++rr) acc = __fadd_rn(acc, sp[rr * kFoldCols + col]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
  }
  if (ok) a.dw[int64_t(e) * a.H + cb * kFoldCols + col] = count > 0 ? acc : 0.0f;
}

template <int NJ>
static cudaError_t launch_bwd(const NormBwdArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaError_t st = cudaFuncSetAttribute(add_rmsnorm_bwd_kernel<NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(smem));
  if (st != cudaSuccess) return st;
  return launch_dependent(add_rmsnorm_bwd_kernel<NJ>, dim3(grid), dim3(32 * (1 + a.consumers)), smem, s, a);
}

}  // namespace bwd
}  // namespace mot

using namespace mot;

extern "C" int mot_add_rmsnorm_backward(const mot_bf16* dy, const mot_bf16* d_res_out, const mot_bf16* s,
                                        const mot_bf16* w, int64_t T, int H, float eps, void* ws, size_t ws_bytes,
                                        mot_bf16* dx, float* rstd, float* dw_partials, int partial_sets,
                                        void* stream) {
  if (!dy || !s || !w || !ws || !dx || !rstd) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || H < 256 || H > 8192 || H % 256 != 0) return MOT_ERR_GEOMETRY;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return MOT_ERR_ARG;
  if (dw_partials && (partial_sets < MOT_SET_UND || partial_sets > MOT_SET_BOTH)) return MOT_ERR_ARG;
  if (!aligned16(dy) || (d_res_out && !aligned16(d_res_out)) || !aligned16(s) || !aligned16(w) || !aligned16(ws) ||
      !aligned16(dx) || !aligned16(rstd) || (dw_partials && !aligned16(dw_partials)))
    return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {dy, d_res_out, s, w, ws, dx, rstd, dw_partials};
  int dev = -1;
  int rc = check_device(st, ptrs, 8, &dev);
  if (rc != MOT_OK) return rc;
  DeviceGuard guard(dev);
  bwd::NormBwdArgs a{};
  a.dy = dy;
  a.s = s;
  a.dro = d_res_out;
  a.w = w;
  a.T = int(T);
  a.H = H;
  a.eps = eps;
  a.dx = reinterpret_cast<uint4*>(dx);
  a.rstd = rstd;
  a.part = dw_partials;
  a.psets = partial_sets;
  a.ws = static_cast<const uint8_t*>(ws);
  a.err = &static_cast<PlanHeader*>(ws)->error;
  const size_t row_bytes = size_t(H) * 2;
  const int nrows = d_res_out ? 3 : 2;
  int C = int(bwd::kBwdSlotBudget / (nrows * row_bytes));
  C = C > bwd::kBwdMaxConsumers ? bwd::kBwdMaxConsumers : C;
  a.consumers = C;
  const size_t smem =
      2 * row_bytes + size_t(C) * nrows * row_bytes + (2 * bwd::kBwdMaxConsumers + 2) * sizeof(uint64_t);
  const int sms = sm_count(dev);
  const int grid = int(T < sms ? T : sms);
  const int nj = H / 256;
  cudaError_t e;
  if (nj <= 4)
    e = bwd::launch_bwd<4>(a, grid, smem, st);
  else if (nj <= 8)
    e = bwd::launch_bwd<8>(a, grid, smem, st);
  else if (nj <= 16)
    e = bwd::launch_bwd<16>(a, grid, smem, st);
  else
    e = bwd::launch_bwd<32>(a, grid, smem, st);
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

extern "C" int mot_rmsnorm_dweight(const float* dw_partials, int64_t T, int H, int sets, void* ws, size_t ws_bytes,
                                   float* dw, void* stream) {
  if (!dw_partials || !ws || !dw) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || H < 256 || H > 8192 || H % 256 != 0) return MOT_ERR_GEOMETRY;
  if (sets < MOT_SET_UND || sets > MOT_SET_BOTH) return MOT_ERR_ARG;
  if (!aligned16(dw_partials) || !aligned16(ws) || !aligned16(dw)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {dw_partials, ws, dw};
  int dev = -1;
  int rc = check_device(st, ptrs, 3, &dev);
  if (rc != MOT_OK) return rc;
  DeviceGuard guard(dev);
  if (cudaFuncSetAttribute(bwd::rmsnorm_dw_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(bwd::kFoldSmem)) != cudaSuccess)
    return MOT_ERR_CUDA;
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return MOT_ERR_CUDA;
  // the partials as a 2D fp32 tensor of (H / 64) * T rows of 64 columns
  CUtensorMap tm_part;
  cuuint64_t dims[2] = {uint64_t(bwd::kFoldCols), uint64_t(H / bwd::kFoldCols) * uint64_t(T)};
  cuuint64_t strides[1] = {uint64_t(bwd::kFoldCols) * 4};
  cuuint32_t box[2] = {uint32_t(bwd::kFoldCols), uint32_t(bwd::kFoldRows)};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&tm_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(dw_partials), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MOT_ERR_CUDA;
  bwd::FoldArgs a{};
  a.ws = static_cast<const uint8_t*>(ws);
  a.T = int(T);
  a.H = H;
  a.dw = dw;
  a.err = &static_cast<PlanHeader*>(ws)->error;
  a.set_lo = sets == MOT_SET_GEN ? 1 : 0;
  const int nsets = sets == MOT_SET_BOTH ? 2 : 1;
  const cudaError_t e = launch_dependent(bwd::rmsnorm_dw_fold_kernel, dim3(nsets * (H / bwd::kFoldCols)),
                                         dim3(bwd::kFoldThreads), bwd::kFoldSmem, st, tm_part, a);
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
