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
// Each thread owns a contiguous segment of rows, so a block-wide scan of the und counts gives
// every row its slot in the stable ascending lists. Works for any block of 32..1024 threads.
__device__ void route_plan_block(const uint8_t* __restrict__ mod, int T, uint8_t* __restrict__ ws) {
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + perm_offset());
  Tile* tiles = reinterpret_cast<Tile*>(ws + tiles_offset(T));
  __shared__ int warp_incl[32];

  const int nthr = blockDim.x, nwarps = nthr >> 5;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (T + nthr - 1) / nthr;
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
    int v = lane < nwarps ? warp_incl[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += u;
    }
    warp_incl[lane] = v;
  }
  __syncthreads();
  const int total_und = warp_incl[nwarps - 1];
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
  for (int t = tid; t < nt0 + nt1; t += nthr) {
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

constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) route_plan_kernel(const uint8_t* __restrict__ mod, int T,
                                                                    uint8_t* __restrict__ ws) {
  route_plan_block(mod, T, ws);
}

// ---------------------------------------------------------------------------
// routing pre-pass over many CTAs, for packs above kPlanOneCta rows: the same plan, built by
// four small kernels. Block b owns rows [b C, b C + C) with C = kPlanChunk; within a block,
// round i covers rows b C + 256 i + t (thread t), so every load of the modality bytes is
// coalesced and a block-wide prefix over each round keeps the lists stable.
//   plan_count_kernel    und rows per block (-1 for a block with a bad modality byte), into
//                        the tile table's space, which is rewritten last
//   plan_scan_kernel     one CTA: the exclusive prefix of the und counts, the header
//   plan_scatter_kernel  every row to its slot: und rows ascending, then gen rows ascending
//   plan_tiles_kernel    the 128-row tile records, as route_plan_block writes them
// ---------------------------------------------------------------------------
constexpr int kPlanOneCta = 65536;
constexpr int kPlanThreads = 256;
constexpr int kPlanRounds = 32;
constexpr int kPlanChunk = kPlanThreads * kPlanRounds;  // 8192 rows per block

__device__ __forceinline__ int32_t* plan_block_scratch(uint8_t* ws, int T) {
  return reinterpret_cast<int32_t*>(ws + tiles_offset(T));
}

__global__ void __launch_bounds__(kPlanThreads) plan_count_kernel(const uint8_t* __restrict__ mod, int T,
                                                                   uint8_t* __restrict__ ws) {
  __shared__ int wsum[kPlanThreads / 32];
  const int b = int(blockIdx.x), t = int(threadIdx.x);
  const int64_t base = int64_t(b) * kPlanChunk;
  int n_und = 0, bad = 0;
#pragma unroll 4
  for (int i = 0; i < kPlanRounds; ++i) {
    const int64_t r = base + int64_t(i) * kPlanThreads + t;
    if (r < T) {
      const int m = mod[r];
      bad |= (m > 1);
      n_und += (m == 0);
    }
  }
  bad = __syncthreads_or(bad);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) n_und += __shfl_xor_sync(0xffffffffu, n_und, off);
  if ((t & 31) == 0) wsum[t >> 5] = n_und;
  __syncthreads();
  if (t == 0) {
    int tot = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) tot += wsum[w];
    plan_block_scratch(ws, T)[b] = bad ? -1 : tot;
  }
}

__global__ void __launch_bounds__(1024) plan_scan_kernel(int T, int nblocks, uint8_t* __restrict__ ws) {
  __shared__ int warp_incl[32];
  int32_t* cnt = plan_block_scratch(ws, T);
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  // thread tid owns blocks [tid k, tid k + k), k = ceil(nblocks / 1024)
  const int k = (nblocks + 1023) / 1024;
  const int begin = min(tid * k, nblocks), end = min(begin + k, nblocks);
  int sum = 0, bad = 0;
  for (int i = begin; i < end; ++i) {
    const int c = cnt[i];
    bad |= (c < 0);
    sum += c < 0 ? 0 : c;
  }
  bad = __syncthreads_or(bad);
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
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_incl[warp] = incl;
  __syncthreads();
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
  int run = (warp > 0 ? warp_incl[warp - 1] : 0) + incl - sum;  // und rows before block `begin`
  for (int i = begin; i < end; ++i) {
    const int c = cnt[i];
    cnt[i] = run;  // und rows before block i
    run += c;
  }
  if (tid == 0) {
    const int total_gen = T - total_und;
    hdr->T = T;
    hdr->count[0] = total_und;
    hdr->count[1] = total_gen;
    hdr->num_m_tiles = (total_und + kTileRows - 1) / kTileRows + (total_gen + kTileRows - 1) / kTileRows;
    hdr->error = 0;
    hdr->magic = kPlanMagic;
  }
}

__global__ void __launch_bounds__(kPlanThreads) plan_scatter_kernel(const uint8_t* __restrict__ mod, int T,
                                                                     uint8_t* __restrict__ ws) {
  __shared__ int wcnt[kPlanThreads / 32];
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(ws);
  if (hdr->error != 0) return;  // bad modality: no lists (uniform across the grid)
  int32_t* perm = reinterpret_cast<int32_t*>(ws + perm_offset());
  const int b = int(blockIdx.x), t = int(threadIdx.x), lane = t & 31, warp = t >> 5;
  const int64_t base = int64_t(b) * kPlanChunk;
  const int total_und = hdr->count[0];
  int und = plan_block_scratch(ws, T)[b];     // und rows before this block's next round
  int gen = int(base) - und;                  // gen rows before it
  for (int i = 0; i < kPlanRounds; ++i) {
    const int64_t r = base + int64_t(i) * kPlanThreads + t;
    if (base + int64_t(i) * kPlanThreads >= T) break;  // uniform across the block
    const bool live = r < T;
    const bool is_und = live && mod[r] == 0;
    const uint32_t bu = __ballot_sync(0xffffffffu, is_und), bl = __ballot_sync(0xffffffffu, live);
    if (lane == 0) wcnt[warp] = __popc(bu);
    __syncthreads();
    int und_before = und, live_before = 0;
    for (int w = 0; w < warp; ++w) und_before += wcnt[w];
    live_before = min(max(int(T - (base + int64_t(i) * kPlanThreads)), 0), warp * 32);  // live rows of earlier warps
    const uint32_t lt = (1u << lane) - 1u;
    und_before += __popc(bu & lt);
    const int gen_before = gen + live_before + __popc(bl & lt) - (und_before - und);
    if (live) perm[is_und ? und_before : total_und + gen_before] = int32_t(r);
    int round_und = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) round_und += wcnt[w];
    const int round_live = int(min(int64_t(kPlanThreads), T - (base + int64_t(i) * kPlanThreads)));
    __syncthreads();  // wcnt is rewritten by the next round
    und += round_und;
    gen += round_live - round_und;
  }
}

__global__ void __launch_bounds__(kPlanThreads) plan_tiles_kernel(int T, uint8_t* __restrict__ ws) {
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(ws);
  if (hdr->error != 0) return;
  const int32_t* perm = reinterpret_cast<const int32_t*>(ws + perm_offset());
  Tile* tiles = reinterpret_cast<Tile*>(ws + tiles_offset(T));
  const int total_und = hdr->count[0], total_gen = hdr->count[1];
  const int nt0 = (total_und + kTileRows - 1) / kTileRows;
  const int nt1 = (total_gen + kTileRows - 1) / kTileRows;
  for (int t = int(blockIdx.x) * kPlanThreads + int(threadIdx.x); t < nt0 + nt1; t += int(gridDim.x) * kPlanThreads) {
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
}

// ---------------------------------------------------------------------------
// fused residual add + routed RMSNorm, fed by bulk copies through shared memory
// ---------------------------------------------------------------------------
// One CTA per SM, persistent over rows (blockIdx.x - 1) + k G. Warp 0 streams whole rows of x
// and res into C shared-memory slots with 1D bulk copies (cp.async.bulk); consumer warp c owns
// slot c and processes every C-th row of the CTA, keeping the row's s = bf16(x + res) in
// registers so the slot returns to the producer right after the first pass; the norm weights
// of both experts are copied into shared memory once per CTA. The arithmetic of a row is the
// fixed tree: lane l owns columns 256 j + 8 l + t, sequential fp32 sum of s^2 (j outer, t
// inner), xor butterfly 16, 8, 4, 2, 1. When a workspace is given, CTA 0 of the same launch
// builds the routing plan (it is scheduled first and has an SM of its own).
constexpr int kNormMaxConsumers = 12;
constexpr size_t kNormSlotBudget = 180 * 1024;

struct NormArgs {
  const uint16_t* x;
  const uint16_t* res;
  const uint16_t* w;
  const uint8_t* mod;
  int T, H;
  float eps;
  uint16_t* y;
  uint16_t* res_out;
  uint32_t* err;     // error word or null
  uint8_t* plan_ws;  // if not null, CTA 0 writes the routing plan here
  int norm_blocks;
  int consumers;     // consumer warps = row slots
};

template <int NJ>
__global__ void __launch_bounds__(32 * (1 + kNormMaxConsumers), 1) add_rmsnorm_kernel(const NormArgs a) {
  pdl_trigger();  // a dependent GEMM may be scheduled now; it waits for this grid before any read
  const int plan_ctas = a.plan_ws != nullptr ? 1 : 0;
  if (int(blockIdx.x) < plan_ctas) {
    route_plan_block(a.mod, a.T, a.plan_ws);
    return;
  }
  const int b = int(blockIdx.x) - plan_ctas;
  extern __shared__ __align__(128) uint8_t smem[];
  const int C = a.consumers;
  const uint32_t row_bytes = uint32_t(a.H) * 2;
  uint8_t* wbuf = smem;                   // [2][H] norm weights
  uint8_t* slots = smem + 2 * row_bytes;  // C x (x row, res row)
  uint64_t* full = reinterpret_cast<uint64_t*>(slots + size_t(C) * 2 * row_bytes);
  uint64_t* empty = full + kNormMaxConsumers;
  uint64_t* wbar = empty + kNormMaxConsumers;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(wbar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.norm_blocks;
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

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_u32(wbar), 2 * row_bytes);
      bulk_load(smem_u32(wbuf), a.w, 2 * row_bytes, smem_u32(wbar));
      int issued = 0;
      for (int k = 0;; ++k) {
        const int64_t row = int64_t(b) + int64_t(k) * G;
        if (row >= a.T) break;
        const int c = k % C;
        const uint32_t round = uint32_t(k / C);
        if (!mbar_wait(smem_u32(&empty[c]), (round & 1u) ^ 1u, abort_flag, a.err)) break;
        uint8_t* slot = slots + size_t(c) * 2 * row_bytes;
        const uint32_t fb = smem_u32(&full[c]);
        mbar_arrive_expect_tx(fb, 2 * row_bytes);
        bulk_load(smem_u32(slot), a.x + row * a.H, row_bytes, fb);
        bulk_load(smem_u32(slot + row_bytes), a.res + row * a.H, row_bytes, fb);
        issued = k + 1;
      }
      // no copy may still be landing when the CTA exits: wait for the last fill of every slot
      mbar_drain(smem_u32(wbar), 0);
      for (int k = issued - C > 0 ? issued - C : 0; k < issued; ++k)
        mbar_drain(smem_u32(&full[k % C]), uint32_t(k / C) & 1u);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int c = warp - 1;
  if (c >= C) return;
  const int nj = a.H >> 8;
  const uint4* sx = reinterpret_cast<const uint4*>(slots + size_t(c) * 2 * row_bytes);
  const uint4* sr = reinterpret_cast<const uint4*>(slots + size_t(c) * 2 * row_bytes + row_bytes);
  if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(wbar), 0, abort_flag, a.err))) return;
  for (int k = c;; k += C) {
    const int64_t row = int64_t(b) + int64_t(k) * G;
    if (row >= a.T) break;
    const int m = a.mod[row];
    const uint32_t round = uint32_t(k / C);
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[c]), round & 1u, abort_flag, a.err))) break;
    const int64_t base = row * (a.H >> 3);  // row start in 16-byte units
    uint4* ro = reinterpret_cast<uint4*>(a.res_out) + base;
    uint4 sv[NJ];
    float p = 0.0f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (j < nj) {
        const uint4 xv4 = sx[32 * j + lane], rv4 = sr[32 * j + lane];
        const uint32_t xv[4] = {xv4.x, xv4.y, xv4.z, xv4.w};
        const uint32_t rv[4] = {rv4.x, rv4.y, rv4.z, rv4.w};
        uint32_t s4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          s4[q] = pack_bf2(__fadd_rn(bf_lo(xv[q]), bf_lo(rv[q])), __fadd_rn(bf_hi(xv[q]), bf_hi(rv[q])));
          const float s0 = bf_lo(s4[q]), s1 = bf_hi(s4[q]);
          p = __fadd_rn(p, __fmul_rn(s0, s0));  // t = 2q
          p = __fadd_rn(p, __fmul_rn(s1, s1));  // t = 2q + 1
        }
        sv[j] = make_uint4(s4[0], s4[1], s4[2], s4[3]);
        __stcs(ro + 32 * j + lane, sv[j]);
      }
    }
    // the row now lives in registers: hand the slot back to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[c]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, off));
    if (m <= 1) {
      const float ms = __fdiv_rn(p, float(a.H));
      const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
      const uint4* wv = reinterpret_cast<const uint4*>(wbuf + size_t(m) * row_bytes);
      uint4* yo = reinterpret_cast<uint4*>(a.y) + base;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (j < nj) {
          const uint4 ww = wv[32 * j + lane];
          const uint32_t s4[4] = {sv[j].x, sv[j].y, sv[j].z, sv[j].w};
          const uint32_t wq[4] = {ww.x, ww.y, ww.z, ww.w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            o[q] = pack_bf2(__fmul_rn(__fmul_rn(bf_lo(s4[q]), rstd), bf_lo(wq[q])),
                            __fmul_rn(__fmul_rn(bf_hi(s4[q]), rstd), bf_hi(wq[q])));
          yo[32 * j + lane] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    } else if (lane == 0 && a.err != nullptr && a.plan_ws == nullptr) {
      atomicOr(a.err, MOT_DEV_BAD_MODALITY);  // with a plan CTA in the launch, the plan reports it
    }
  }
}

template <int NJ>
static cudaError_t launch_norm(const NormArgs& a, int grid, size_t smem, cudaStream_t s) {
  if (cudaFuncSetAttribute(add_rmsnorm_kernel<NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return cudaErrorInvalidValue;
  add_rmsnorm_kernel<NJ><<<grid, 32 * (1 + a.consumers), smem, s>>>(a);
  return cudaGetLastError();
}

// dst[i] = src[perm[i]]: one warp per row, 16-byte vectors, persistent grid
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src, int T, int K8,
                                                          const uint8_t* __restrict__ ws, uint4* __restrict__ dst) {
  // a programmatic dependent: launched while the preceding grid runs, it reads nothing before
  // that grid has completed
  pdl_trigger();
  pdl_wait();
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(ws);
  if (hdr->magic != kPlanMagic || hdr->T != T) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(const_cast<uint32_t*>(&hdr->error), MOT_DEV_PLAN_MISMATCH);
    return;
  }
  if (hdr->count[0] + hdr->count[1] != T) return;  // no plan (bad modality): nothing is defined
  const int32_t* perm = reinterpret_cast<const int32_t*>(ws + perm_offset());
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int64_t i = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < T; i += warps) {
    const uint4* s = src + int64_t(perm[i]) * K8;
    uint4* d = dst + i * K8;
    int k = lane;
    for (; k + 96 < K8; k += 128) {  // four loads in flight per lane
      const uint4 v0 = __ldcs(s + k), v1 = __ldcs(s + k + 32), v2 = __ldcs(s + k + 64), v3 = __ldcs(s + k + 96);
      __stcs(d + k, v0);
      __stcs(d + k + 32, v1);
      __stcs(d + k + 64, v2);
      __stcs(d + k + 96, v3);
    }
    for (; k < K8; k += 32) __stcs(d + k, __ldcs(s + k));
  }
}

int enqueue_route_plan(const uint8_t* mod, int T, uint8_t* ws, cudaStream_t s) {
  if (T <= kPlanOneCta) {
    route_plan_kernel<<<1, kRouteThreads, 0, s>>>(mod, T, ws);
    return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
  }
  const int nblocks = (T + kPlanChunk - 1) / kPlanChunk;  // <= 2048 for T <= MOT_MAX_TOKENS
  plan_count_kernel<<<nblocks, kPlanThreads, 0, s>>>(mod, T, ws);
  plan_scan_kernel<<<1, 1024, 0, s>>>(T, nblocks, ws);
  plan_scatter_kernel<<<nblocks, kPlanThreads, 0, s>>>(mod, T, ws);
  const int ntiles = int(max_m_tiles(T));
  plan_tiles_kernel<<<(ntiles + kPlanThreads - 1) / kPlanThreads, kPlanThreads, 0, s>>>(T, ws);
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
  return enqueue_route_plan(mod, int(T), static_cast<uint8_t*>(ws), s);
}

extern "C" int mot_fused_add_rmsnorm(const mot_bf16* x, const mot_bf16* res, const mot_bf16* w,
                                     const uint8_t* mod, int64_t T, int H, float eps, mot_bf16* y,
                                     mot_bf16* res_out, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !res || !w || !mod || !y || !res_out) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || H < 256 || H > 8192 || H % 256 != 0) return MOT_ERR_GEOMETRY;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return MOT_ERR_ARG;
  if (!aligned16(x) || !aligned16(res) || !aligned16(w) || !aligned16(y) || !aligned16(res_out) ||
      (ws && !aligned16(ws)))
    return MOT_ERR_ALIGN;
  if (ws && ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {x, res, w, mod, y, res_out, ws};
  int dev = -1;
  int st = check_device(s, ptrs, 7, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const size_t row_bytes = size_t(H) * 2;
  int C = int(kNormSlotBudget / (2 * row_bytes));
  C = C > kNormMaxConsumers ? kNormMaxConsumers : C;
  NormArgs a{};
  a.x = x;
  a.res = res;
  a.w = w;
  a.mod = mod;
  a.T = int(T);
  a.H = H;
  a.eps = eps;
  a.y = y;
  a.res_out = res_out;
  // up to kPlanOneCta rows one extra CTA of this launch builds the plan; a larger pack's plan
  // is built first by the many-CTA kernels (one CTA would then outlast a narrow norm)
  const bool embed_plan = ws != nullptr && T <= kPlanOneCta;
  if (ws != nullptr && !embed_plan) {
    st = enqueue_route_plan(mod, int(T), static_cast<uint8_t*>(ws), s);
    if (st != MOT_OK) return st;
  }
  a.err = ws ? &static_cast<PlanHeader*>(ws)->error : nullptr;
  a.plan_ws = embed_plan ? static_cast<uint8_t*>(ws) : nullptr;
  const int sms = sm_count(dev);
  const int avail = embed_plan ? (sms > 1 ? sms - 1 : 1) : sms;  // the plan CTA gets an SM of its own
  a.norm_blocks = int(T < avail ? T : avail);
  a.consumers = C;
  const size_t smem = 2 * row_bytes + size_t(C) * 2 * row_bytes + (2 * kNormMaxConsumers + 2) * sizeof(uint64_t);
  const int grid = a.norm_blocks + (embed_plan ? 1 : 0);
  const int nj = H / 256;
  cudaError_t e;
  if (nj <= 4)
    e = launch_norm<4>(a, grid, smem, s);
  else if (nj <= 8)
    e = launch_norm<8>(a, grid, smem, s);
  else if (nj <= 16)
    e = launch_norm<16>(a, grid, smem, s);
  else
    e = launch_norm<32>(a, grid, smem, s);
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

extern "C" int mot_gather_rows(const mot_bf16* src, int64_t T, int K, void* ws, size_t ws_bytes, mot_bf16* dst,
                               void* stream) {
  if (!src || !ws || !dst) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS || K < 8 || K % 8 != 0 || K > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (!aligned16(src) || !aligned16(ws) || !aligned16(dst)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  if (src == dst) return MOT_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {src, ws, dst};
  int dev = -1;
  int st = check_device(s, ptrs, 3, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  const int grid = 4 * sm_count(dev);
  const cudaError_t e = launch_dependent(gather_rows_kernel, dim3(grid), dim3(256), 0, s,
                                         reinterpret_cast<const uint4*>(src), int(T), K / 8,
                                         static_cast<const uint8_t*>(ws), reinterpret_cast<uint4*>(dst));
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
