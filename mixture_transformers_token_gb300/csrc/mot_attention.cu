// Joint attention of packed sequences on the 5th-generation tensor cores.
//
// Sources: [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435
// (§1 Motivation item 2: latent tokens query the prompt KV non-causally at every step; §2
// Reference hazards: cached prefill needs a bottom-right causal mask; §3 Numerical contract:
// no split-KV, fixed accumulation order; §5 claim order: gen_joint_attention).
//
// A sequence is (q_start, k_start, nq, nk, n_causal): its queries are the last nq of its nk key
// positions; query rows below n_causal (prompt rows) see keys j <= nk - nq + i, the others
// (latent rows) see all nk keys. Query head h reads KV head h / (Hq / Hkv). Q, K and V are read
// in place from the fused QKV output (row stride (Hq + 2 Hkv) D).
//
// Arithmetic, the same for every tile of every pack: S = Q K^T in fp32 on the tensor cores;
// per row, in 128-key blocks in ascending key order: x = S * (scale * log2 e) (masked keys
// -inf), m' = max(m, max_block x), alpha = exp2(m - m'), p = exp2(x - m'), l = l * alpha +
// (sum of the block's p, left to right), O = O * alpha + bf16(p) V (fp32, tensor cores); out =
// bf16(O / l). Blocks start at the sequence's first key, so a row's bits do not depend on the
// other sequences of the pack.
//
// One CTA per (128-row query tile, head); tiles of a sequence are visited last first (the
// causal tiles near the end carry the most keys). Warp 0 loads Q once and K, V blocks into
// two-stage rings (TMA, 128-byte swizzle); warp 1 issues S = Q K^T into one of two TMEM S
// buffers one block ahead, then O += P V (V read as an MN-major operand); warps 2-5 hold one
// query row per thread: they read S from TMEM, form p, rescale O in TMEM when the row maximum
// moves, and write P (bf16, swizzled K-major) to shared memory for the next MMA.

#include <cuda.h>
#include <cuda_runtime.h>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {
namespace attn {

constexpr int BQ = 128, BKV = 128;
constexpr int THREADS = 192;  // producer, MMA, 4 softmax warps
constexpr int KV_STAGES = 2;
constexpr uint32_t SUB = 128 * 64 * 2;  // one [128 rows x 64 columns] bf16 swizzled sub-tile

template <int D>
struct Layout {
  static constexpr uint32_t TILE = BQ * D * 2;  // Q tile, or one K or V block
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = Q + TILE;
  static constexpr uint32_t V = K + KV_STAGES * TILE;
  static constexpr uint32_t P = V + KV_STAGES * TILE;  // [128 rows x 128 keys] bf16
  static constexpr uint32_t BAR = P + BQ * BKV * 2;
  static constexpr size_t BYTES = 1024 + size_t(BAR) + 256;
  static constexpr uint32_t TMEM_S0 = 0, TMEM_S1 = BKV, TMEM_O = 2 * BKV, TMEM_COLS = 512;
};

struct Args {
  const int32_t* seqs;  // [n_seq][5]
  int n_seq;
  int T, Hq, Hkv;
  float c;              // scale * log2(e)
  uint16_t* out;        // [T][Hq D]
  uint32_t* err;
};

__device__ __forceinline__ bool bad_seq(const int32_t* d, int T) {
  const int q0 = d[0], k0 = d[1], nq = d[2], nk = d[3], c = d[4];
  return q0 < 0 || k0 < 0 || nq < 0 || nk < 1 || c < 0 || c > nq || (c > 0 && nk < nq) ||
         int64_t(q0) + nq > T || int64_t(k0) + nk > T;
}

// The tile u of the grid: sequence s, first query row i0 of the tile (tiles of a sequence in
// reverse order). Returns false past the last tile; a bad descriptor contributes no tiles.
__device__ __forceinline__ bool find_tile(const Args& a, int u, int4& sq, int& nc, int& i0) {
  int acc = 0;
  for (int s = 0; s < a.n_seq; ++s) {
    const int32_t* d = a.seqs + 5 * s;
    const int nt = bad_seq(d, a.T) ? 0 : (d[2] + BQ - 1) / BQ;
    if (u < acc + nt) {
      sq = make_int4(d[0], d[1], d[2], d[3]);
      nc = d[4];
      i0 = (nt - 1 - (u - acc)) * BQ;
      return true;
    }
    acc += nt;
  }
  return false;
}

// CTA (0, 0) checks every descriptor, that the query ranges do not overlap (their rows sum to
// at most T) and that the grid covers every tile; a failure sets MOT_DEV_BAD_SEQUENCE.
__device__ void check_sequences(const Args& a) {
  int64_t tiles = 0, rows = 0;
  bool bad = false;
  for (int s = 0; s < a.n_seq; ++s) {
    const int32_t* d = a.seqs + 5 * s;
    if (bad_seq(d, a.T)) {
      bad = true;
      continue;
    }
    tiles += (d[2] + BQ - 1) / BQ;
    rows += d[2];
  }
  if (bad || rows > a.T || tiles > int64_t(gridDim.x)) atomicOr(a.err, MOT_DEV_BAD_SEQUENCE);
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    joint_attention_kernel(const __grid_constant__ CUtensorMap tm_qkv, const Args a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* v_full = bars + 3;   // [2]
  uint64_t* k_empty = bars + 5;  // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2]
  uint64_t* s_free = bars + 11;  // [2]
  uint64_t* p_full = bars + 13;
  uint64_t* o_full = bars + 14;
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) check_sequences(a);
  int4 sq;
  int nc, i0;
  if (!find_tile(a, int(blockIdx.x), sq, nc, i0)) return;  // uniform across the CTA
  const int q0 = sq.x, k0 = sq.y, nq = sq.z, nk = sq.w;
  const int h = int(blockIdx.y), g = h / (a.Hq / a.Hkv);
  const int i1 = i0 + BQ < nq ? i0 + BQ : nq;  // query rows [i0, i1) of the sequence
  const int kmax = i1 > nc ? nk : nk - nq + i1;   // keys the tile needs
  const int nblk = (kmax + BKV - 1) / BKV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&k_full[i]), 1);
      mbar_init(smem_u32(&v_full[i]), 1);
      mbar_init(smem_u32(&k_empty[i]), 1);
      mbar_init(smem_u32(&v_empty[i]), 1);
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_free[i]), 4);
    }
    mbar_init(smem_u32(p_full), 4);
    mbar_init(smem_u32(o_full), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      int kdone = 0, vdone = 0;  // blocks whose K / V copies were issued
      mbar_arrive_expect_tx(smem_u32(q_full), L::TILE);
      for (int b = 0; b < D / 64; ++b)
        tma_load_2d(smem_u32(smem + L::Q + b * SUB), &tm_qkv, h * D + 64 * b, q0 + i0, smem_u32(q_full));
      for (int j = 0; j < nblk && ok; ++j) {
        const int st = j % KV_STAGES;
        const uint32_t ph = uint32_t(j / KV_STAGES) & 1u;
        const int y = k0 + j * BKV;
        ok = mbar_wait(smem_u32(&k_empty[st]), ph ^ 1u, abort_flag, a.err);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&k_full[st]), L::TILE);
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(smem_u32(smem + L::K + st * L::TILE + b * SUB), &tm_qkv, (a.Hq + g) * D + 64 * b, y,
                      smem_u32(&k_full[st]));
        kdone = j + 1;
        ok = mbar_wait(smem_u32(&v_empty[st]), ph ^ 1u, abort_flag, a.err);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&v_full[st]), L::TILE);
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(smem_u32(smem + L::V + st * L::TILE + b * SUB), &tm_qkv, (a.Hq + a.Hkv + g) * D + 64 * b, y,
                      smem_u32(&v_full[st]));
        vdone = j + 1;
      }
      // every issued copy has landed before the CTA can exit
      mbar_drain(smem_u32(q_full), 0);
      for (int j = kdone - KV_STAGES > 0 ? kdone - KV_STAGES : 0; j < kdone; ++j)
        mbar_drain(smem_u32(&k_full[j % KV_STAGES]), uint32_t(j / KV_STAGES) & 1u);
      for (int j = vdone - KV_STAGES > 0 ? vdone - KV_STAGES : 0; j < vdone; ++j)
        mbar_drain(smem_u32(&v_full[j % KV_STAGES]), uint32_t(j / KV_STAGES) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV);
    constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, D) | kIdescBMnMajor;
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(q_full), 0, abort_flag, a.err));
    for (int j = 0; j <= nblk && ok; ++j) {
      if (j < nblk) {
        const int st = j % KV_STAGES, sb = j & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&k_full[st]), uint32_t(j / KV_STAGES) & 1u, abort_flag,
                                               a.err));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_free[sb]), (uint32_t(j >> 1) & 1u) ^ 1u,
                                                       abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t qa = smem_u32(smem + L::Q), kb = smem_u32(smem + L::K + st * L::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16(tmem + (sb ? L::TMEM_S1 : L::TMEM_S0), smem_desc_sw128(qa + (kk / 4) * SUB + (kk % 4) * 32),
                     smem_desc_sw128(kb + (kk / 4) * SUB + (kk % 4) * 32), idesc_s, kk > 0);
          mma_commit(smem_u32(&s_full[sb]));
          mma_commit(smem_u32(&k_empty[st]));
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jj = j - 1, st = jj % KV_STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(p_full), uint32_t(jj) & 1u, abort_flag, a.err));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&v_full[st]), uint32_t(jj / KV_STAGES) & 1u,
                                                       abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t pa = smem_u32(smem + L::P), vb = smem_u32(smem + L::V + st * L::TILE);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            mma_bf16(tmem + L::TMEM_O, smem_desc_sw128(pa + (kk / 4) * SUB + (kk % 4) * 32),
                     smem_desc_mn_sw128(vb + kk * 2048, SUB), idesc_o, (jj | kk) != 0);
          mma_commit(smem_u32(o_full));
          mma_commit(smem_u32(&v_empty[st]));
        }
        __syncwarp();
      }
    }
    // every MMA issued has completed before tensor memory is released
    if (lane == 0) mma_commit(smem_u32(drain));
    __syncwarp();
    mbar_drain(smem_u32(drain), 0);
  } else {
    // ---------------- softmax: one query row per thread ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int i = i0 + row;                                   // query row within the sequence
    const bool valid = i < nq;
    const int lim = (valid && i < nc) ? nk - nq + i + 1 : nk;  // keys [0, lim) are visible
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    uint8_t* prow = smem + L::P + row * 128;  // row `row` of each 64-key sub-tile
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[sb]), uint32_t(j >> 1) & 1u, abort_flag, a.err));
      if (!ok) break;
      tc_fence_after();
      float x[BKV];
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_off + (sb ? L::TMEM_S1 : L::TMEM_S0) + c * 32, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) x[c * 32 + t] = v[t];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_free[sb]));
      // scale into the log2 domain, mask, block maximum
      float bmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < BKV; ++c) {
        const float xs = j * BKV + c < lim ? __fmul_rn(x[c], a.c) : -INFINITY;
        x[c] = xs;
        bmax = fmaxf(bmax, xs);
      }
      const float m_new = fmaxf(m, bmax);
      const float alpha = exp2f(__fsub_rn(m, m_new));  // 0 on the first block (m = -inf)
      float psum = 0.0f;
#pragma unroll
      for (int c = 0; c < BKV; ++c) {
        const float p = exp2f(__fsub_rn(x[c], m_new));
        x[c] = p;
        psum = __fadd_rn(psum, p);
      }
      l = __fadd_rn(__fmul_rn(l, alpha), psum);
      m = m_new;
      if (j >= 1) {
        // the previous block's P V is done: the P buffer is free and O may be rescaled
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(o_full), uint32_t(j - 1) & 1u, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_off + L::TMEM_O + c * 32, o);
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __fmul_rn(o[t], alpha);
            tmem_st32(tmem + lane_off + L::TMEM_O + c * 32, o);
          }
        }
      }
      // P as bf16 into the swizzled K-major tile: keys 8 cc .. 8 cc + 7 of sub-tile b go to
      // the 16-byte chunk cc ^ (row & 7) of the row
#pragma unroll
      for (int cch = 0; cch < BKV / 8; ++cch) {
        const int b = cch >> 3, cc = cch & 7;
        const uint4 v = make_uint4(pack_bf2(x[8 * cch], x[8 * cch + 1]), pack_bf2(x[8 * cch + 2], x[8 * cch + 3]),
                                   pack_bf2(x[8 * cch + 4], x[8 * cch + 5]), pack_bf2(x[8 * cch + 6], x[8 * cch + 7]));
        *reinterpret_cast<uint4*>(prow + b * SUB + ((cc ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full));
    }
    if (ok && nblk > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(o_full), uint32_t(nblk - 1) & 1u, abort_flag, a.err));
      if (ok) {
        tc_fence_after();
        uint16_t* orow = a.out + int64_t(q0 + i) * (int64_t(a.Hq) * D) + int64_t(h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_off + L::TMEM_O + c * 32, o);
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) pk[t] = pack_bf2(__fdiv_rn(o[2 * t], l), __fdiv_rn(o[2 * t + 1], l));
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int t = 0; t < 4; ++t) dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// Both head dims launch with the D = 128 shared-memory size: one CTA per SM, so two CTAs never
// compete for the 512 tensor-memory columns each allocates.
constexpr size_t kSmemBytes = Layout<128>::BYTES;

template <int D>
static int launch(const mot_bf16* qkv, const Args& a, int n_tiles_max, cudaStream_t s) {
  CUtensorMap tm;
  const uint64_t ncol = uint64_t(a.Hq + 2 * a.Hkv) * D;
  if (!make_tmap_bf16(&tm, qkv, ncol, uint64_t(a.T), 64, BQ)) return MOT_ERR_CUDA;
  if (cudaFuncSetAttribute(joint_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemBytes)) != cudaSuccess)
    return MOT_ERR_CUDA;
  joint_attention_kernel<D><<<dim3(unsigned(n_tiles_max), unsigned(a.Hq)), THREADS, kSmemBytes, s>>>(tm, a);
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

}  // namespace attn
}  // namespace mot

using namespace mot;

extern "C" int mot_joint_attention(const mot_bf16* qkv, int64_t T, int Hq, int Hkv, int D, const int32_t* seqs,
                                   int n_seq, float scale, void* ws, size_t ws_bytes, mot_bf16* out, void* stream) {
  if (!qkv || !seqs || !ws || !out) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (D != 64 && D != 128) return MOT_ERR_GEOMETRY;
  if (Hq < 1 || Hkv < 1 || Hq > 1024 || Hkv > 1024 || Hq % Hkv != 0) return MOT_ERR_GEOMETRY;
  if (n_seq < 1 || n_seq > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (!(scale > 0.0f) || !(scale < 3.0e38f)) return MOT_ERR_ARG;
  if (!aligned16(qkv) || !aligned16(seqs) || !aligned16(ws) || !aligned16(out)) return MOT_ERR_ALIGN;
  if (ws_bytes < sizeof(PlanHeader)) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {qkv, seqs, ws, out};
  int dev = -1;
  int st = check_device(s, ptrs, 4, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  attn::Args a{};
  a.seqs = seqs;
  a.n_seq = n_seq;
  a.T = int(T);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.c = scale * 1.4426950408889634f;
  a.out = out;
  a.err = &static_cast<PlanHeader*>(ws)->error;
  // every sequence has at most nq / 128 + 1 tiles and the query ranges do not overlap (checked
  // on the device), so T / 128 + n_seq bounds the tile count
  const int64_t tiles = (T + attn::BQ - 1) / attn::BQ + n_seq;
  if (tiles > (int64_t(1) << 30)) return MOT_ERR_GEOMETRY;
  if (D == 64) return attn::launch<64>(qkv, a, int(tiles), s);
  return attn::launch<128>(qkv, a, int(tiles), s);
}
