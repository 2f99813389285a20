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
// per row, in 128-key blocks in ascending key order, with c = scale * log2 e: the running
// maximum m of S (masked keys excluded) moves to the block maximum only when that exceeds it
// by more than 8 / c (then O and l are scaled by 2^((m_old - m) c)); p = 2^((S - m) c) (the
// difference and then the product each rounded to fp32, then CUDA's accurate exp2f -- no fused
// multiply-add, no approximate or flush-to-zero instruction, as the numerical contract
// requires; a subtraction that feeds a product cannot be fused into one, so the pair runs as
// packed f32x2 instructions, which a product feeding a packed addition did not survive);
// l += the block's p (four interleaved partial sums);
// O += bf16(p) V (fp32, tensor cores); out = bf16(O * (1 / l)), 1 / l rounded to fp32 once
// per row. Blocks start at the sequence's first
// key, so a row's bits do not depend on the other sequences of the pack.
//
// One CTA per (pair of 128-row query tiles, head); pairs of a sequence are visited last first
// (the causal tiles near the end carry the most keys). Warp 0 loads both Q tiles once, each
// 128-key K block into one buffer and each V block into a two-stage ring (TMA, 128-byte
// swizzle); warp 1 issues, per key block, S = Q K^T for both tiles (M128 N128: every tcgen05
// instruction costs at least about 107 cycles, so 128 keys per instruction keep it at 60 % of
// the tensor rate where 64 keys reached 30 %), then O += P V of the previous block for both
// (P and V from shared memory, V as an MN-major operand); warps 2-5 and 6-9 are the softmax
// warpgroups of the two tiles, one query row per thread: they read a block's 128 scores from
// TMEM, form p, rescale O in TMEM when the row maximum moves, and write P (bf16, swizzled
// K-major) into the tile's shared-memory P tile once the previous P V has read it. Each tile's
// softmax runs while the tensor cores work on the other tile. Warp 0 first finds the CTA's work
// item, reading the sequence descriptors one per lane. A whole output tile goes, as bf16, to the
// tile's Q buffer (idle after its last S MMA) and out by TMA tensor stores; a ragged tile is
// written row by row so that rows of other sequences are never touched.

#include <cuda.h>
#include <cuda_runtime.h>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {
namespace attn {

constexpr int BQ = 128, BKV = 128;
constexpr int TILES = 2;        // query tiles per CTA (ping-pong between two softmax warpgroups)
constexpr int THREADS = 320;    // producer, MMA, 2 x 4 softmax warps
constexpr int K_STAGES = 1, V_STAGES = 2;
constexpr uint32_t SUB = 128 * 64 * 2;   // a [128 rows x 64 columns] bf16 swizzled tile (Q, P half)
constexpr uint32_t KSUB = BKV * 64 * 2;  // a [128 keys x 64 columns] bf16 swizzled tile (K, V half)

template <int D>
struct Layout {
  static constexpr uint32_t QTILE = BQ * D * 2;    // a Q tile
  static constexpr uint32_t KVBLK = BKV * D * 2;   // one K or V block
  static constexpr uint32_t PTILE = BQ * BKV * 2;  // a tile's P: [128 rows x 128 keys] bf16, two halves
  static constexpr uint32_t Q = 0;                          // TILES Q tiles
  static constexpr uint32_t K = Q + TILES * QTILE;          // K_STAGES K blocks
  static constexpr uint32_t V = K + K_STAGES * KVBLK;       // V_STAGES V blocks
  static constexpr uint32_t P = V + V_STAGES * KVBLK;       // TILES P tiles
  static constexpr uint32_t BAR = P + TILES * PTILE;
  static constexpr size_t BYTES = 1024 + size_t(BAR) + 512;  // barriers, tensor-memory slot, work item
  // tensor memory: S of tile t at 128 t (128 keys), O of tile t at 256 + 128 t
  static constexpr uint32_t TMEM_S = 0, TMEM_O = 256, TMEM_COLS = 512;
};

struct Args {
  const int32_t* seqs;  // [n_seq][5]
  int n_seq;
  int T, Hq, Hkv;
  float c;              // scale * log2(e)
  uint16_t* out;        // [T][Hq D]
  uint32_t* err;
};

// 2^x: CUDA's exp2f (the library's accurate function, with subnormal results; this code is
// built without fast-math options).
__device__ __forceinline__ float ex2(float x) { return exp2f(x); }

// Packed pairs of fp32 (Blackwell f32x2 arithmetic: two IEEE operations per instruction, each
// rounded as the scalar one would be).
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The running maximum moves only when a block's maximum exceeds it by more than this many
// powers of two: until then p = 2^((S - m) c) stays below 2^8, and O and l, which share m,
// need no rescaling.
constexpr float kLazyLog2 = 8.0f;

__device__ __forceinline__ bool bad_seq(const int32_t* d, int T) {
  const int q0 = d[0], k0 = d[1], nq = d[2], nk = d[3], c = d[4];
  return q0 < 0 || k0 < 0 || nq < 0 || nk < 1 || c < 0 || c > nq || (c > 0 && nk < nq) ||
         int64_t(q0) + nq > T || int64_t(k0) + nk > T;
}

// The work items of a sequence are its 256-row pairs of query tiles; item r counts from the
// end (r = 0 is the last pair, which sees the most keys). The grid visits items heaviest
// first with the heads fastest: all heads of item 0 of every sequence, then item 1 of every
// sequence, ... (for up to 64 sequences; beyond that, sequence by sequence), so the in-order
// block dispatch balances the uneven causal work. CTA u takes head u % Hq of item u / Hq.
// Returns false past the last item; a bad descriptor contributes none.
constexpr int kSortedSeqs = 64;

__device__ __forceinline__ int seq_items(const Args& a, int s) {
  const int32_t* d = a.seqs + 5 * s;
  return bad_seq(d, a.T) ? 0 : (d[2] + TILES * BQ - 1) / (TILES * BQ);
}

// Finds the item of CTA index k; called by a whole warp, every lane returns the same answer.
// The lanes fetch the descriptors in parallel (one sequence per lane and round of 32), so the
// lookup costs a few memory round trips, not one per sequence.
__device__ bool find_tile(const Args& a, int k, int lane, int4& sq, int& nc, int& i0) {
  int found_s = -1, r = -1;
  if (a.n_seq <= kSortedSeqs) {
    // items of sequences lane and lane + 32; round rr takes every sequence with more than rr
    // items, in sequence order
    const int it0 = lane < a.n_seq ? seq_items(a, lane) : 0;
    const int it1 = lane + 32 < a.n_seq ? seq_items(a, lane + 32) : 0;
    int most = it0 > it1 ? it0 : it1;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const int o = __shfl_xor_sync(0xffffffffu, most, off);
      most = o > most ? o : most;
    }
    int acc = 0;
    for (int rr = 0; rr < most; ++rr) {
      const uint32_t m0 = __ballot_sync(0xffffffffu, it0 > rr), m1 = __ballot_sync(0xffffffffu, it1 > rr);
      const int c0 = __popc(m0), c1 = __popc(m1);
      if (k < acc + c0 + c1) {
        const int t = k - acc;  // the t-th sequence (from 0) taking part in this round
        found_s = t < c0 ? int(__fns(m0, 0, t + 1)) : 32 + int(__fns(m1, 0, t - c0 + 1));
        r = rr;
        break;
      }
      acc += c0 + c1;
    }
    if (found_s < 0) return false;
  } else {
    // sequence by sequence: a warp-wide running count over rounds of 32 sequences
    int acc = 0;
    for (int s0 = 0; s0 < a.n_seq && found_s < 0; s0 += 32) {
      const int s = s0 + lane;
      const int nt = s < a.n_seq ? seq_items(a, s) : 0;
      int incl = nt;  // inclusive prefix sum over the lanes
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const uint32_t hit = __ballot_sync(0xffffffffu, k < acc + incl && k >= acc + incl - nt);
      if (hit != 0u) {
        const int l = __ffs(hit) - 1;
        found_s = s0 + l;
        r = k - acc - (__shfl_sync(0xffffffffu, incl, l) - __shfl_sync(0xffffffffu, nt, l));
      }
      acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (found_s < 0) return false;
  }
  const int32_t* d = a.seqs + 5 * found_s;
  sq = make_int4(d[0], d[1], d[2], d[3]);
  nc = d[4];
  i0 = (seq_items(a, found_s) - 1 - r) * (TILES * BQ);
  return true;
}

// CTA 0 checks every descriptor, that the query ranges do not overlap (their rows sum to
// at most T) and that the grid covers every tile; a failure sets MOT_DEV_BAD_SEQUENCE. Called
// by a whole warp, one sequence per lane and round.
__device__ void check_sequences(const Args& a, int lane) {
  int64_t tiles = 0, rows = 0;
  bool bad = false;
  for (int s = lane; s < a.n_seq; s += 32) {
    const int32_t* d = a.seqs + 5 * s;
    if (bad_seq(d, a.T)) {
      bad = true;
      continue;
    }
    tiles += (d[2] + TILES * BQ - 1) / (TILES * BQ);
    rows += d[2];
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    tiles += __shfl_xor_sync(0xffffffffu, tiles, off);
    rows += __shfl_xor_sync(0xffffffffu, rows, off);
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0 && (bad || rows > a.T || tiles * a.Hq > int64_t(gridDim.x))) atomicOr(a.err, MOT_DEV_BAD_SEQUENCE);
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    joint_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                           const __grid_constant__ CUtensorMap tm_out, const Args a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR);
  uint64_t* q_full = bars;        // both Q tiles
  uint64_t* k_full = bars + 1;    // [K_STAGES]
  uint64_t* k_empty = bars + 4;   // [K_STAGES]: both tiles' S MMAs have read the block
  uint64_t* v_full = bars + 7;    // [V_STAGES]
  uint64_t* v_empty = bars + 10;  // [V_STAGES]: both tiles' P V MMAs have read the block
  uint64_t* s_full = bars + 13;   // [TILES]
  uint64_t* s_free = bars + 17;   // [TILES]: the tile's softmax warps have read S
  uint64_t* p_full = bars + 21;   // [TILES]
  uint64_t* o_full = bars + 23;   // [TILES]: the tile's P V of the block is done (and every earlier one)
  uint64_t* drain = bars + 27;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 28);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  // warp 0 finds the CTA's work item; the others read it from shared memory
  int* item = reinterpret_cast<int*>(tmem_slot + 2);  // found, q0, k0, nq, nk, n_causal, i0
  if (threadIdx.x < 32) {
    if (blockIdx.x == 0) check_sequences(a, int(threadIdx.x));
    int4 sq4 = make_int4(0, 0, 0, 0);
    int c4 = 0, i04 = 0;
    const bool found = find_tile(a, int(blockIdx.x) / a.Hq, int(threadIdx.x), sq4, c4, i04);
    if (threadIdx.x == 0) {
      item[0] = found ? 1 : 0;
      item[1] = sq4.x;
      item[2] = sq4.y;
      item[3] = sq4.z;
      item[4] = sq4.w;
      item[5] = c4;
      item[6] = i04;
    }
  }
  __syncthreads();
  if (!item[0]) return;  // uniform across the CTA
  const int q0 = item[1], k0 = item[2], nq = item[3], nk = item[4], nc = item[5], i0 = item[6];
  const int h = int(blockIdx.x) % a.Hq, g = h / (a.Hq / a.Hkv);
  const int i1 = i0 + TILES * BQ < nq ? i0 + TILES * BQ : nq;  // query rows [i0, i1) of the sequence
  const int kmax = i1 > nc ? nk : nk - nq + i1;                 // keys the pair needs
  const int nblk = (kmax + BKV - 1) / BKV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int i = 0; i < K_STAGES; ++i) {
      mbar_init(smem_u32(&k_full[i]), 1);
      mbar_init(smem_u32(&k_empty[i]), 1);
    }
    for (int i = 0; i < V_STAGES; ++i) {
      mbar_init(smem_u32(&v_full[i]), 1);
      mbar_init(smem_u32(&v_empty[i]), 1);
    }
    for (int t = 0; t < TILES; ++t) {
      mbar_init(smem_u32(&s_full[t]), 1);
      mbar_init(smem_u32(&s_free[t]), 4);
      mbar_init(smem_u32(&p_full[t]), 4);
      mbar_init(smem_u32(&o_full[t]), 1);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_out);
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
      mbar_arrive_expect_tx(smem_u32(q_full), TILES * L::QTILE);
      for (int t = 0; t < TILES; ++t)
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(smem_u32(smem + L::Q + t * L::QTILE + b * SUB), &tm_q, h * D + 64 * b, q0 + i0 + t * BQ,
                      smem_u32(q_full));
      for (int j = 0; j < nblk && ok; ++j) {
        const int ks = j % K_STAGES, vs = j % V_STAGES;
        const int y = k0 + j * BKV;
        ok = mbar_wait(smem_u32(&k_empty[ks]), (uint32_t(j / K_STAGES) & 1u) ^ 1u, abort_flag, a.err);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&k_full[ks]), L::KVBLK);
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(smem_u32(smem + L::K + ks * L::KVBLK + b * KSUB), &tm_kv, (a.Hq + g) * D + 64 * b, y,
                      smem_u32(&k_full[ks]));
        kdone = j + 1;
        ok = mbar_wait(smem_u32(&v_empty[vs]), (uint32_t(j / V_STAGES) & 1u) ^ 1u, abort_flag, a.err);
        if (!ok) break;
        mbar_arrive_expect_tx(smem_u32(&v_full[vs]), L::KVBLK);
        for (int b = 0; b < D / 64; ++b)
          tma_load_2d(smem_u32(smem + L::V + vs * L::KVBLK + b * KSUB), &tm_kv, (a.Hq + a.Hkv + g) * D + 64 * b, y,
                      smem_u32(&v_full[vs]));
        vdone = j + 1;
      }
      // every issued copy has landed before the CTA can exit
      mbar_drain(smem_u32(q_full), 0);
      for (int j = kdone - K_STAGES > 0 ? kdone - K_STAGES : 0; j < kdone; ++j)
        mbar_drain(smem_u32(&k_full[j % K_STAGES]), uint32_t(j / K_STAGES) & 1u);
      for (int j = vdone - V_STAGES > 0 ? vdone - V_STAGES : 0; j < vdone; ++j)
        mbar_drain(smem_u32(&v_full[j % V_STAGES]), uint32_t(j / V_STAGES) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // per block j: S of both tiles (M128 N128: 128 keys per instruction), then P V of block
    // j - 1 for both (P from shared memory, V MN-major)
    constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV);
    constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, D) | kIdescBMnMajor;
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(q_full), 0, abort_flag, a.err));
    for (int j = 0; j <= nblk && ok; ++j) {
      if (j < nblk) {
        const int ks = j % K_STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&k_full[ks]), uint32_t(j / K_STAGES) & 1u, abort_flag,
                                               a.err));
        for (int t = 0; t < TILES && ok; ++t) {
          if (j >= 1) {  // the softmax warps have read S of block j - 1
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_free[t]), uint32_t(j - 1) & 1u, abort_flag, a.err));
            if (!ok) break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t qa = smem_u32(smem + L::Q + t * L::QTILE), kb = smem_u32(smem + L::K + ks * L::KVBLK);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_bf16(tmem + L::TMEM_S + t * BKV, smem_desc_sw128(qa + (kk / 4) * SUB + (kk % 4) * 32),
                       smem_desc_sw128(kb + (kk / 4) * KSUB + (kk % 4) * 32), idesc_s, kk > 0);
            mma_commit(smem_u32(&s_full[t]));
            if (t == TILES - 1) mma_commit(smem_u32(&k_empty[ks]));
          }
          __syncwarp();
        }
        if (!ok) break;
      }
      if (j >= 1) {
        const int jj = j - 1, vs = jj % V_STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&v_full[vs]), uint32_t(jj / V_STAGES) & 1u, abort_flag,
                                               a.err));
        for (int t = 0; t < TILES && ok; ++t) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_full[t]), uint32_t(jj) & 1u, abort_flag, a.err));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t pa = smem_u32(smem + L::P + t * L::PTILE);
            const uint32_t vb = smem_u32(smem + L::V + vs * L::KVBLK);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
              mma_bf16(tmem + L::TMEM_O + t * 128, smem_desc_sw128(pa + (kk / 4) * SUB + (kk % 4) * 32),
                       smem_desc_mn_sw128(vb + kk * 2048, KSUB), idesc_o, (jj | kk) != 0);
            mma_commit(smem_u32(&o_full[t]));
            if (t == TILES - 1) mma_commit(smem_u32(&v_empty[vs]));
          }
          __syncwarp();
        }
      }
    }
    // every MMA issued has completed before tensor memory is released
    if (lane == 0) mma_commit(smem_u32(drain));
    __syncwarp();
    mbar_drain(smem_u32(drain), 0);
  } else {
    // ---------------- softmax: warpgroup t = (warp - 2) / 4, one query row per thread ----------------
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int i = i0 + t * BQ + row;                             // query row within the sequence
    const bool valid = i < nq;
    const int lim = (valid && i < nc) ? nk - nq + i + 1 : nk;   // keys [0, lim) are visible
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t to = tmem + lane_off + L::TMEM_O + t * 128;
    uint8_t* prow = smem + L::P + t * L::PTILE + row * 128;  // the row in the tile's P (half 0)
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[t]), uint32_t(j) & 1u, abort_flag, a.err));
      if (!ok) break;
      tc_fence_after();
      float x[BKV];
      {
        float (&x0)[64] = *reinterpret_cast<float (*)[64]>(&x[0]);
        float (&x1)[64] = *reinterpret_cast<float (*)[64]>(&x[64]);
        tmem_ld64(tmem + lane_off + L::TMEM_S + t * BKV, x0);
        tmem_ld64(tmem + lane_off + L::TMEM_S + t * BKV + 64, x1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_free[t]));  // S may be overwritten by the next block
      if (__any_sync(0xffffffffu, j * BKV + BKV > lim)) {  // the block reaches past a row's keys
        const int lim_b = lim - j * BKV;
#pragma unroll
        for (int c = 0; c < BKV; ++c) x[c] = c < lim_b ? x[c] : -INFINITY;
      }
      // block maximum of the raw scores, four interleaved chains
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < BKV; ++c) mx[c & 3] = fmaxf(mx[c & 3], x[c]);
      const float bmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      float alpha = 1.0f;
      if (m == -INFINITY) {
        m = bmax;  // the first block with a visible key (block 0 for every valid row)
      } else if (__fmul_rn(__fsub_rn(bmax, m), a.c) > kLazyLog2) {
        alpha = ex2(__fmul_rn(__fsub_rn(m, bmax), a.c));
        m = bmax;
      }
      const float nm = m == -INFINITY ? 0.0f : -m;  // no visible key yet: every score is -inf
      // the tile's single P buffer and O are free once the P V of block j - 1 is done
      if (j >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&o_full[t]), uint32_t(j - 1) & 1u, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
      }
      // p = 2^(fp32(fp32(S - m) c)), four interleaved partial sums (key c adds to sum c mod 4), as f32x2
      // pairs; every 8 keys go as bf16 to the 16-byte chunk (cc ^ (row & 7)) of the row in half
      // cc / 8 of the swizzled P tile
      const unsigned long long c2 = f2_pack(a.c, a.c), nm2 = f2_pack(nm, nm);
      unsigned long long ps01 = 0ull, ps23 = 0ull;  // (sum 0, sum 1), (sum 2, sum 3), from +0
#pragma unroll
      for (int cc = 0; cc < BKV / 8; ++cc) {
        uint32_t pk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = 8 * cc + 2 * u;
          float t0, t1;
          f2_unpack(f2_mul(f2_add(f2_pack(x[c], x[c + 1]), nm2), c2), t0, t1);
          const float p0 = ex2(t0), p1 = ex2(t1);
          const unsigned long long p01 = f2_pack(p0, p1);
          if (u & 1) ps23 = f2_add(ps23, p01);
          else ps01 = f2_add(ps01, p01);
          pk[u] = pack_bf2(p0, p1);
        }
        *reinterpret_cast<uint4*>(prow + (cc >> 3) * SUB + (((cc & 7) ^ (row & 7)) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      float ps[4];
      f2_unpack(ps01, ps[0], ps[1]);
      f2_unpack(ps23, ps[2], ps[3]);
      const float psum = __fadd_rn(__fadd_rn(ps[0], ps[1]), __fadd_rn(ps[2], ps[3]));
      l = __fadd_rn(__fmul_rn(l, alpha), psum);
      // O takes the new maximum before the P V of block j adds to it
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(to + c * 32, o);
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __fmul_rn(o[u], alpha);
          tmem_st32(to + c * 32, o);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[t]));
    }
    if (nblk > 0) {
      // the last P V (and with it every earlier one) is done
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&o_full[t]), uint32_t(nblk - 1) & 1u, abort_flag, a.err));
      const float rl = __frcp_rn(l);  // one rounded reciprocal per row, then products
      if (i0 + t * BQ + BQ <= nq) {
        // every row of the tile is a query: the bf16 tile goes to the tile's Q buffer (no MMA
        // reads it any more) in the 128-byte swizzled box layout, then out by tensor stores.
        // Every warp of the tile reaches the barrier, the stores go only if no wait gave up.
        if (ok) {
          tc_fence_after();
          uint8_t* qrow = smem + L::Q + t * L::QTILE + row * 128;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(to + c * 32, o);
            uint32_t ok16[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) ok16[u] = pack_bf2(__fmul_rn(o[2 * u], rl), __fmul_rn(o[2 * u + 1], rl));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = 4 * c + u;  // 16-byte piece of the row: box k / 8, chunk k % 8
              *reinterpret_cast<uint4*>(qrow + (k >> 3) * SUB + (((k & 7) ^ (row & 7)) << 4)) =
                  make_uint4(ok16[4 * u], ok16[4 * u + 1], ok16[4 * u + 2], ok16[4 * u + 3]);
            }
          }
          fence_proxy_async_smem();
        }
        named_bar_sync(1 + t, 4 * 32);
        if (warp == 2 + 4 * t && lane == 0 && *abort_flag == 0u) {
          for (int b = 0; b < D / 64; ++b)
            tma_store_2d(&tm_out, smem_u32(smem + L::Q + t * L::QTILE + b * SUB), h * D + 64 * b, q0 + i0 + t * BQ);
          bulk_store_commit_and_wait_read();
        }
      } else if (ok) {
        // a ragged tile (rows past the sequence's queries belong to others): row by row
        tc_fence_after();
        uint16_t* orow = a.out + int64_t(q0 + i) * (int64_t(a.Hq) * D) + int64_t(h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(to + c * 32, o);
          if (valid) {
            uint32_t ok16[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) ok16[u] = pack_bf2(__fmul_rn(o[2 * u], rl), __fmul_rn(o[2 * u + 1], rl));
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[u] = make_uint4(ok16[4 * u], ok16[4 * u + 1], ok16[4 * u + 2], ok16[4 * u + 3]);
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
  CUtensorMap tm_q, tm_kv, tm_out;
  const uint64_t ncol = uint64_t(a.Hq + 2 * a.Hkv) * D;
  if (!make_tmap_bf16(&tm_q, qkv, ncol, uint64_t(a.T), 64, BQ) ||
      !make_tmap_bf16(&tm_kv, qkv, ncol, uint64_t(a.T), 64, BKV) ||
      !make_tmap_bf16(&tm_out, a.out, uint64_t(a.Hq) * D, uint64_t(a.T), 64, BQ))
    return MOT_ERR_CUDA;
  if (cudaFuncSetAttribute(joint_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kSmemBytes)) != cudaSuccess)
    return MOT_ERR_CUDA;
  joint_attention_kernel<D><<<unsigned(int64_t(n_tiles_max) * a.Hq), THREADS, kSmemBytes, s>>>(tm_q, tm_kv, tm_out, a);
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
  // every sequence has at most nq / 256 + 1 work items (pairs of 128-row tiles) and the query
  // ranges do not overlap (checked on the device), so T / 256 + n_seq bounds their count
  const int64_t tiles = (T + attn::TILES * attn::BQ - 1) / (attn::TILES * attn::BQ) + n_seq;
  if (tiles * Hq > (int64_t(1) << 31) - 1) return MOT_ERR_GEOMETRY;
  if (D == 64) return attn::launch<64>(qkv, a, int(tiles), s);
  return attn::launch<128>(qkv, a, int(tiles), s);
}
