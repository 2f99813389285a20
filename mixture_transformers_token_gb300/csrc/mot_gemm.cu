// Routed dense GEMM on the 5th-generation tensor cores, with three fused epilogues:
//   cast          out = bf16(acc)                                  (O and down projections)
//   SwiGLU        out = bf16(silu(bf16(acc_gate)) * bf16(acc_up))  (gate/up projection)
//   QK-norm+RoPE  per-head fp32 RMSNorm, then BF16 RoPE           (fused QKV projection)
//                 or, in the FP32 RoPE profile, RoPE in fp32 on the fp32 normalized head
//                 with one bf16 cast (open question 4 of the roadmap below)
//
// Sources: [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435
// (§1 item 1: per-token weight sets; §2 Reference hazards: QK norm in FP32, then RoPE and Q/K
// in BF16; §3 Numerical contract: fixed accumulation order, no split-K / stream-K / atomics,
// casts only at declared boundaries); feat: support Bagel in SeedOmni - #1402 ("What does this
// PR do?": routed Q/K/V and O projections, fused qkv_proj_{und,gen}, per-head QK RMSNorm,
// packed RoPE); [WS1][CUDA][Qwen3-Next] MoE route/combine contract ... #503 (grouped expert
// GEMM commit: one writer per row, grouped result equal to the per-expert GEMM; SwiGLU in
// FP32 with one BF16 cast; gated-norm commit: accurate expf).
//
// Design (persistent, one CTA per SM, CTA pairs in clusters of two):
//   A pair of CTAs computes a 256 x 256 output tile with the 2-SM MMA: each CTA holds its own
//   128-row tile of A (one 128-row tile of the routing plan; both tiles of the same expert) and
//   half of the 256 weight rows, so a pipeline stage is 32 KB per CTA and six stages fit.
//   warp 0      TMA producer of each CTA: its A tile (one tiled load when the tile's rows are
//               consecutive, else 32 four-row gathers, one per lane) and its B half, signalled
//               on the leader CTA's stage barrier.
//   warp 1      allocates 512 TMEM columns in both CTAs (two 128 x 256 fp32 accumulators per
//               CTA); in the leader CTA one thread issues tcgen05.mma.cta_group::2 (M 256,
//               N 256, K 16), K blocks in ascending order, and multicasts its commits to both
//               CTAs.
//   warps 2-9   epilogue of each CTA: two warps per TMEM lane quarter, one per 128-column half;
//               one thread per accumulator row (its TMEM lane), read with tcgen05.ld, written
//               to the row's original position (or its plan position).
// Every tile of every pack uses the same tile shape, K order and instruction sequence, so a
// row's bits depend only on the row and its expert's weights.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "mot.h"
#include "mot_device.cuh"
#include "mot_host.hpp"

namespace mot {
namespace gemm {

constexpr int BM = 128;       // A rows per CTA (the pair covers 256)
constexpr int BN = 256;       // output columns per pair tile
constexpr int BN_HALF = 128;  // weight rows held by each CTA of the pair
constexpr int BK = 64, STAGES = 6;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN_HALF * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 320;  // producer, MMA, 8 epilogue warps
constexpr int EPI_WARPS = 8;
constexpr uint32_t ACC_COLS = BN;
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + 256 + 2048;  // + QK-norm weights (fp32)

enum Epi { EPI_CAST = 0, EPI_SWIGLU = 1, EPI_QKV64 = 2, EPI_QKV128 = 3, EPI_QKV64_F32 = 4, EPI_QKV128_F32 = 5 };

__host__ __device__ constexpr bool is_qkv(int epi) { return epi >= EPI_QKV64; }
__host__ __device__ constexpr bool rope_f32(int epi) { return epi == EPI_QKV64_F32 || epi == EPI_QKV128_F32; }
__host__ __device__ constexpr int head_dim(int epi) { return epi == EPI_QKV64 || epi == EPI_QKV64_F32 ? 64 : 128; }

struct Args {
  const uint8_t* ws;  // routing plan
  uint32_t* err;      // plan error word
  int T, N, K;        // N weight rows per expert, K reduction length
  int n_tiles;        // N / BN
  uint16_t* out;
  int ldo;
  const uint16_t* bias;  // [2][N] or null (QKV only)
  const uint16_t* qn;    // [2][D]
  const uint16_t* kn;    // [2][D]
  const int32_t* pos;    // [T]
  const uint16_t* cs;    // [P][D/2][2] bf16 (BF16 RoPE profile)
  const float* cs32;     // [P][D/2][2] fp32 (FP32 RoPE profile)
  int P;
  int Hq, Hkv;
  float eps;
  int a_plan_order;      // rows of A are in plan order
  int out_plan_order;    // rows of out are written in plan order
  int st32;              // out and its row pitch are 32-byte aligned: 32-byte stores (set at launch)
};

// n_u4 (even) 16-byte pieces of a row: one lane writes whole 32-byte sectors when the output
// allows 32-byte stores, else 16-byte ones.
__device__ __forceinline__ void store_row_u4(const Args& a, uint16_t* dst, const uint32_t* pk, int n_u4) {
  if (a.st32) {
#pragma unroll
    for (int i = 0; i < n_u4; i += 2)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * i), "r"(pk[4 * i]),
                   "r"(pk[4 * i + 1]), "r"(pk[4 * i + 2]), "r"(pk[4 * i + 3]), "r"(pk[4 * i + 4]), "r"(pk[4 * i + 5]),
                   "r"(pk[4 * i + 6]), "r"(pk[4 * i + 7])
                   : "memory");
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < n_u4; ++i) d[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
}

// Epilogue warps: two per TMEM lane quarter; warp "half" h handles the tile's columns
// [128 h, 128 h + 128) of its 32 rows.

// out = bf16(acc): 128 columns
__device__ __forceinline__ void epi_cast(const Args& a, uint32_t taddr, bool valid, int grow, int nt, int half) {
  uint16_t* orow = a.out + int64_t(grow) * a.ldo + int64_t(nt) * BN + half * 128;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    tmem_ld32(taddr + half * 128 + c * 32, v);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf2(v[2 * i], v[2 * i + 1]);
    if (valid) store_row_u4(a, orow + c * 32, pk, 4);
  }
}

// gate columns 0..127 and up columns 128..255 of the tile -> 128 outputs; half h makes outputs
// [64 h, 64 h + 64) from gate columns 64 h + i and up columns 128 + 64 h + i
__device__ __forceinline__ void epi_swiglu(const Args& a, uint32_t taddr, bool valid, int grow, int nt, int half) {
  uint16_t* orow = a.out + int64_t(grow) * a.ldo + int64_t(nt) * (BN / 2) + half * 64;
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    float g[32], u[32];
    tmem_ld32(taddr + half * 64 + c * 32, g);
    tmem_ld32(taddr + 128 + half * 64 + c * 32, u);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float h[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float gb = bf_round(g[i + t]);
        const float ub = bf_round(u[i + t]);
        const float sg = __fdiv_rn(gb, __fadd_rn(1.0f, expf(-gb)));
        h[t] = __fmul_rn(sg, ub);
      }
      pk[i / 2] = pack_bf2(h[0], h[1]);
    }
    if (valid) store_row_u4(a, orow + c * 32, pk, 4);
  }
}

// bf16x2 arithmetic with one round-to-nearest-even of the exact result (the product of two
// bf16 numbers, and the sum of two, are exact in fp32, so this equals the fp32 operation
// followed by a bf16 cast)
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_neg(uint32_t a) { return a ^ 0x80008000u; }

// Two fp32 multiplies in one instruction, each rounded as the scalar one would be; the pair
// moves between float2 and the 64-bit register pair by mov.b64.
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  unsigned long long pa, pb, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(pa) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(pb) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pa), "l"(pb));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) { return make_float2(bf_lo(w), bf_hi(w)); }

// The RoPE (cos, sin) words of the row's position for the head dimension D, loaded before the
// accumulator is ready. Word i holds (cos_i, sin_i).
template <int D>
__device__ __forceinline__ void load_cs_row(const Args& a, bool valid, int grow, uint32_t (&cw)[D / 2]) {
  int p = valid ? a.pos[grow] : 0;
  if (p < 0 || p >= a.P) {
    atomicOr(a.err, MOT_DEV_BAD_POSITION);
    p = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(a.cs + int64_t(p) * D);
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const uint4 v = __ldg(src + i);
    cw[4 * i] = v.x;
    cw[4 * i + 1] = v.y;
    cw[4 * i + 2] = v.z;
    cw[4 * i + 3] = v.w;
  }
}

// The fp32 (cos, sin) row of the row's position (FP32 RoPE profile): D floats, pairs
// (cos_i, sin_i). Read chunk by chunk in pass 2; the table stays in L2.
template <int D>
__device__ __forceinline__ const float4* cs32_row(const Args& a, bool valid, int grow) {
  int p = valid ? a.pos[grow] : 0;
  if (p < 0 || p >= a.P) {
    atomicOr(a.err, MOT_DEV_BAD_POSITION);
    p = 0;
  }
  return reinterpret_cast<const float4*>(a.cs32 + int64_t(p) * D);
}

// Adds the bias of columns [col, col + n) (n a multiple of 8) to v when a bias is given.
template <int NV>
__device__ __forceinline__ void add_bias(const Args& a, int e, int64_t col, float (&v)[NV]) {
  if (a.bias == nullptr) return;
  const uint4* bp = reinterpret_cast<const uint4*>(a.bias + int64_t(e) * a.N + col);
#pragma unroll
  for (int q4 = 0; q4 < NV / 8; ++q4) {
    const uint4 bb = __ldg(bp + q4);
    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * q4 + 2 * k] = __fadd_rn(v[8 * q4 + 2 * k], bf_lo(bw[k]));
      v[8 * q4 + 2 * k + 1] = __fadd_rn(v[8 * q4 + 2 * k + 1], bf_hi(bw[k]));
    }
  }
}

// Per-head QK RMSNorm (fp32, fixed chunk tree) and RoPE on this warp's half of the tile;
// V heads pass through. gs: the norm weights in shared memory, [q / k][expert][D/2] words;
// cw: the bf16 (cos, sin) words of the row's position (BF16 profile); crow: the fp32 table
// row of the row's position (FP32 profile). Pass 1 reads the head from TMEM for its sum of
// squares; pass 2 reads it again, 16 columns of each rotation pair (i, i + D/2) at a time,
// and writes the outputs.
template <int D, bool F32>
__device__ __forceinline__ void epi_qkv(const Args& a, uint32_t taddr, bool valid, int grow, int e, int nt, int half,
                                        const float2* gs, const uint32_t (&cw)[D / 2], const float4* crow) {
  constexpr int HEADS = 128 / D;  // heads in this half
  constexpr int NP = D / 2;       // packed words per head
  uint16_t* orow = a.out + int64_t(grow) * a.ldo + int64_t(nt) * BN + half * 128;
#pragma unroll 1
  for (int hh = 0; hh < HEADS; ++hh) {
    const int h = nt * (BN / D) + half * HEADS + hh;
    const int kind = h < a.Hq ? 0 : (h < a.Hq + a.Hkv ? 1 : 2);  // q, k, v
    const int col0 = half * 128 + hh * D;
    const int64_t gcol0 = int64_t(nt) * BN + col0;  // column in the full output
    uint16_t* ohead = orow + hh * D;
    if (kind == 2) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32(taddr + col0 + c * 32, v);
        add_bias<32>(a, e, gcol0 + c * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf2(v[2 * i], v[2 * i + 1]);
        if (valid) store_row_u4(a, ohead + c * 32, pk, 4);
      }
      continue;
    }
    // pass 1: q = bf16(acc + b); chunk sums of q^2, folded left to right
    float ss = 0.0f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float v[32];
      tmem_ld32(taddr + col0 + c * 32, v);
      add_bias<32>(a, e, gcol0 + c * 32, v);
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 q = bf2_to_f2(pack_bf2(v[i], v[i + 1]));
        const float2 sq = f2_mul(q, q);
        part = __fadd_rn(part, sq.x);
        part = __fadd_rn(part, sq.y);
      }
      ss = c == 0 ? part : __fadd_rn(ss, part);
    }
    const float ms = __fdiv_rn(ss, float(D));
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
    const float2* g = gs + (kind * 2 + e) * NP;  // (g_2w, g_2w+1) in g[w]
    const float2 rstd2 = make_float2(rstd, rstd);
    if constexpr (F32) {
      // pass 2, FP32 profile: u = (q * rstd) * g in fp32, not rounded;
      // out_i = bf16(u_i c + (-u_{i+D/2}) s), out_{i+D/2} = bf16(u_{i+D/2} c + u_i s), each
      // product and the sum rounded to fp32, one cast
#pragma unroll
      for (int c = 0; c < NP / 16; ++c) {
        float4 t[8];  // (cos, sin) of frequencies 16c + 2j and 16c + 2j + 1 in t[j]
#pragma unroll
        for (int j = 0; j < 8; ++j) t[j] = __ldg(crow + c * 8 + j);
        float v1[16], v2[16];
        tmem_ld16(taddr + col0 + c * 16, v1);
        tmem_ld16(taddr + col0 + NP + c * 16, v2);
        add_bias<16>(a, e, gcol0 + c * 16, v1);
        add_bias<16>(a, e, gcol0 + NP + c * 16, v2);
        uint32_t o1[8], o2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int w = c * 8 + j;
          const uint32_t q1 = pack_bf2(v1[2 * j], v1[2 * j + 1]);
          const uint32_t q2 = pack_bf2(v2[2 * j], v2[2 * j + 1]);
          const float2 u1 = f2_mul(f2_mul(bf2_to_f2(q1), rstd2), g[w]);
          const float2 u2 = f2_mul(f2_mul(bf2_to_f2(q2), rstd2), g[NP / 2 + w]);
          const float u1a = u1.x, u1b = u1.y, u2a = u2.x, u2b = u2.y;
          o1[j] = pack_bf2(__fadd_rn(__fmul_rn(u1a, t[j].x), __fmul_rn(-u2a, t[j].y)),
                           __fadd_rn(__fmul_rn(u1b, t[j].z), __fmul_rn(-u2b, t[j].w)));
          o2[j] = pack_bf2(__fadd_rn(__fmul_rn(u2a, t[j].x), __fmul_rn(u1a, t[j].y)),
                           __fadd_rn(__fmul_rn(u2b, t[j].z), __fmul_rn(u1b, t[j].w)));
        }
        if (valid) {
          store_row_u4(a, ohead + c * 16, o1, 2);
          store_row_u4(a, ohead + NP + c * 16, o2, 2);
        }
      }
    } else {
      // pass 2: u = bf16((q * rstd) * g); out_i = bf16(bf16(u_i c) + bf16(-u_{i+D/2} s)),
      // out_{i+D/2} = bf16(bf16(u_{i+D/2} c) + bf16(u_i s)); two neighbouring i per word
#pragma unroll
      for (int c = 0; c < NP / 16; ++c) {
        float v1[16], v2[16];
        tmem_ld16(taddr + col0 + c * 16, v1);
        tmem_ld16(taddr + col0 + NP + c * 16, v2);
        add_bias<16>(a, e, gcol0 + c * 16, v1);
        add_bias<16>(a, e, gcol0 + NP + c * 16, v2);
        uint32_t o1[8], o2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int w = c * 8 + j;  // word index within the head's first half
          const uint32_t q1 = pack_bf2(v1[2 * j], v1[2 * j + 1]);
          const uint32_t q2 = pack_bf2(v2[2 * j], v2[2 * j + 1]);
          const float2 uf1 = f2_mul(f2_mul(bf2_to_f2(q1), rstd2), g[w]);
          const float2 uf2 = f2_mul(f2_mul(bf2_to_f2(q2), rstd2), g[NP / 2 + w]);
          const uint32_t u1 = pack_bf2(uf1.x, uf1.y);
          const uint32_t u2 = pack_bf2(uf2.x, uf2.y);
          const uint32_t c2 = __byte_perm(cw[2 * w], cw[2 * w + 1], 0x5410);  // (cos_2w, cos_2w+1)
          const uint32_t s2 = __byte_perm(cw[2 * w], cw[2 * w + 1], 0x7632);  // (sin_2w, sin_2w+1)
          o1[j] = bf2_add(bf2_mul(u1, c2), bf2_mul(bf2_neg(u2), s2));
          o2[j] = bf2_add(bf2_mul(u2, c2), bf2_mul(u1, s2));
        }
        if (valid) {
          store_row_u4(a, ohead + c * 16, o1, 2);
          store_row_u4(a, ohead + NP + c * 16, o2, 2);
        }
      }
    }
  }
}

// Which 128-row tile of the plan this CTA of the pair works on for pair tile u.
struct PairTile {
  int expert, mt, nt;  // mt: this CTA's m-tile (its partner's if this half is empty)
  bool has_rows;       // false for the empty half of an expert's last pair
};

// Raster order of the pair tiles: bands of `band` pairs; within a band the pair index varies
// fastest, then the N tile. When all pairs' A rows come to at most 32 MB the band is all pairs
// (A is read once, each weight tile is shared by all pairs at once); otherwise a band holds about
// 32 MB of A rows, so they stay in L2 while the band sweeps all N tiles and the weights stream
// past them. (A single band of 58.7 MB of A, the gate/up GEMM at 8192 rows, came back from DRAM
// about 1.8 GB over the sweep; bands of 32 MB read 0.94 GB and ran 2.6 % faster.) The order never
// changes a tile's arithmetic.
__device__ __forceinline__ int band_pairs(int P, int K) {
  const int64_t a_pair_bytes = int64_t(2 * BM) * K * 2;
  if (int64_t(P) * a_pair_bytes <= (int64_t(32) << 20)) return P;
  const int b = int((int64_t(32) << 20) / a_pair_bytes);
  return b < 2 ? 2 : b;
}

__device__ __forceinline__ PairTile decode_pair(int u, int P0, int P, int band, int n_tiles, int nt0, int nt1,
                                                uint32_t rank) {
  PairTile t;
  const int per_band = band * n_tiles;
  const int first_pair = (u / per_band) * band;
  const int bp = P - first_pair < band ? P - first_pair : band;
  const int r = u % per_band;
  const int p = first_pair + r % bp;
  t.nt = r / bp;
  int first, count;
  if (p < P0) {
    t.expert = 0;
    first = 2 * p;
    count = nt0;
  } else {
    t.expert = 1;
    first = 2 * (p - P0);
    count = nt1;
  }
  const int base = t.expert == 0 ? 0 : nt0;
  t.has_rows = first + int(rank) < count;
  t.mt = base + (t.has_rows ? first + int(rank) : first);
  return t;
}

// B_MN: the weight is read as an MN-major operand -- w is [2][K][N] with N contiguous, the
// reduction running over its rows. This gives the input gradient of a forward GEMM whose
// weight is [2][N_fwd][K_fwd] (here K = N_fwd, N = K_fwd) without a transposed copy.
template <int EPI, bool B_MN = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    routed_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a_rows,
                       const __grid_constant__ CUtensorMap tm_w, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;               // used in the leader: its arrival plus both CTAs' stage bytes
  uint64_t* empty = bars + STAGES;     // per CTA: released by the leader's multicast commit
  uint64_t* tfull = bars + 2 * STAGES; // per CTA: accumulator ready
  uint64_t* tempty = bars + 2 * STAGES + 2;  // used in the leader: both CTAs' epilogues done
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float2* gnorm = reinterpret_cast<float2*>(smem + STAGES * STAGE_BYTES + 256);  // [2][2][D/2] fp32 pairs

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  // Launched as a programmatic dependent: the grid may be resident before the preceding kernel
  // (typically the norm that writes A and the plan) has finished. Nothing in global memory is
  // touched before pdl_wait; the tensor maps are kernel parameters. The barriers and tensor
  // memory are set up while the preceding kernel drains.
  pdl_trigger();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_rows);
    tma_prefetch_desc(&tm_w);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * EPI_WARPS);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers are initialized before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(args.ws);
  const int num_m = hdr->num_m_tiles;
  const int nt0 = (hdr->count[0] + kTileRows - 1) / kTileRows;
  const int nt1 = (hdr->count[1] + kTileRows - 1) / kTileRows;
  const bool plan_ok = hdr->magic == kPlanMagic && hdr->T == args.T && num_m >= 0 && num_m <= max_m_tiles(args.T) &&
                       num_m == nt0 + nt1;
  if (!plan_ok && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(args.err, MOT_DEV_PLAN_MISMATCH);
  const int P0 = (nt0 + 1) / 2, P = P0 + (nt1 + 1) / 2;
  // a bad plan (uniform across the grid) leaves no work; the pair still frees its tensor memory
  const int total = plan_ok ? P * args.n_tiles : 0;
  const int band = P > 0 ? band_pairs(P, args.K) : 1;
  const int cluster = int(blockIdx.x >> 1), nclusters = int(gridDim.x >> 1);

  const Tile* tiles = reinterpret_cast<const Tile*>(args.ws + tiles_offset(args.T));
  const int32_t* perm = reinterpret_cast<const int32_t*>(args.ws + perm_offset());
  const int kblocks = args.K / BK;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = cluster; u < total && ok; u += nclusters) {
      const PairTile pt = decode_pair(u, P0, P, band, args.n_tiles, nt0, nt1, rank);
      const Tile tl = tiles[pt.mt];
      const int wrow = pt.expert * args.N + pt.nt * BN + int(rank) * BN_HALF;
      const int arow0 = args.a_plan_order ? tl.list_begin : tl.row0;
      const bool gather = arow0 < 0;
      int r[4] = {0, 0, 0, 0};
      if (gather) {
        const int last = tl.n_rows - 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) r[j] = perm[tl.list_begin + min(4 * lane + j, last)];
      }
      for (int kb = 0; kb < kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err));
        if (!ok) break;
        const uint32_t fb = map_to_rank(smem_u32(&full[stage]), 0);
        if (lane == 0) {
          // the leader arrives once for both CTAs' bytes; the peer's copies only complete bytes
          // on the leader's barrier (a phase cannot complete before the leader's arrival)
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full[stage]), 2 * STAGE_BYTES);
          if constexpr (B_MN) {
            // this CTA's 128 output columns as two 64-column boxes of the stage's 64 weight rows
            const int bx = pt.nt * BN + int(rank) * BN_HALF, by = pt.expert * args.K + kb * BK;
            tma_load_2d_pair(smem_u32(sb + stage * B_BYTES), &tm_w, bx, by, fb);
            tma_load_2d_pair(smem_u32(sb + stage * B_BYTES + B_BYTES / 2), &tm_w, bx + 64, by, fb);
          } else {
            tma_load_2d_pair(smem_u32(sb + stage * B_BYTES), &tm_w, kb * BK, wrow, fb);
          }
          if (!gather) tma_load_2d_pair(smem_u32(sa + stage * A_BYTES), &tm_a, kb * BK, arow0, fb);
        }
        __syncwarp();
        if (gather)
          tma_gather4_pair(smem_u32(sa + stage * A_BYTES + lane * 512), &tm_a_rows, kb * BK, r[0], r[1], r[2], r[3],
                           fb);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (ok) {
      // every stage released by the leader's MMAs: they no longer read this CTA's shared memory
      for (int i = 0; i < STAGES; ++i) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err))) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader CTA only) ----------------
    if (rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN) | (B_MN ? kIdescBMnMajor : 0u);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = cluster; u < total && ok; u += nclusters) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, args.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = smem_u32(sa + stage * A_BYTES), b0 = smem_u32(sb + stage * B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_bf16_pair(d, smem_desc_sw128(a0 + k * 32),
                            B_MN ? smem_desc_mn_sw128(b0 + k * 2048, B_BYTES / 2) : smem_desc_sw128(b0 + k * 32),
                            idesc, (kb | k) != 0);
            mma_commit_pair_multicast(smem_u32(&empty[stage]), 0x3);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) mma_commit_pair_multicast(smem_u32(&tfull[acc]), 0x3);
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued has completed before tensor memory is released
      if (lane == 0) mma_commit_pair(smem_u32(drain));
      __syncwarp();
      mbar_drain(smem_u32(drain), 0);
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    constexpr int D = head_dim(EPI);
    const int quarter = warp & 3;          // the TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;      // which 128 columns of the tile
    const int row_in_tile = quarter * 32 + lane;
    const int et = threadIdx.x - 64;       // 0 .. 255 among the epilogue threads
    if constexpr (is_qkv(EPI)) {
      // both experts' q and k norm weights, once per CTA
      for (int i = et; i < 2 * D; i += 32 * EPI_WARPS) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(i < D ? args.qn : args.kn);
        gnorm[i] = bf2_to_f2(__ldg(src + (i % D)));
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = cluster; u < total; u += nclusters) {
      const PairTile pt = decode_pair(u, P0, P, band, args.n_tiles, nt0, nt1, rank);
      const Tile tl = tiles[pt.mt];
      const bool valid = pt.has_rows && row_in_tile < tl.n_rows;
      const int grow = !valid ? 0 : (args.out_plan_order ? tl.list_begin + row_in_tile : perm[tl.list_begin + row_in_tile]);
      uint32_t cw[D / 2];
      const float4* crow = nullptr;
      if constexpr (is_qkv(EPI)) {
        // this half holds a q or k head
        if (pt.nt * (BN / D) + half * (128 / D) < args.Hq + args.Hkv) {
          if constexpr (rope_f32(EPI))
            crow = cs32_row<D>(args, valid, grow);
          else
            load_cs_row<D>(args, valid, grow, cw);
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, args.err))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * ACC_COLS + (uint32_t(quarter * 32) << 16);
      if constexpr (EPI == EPI_CAST) epi_cast(args, taddr, valid, grow, pt.nt, half);
      if constexpr (EPI == EPI_SWIGLU) epi_swiglu(args, taddr, valid, grow, pt.nt, half);
      if constexpr (is_qkv(EPI))
        epi_qkv<D, rope_f32(EPI)>(args, taddr, valid, grow, pt.expert, pt.nt, half, gnorm, cw, crow);
      tc_fence_before();
      __syncwarp();
      // the accumulator's TMEM reads have completed (tcgen05.wait::ld), so a relaxed arrive suffices
      if (lane == 0) mbar_arrive_cluster_relaxed(map_to_rank(smem_u32(&tempty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the pair may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Weight gradient of one weight set: dW[n][k] = sum over its rows r (ascending) of
// dout[r][n] * a[r][k], fp32, no cast.
// ---------------------------------------------------------------------------
// Both operands are MN-major (the reduction runs over rows): A' = dout^T, 128 n per CTA, and
// B' = a^T, 128 k per CTA, each staged as two 64-column boxes of 128 rows. The set's rows are
// read in the plan's order, 128 at a time (one tile of the plan): from inputs in the plan's
// order a full block is one tiled load per box; from inputs in token order it is one tiled
// load per box when its rows are consecutive token rows. Any other block (and the last partial
// one) is read in 16-row groups: a group of 16 consecutive token rows of the set by one tiled
// load per box, any other group four rows at a time through the plan's permutation, with rows
// past the set pointed outside the tensor, which the copy fills with zeros. The last block's
// MMAs stop at the last 16-row group that holds a row of the set. Pair tiles cover 256 n x
// 256 k; each accumulates its row blocks in ascending order, 16 rows per MMA, into one fp32
// accumulator (no split of the reduction), and the epilogue writes each accumulator row of dW
// from the lane that reads it, in 32-byte sectors. The tiles from split_from on are each done as
// two 256 n x 128 k halves (N = 128 MMAs, one B box per CTA): the host splits the tiles of a last round that
// would leave at least half the clusters idle, so that round takes half as long and its
// exposed epilogue halves too. A half covers its columns with the same ascending row blocks,
// so the bits do not depend on the split.
constexpr int kDwStages = 3;
constexpr int DW_BK = 128;  // rows of the set per stage (one tile of the plan)
constexpr uint32_t DW_A_BYTES = BM * DW_BK * 2, DW_B_BYTES = BN_HALF * DW_BK * 2;
constexpr uint32_t DW_STAGE_BYTES = DW_A_BYTES + DW_B_BYTES;  // 64 KB
constexpr int kGathered = -0x7fffffff - 1;  // a run of tiles read by gathers
constexpr int kNoTile = 0x7fffffff;
constexpr int kDwBars = 2 * kDwStages + 5;
constexpr size_t kDwSmem = 1024 + size_t(kDwStages) * DW_STAGE_BYTES + 256;

struct DwArgs {
  const uint8_t* ws;
  uint32_t* err;
  int T, N, K;  // dout [T][N], a [T][K], dw [N][K]
  int expert;
  float* dw;
  int st32;     // dw is 32-byte aligned (its rows, K * 4 bytes apart, then are too)
  int split_from;  // tiles from this index on are done as two halves of 128 k
  int token_order;  // dout and a in token order (else in the plan's order)
};

// A work item of the dW grid: full tile u, or half h of tile u.
struct DwItem {
  int mt, nt, h, split;
};

__device__ __forceinline__ DwItem dw_item(int it, int split_from, int m_tiles) {
  DwItem r;
  int u;
  if (it < split_from) {
    u = it;
    r.h = 0;
    r.split = 0;
  } else {
    u = split_from + ((it - split_from) >> 1);
    r.h = (it - split_from) & 1;
    r.split = 1;
  }
  r.mt = u % m_tiles;
  r.nt = u / m_tiles;
  return r;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    routed_gemm_dw_kernel(const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_d_rows,
                          const __grid_constant__ CUtensorMap tm_d16, const __grid_constant__ CUtensorMap tm_a,
                          const __grid_constant__ CUtensorMap tm_a_rows, const __grid_constant__ CUtensorMap tm_a16,
                          const DwArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int STAGES = kDwStages;
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * DW_A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * DW_STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kDwBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  pdl_trigger();  // a programmatic dependent: nothing is read before the preceding grid completes
  pdl_wait();
  const PlanHeader* hdr = reinterpret_cast<const PlanHeader*>(args.ws);
  if (hdr->magic != kPlanMagic || hdr->T != args.T) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(args.err, MOT_DEV_PLAN_MISMATCH);
    return;  // uniform across the grid
  }
  if (hdr->count[0] + hdr->count[1] != args.T) return;  // no plan (bad modality): nothing is defined
  const int row_start = args.expert == 0 ? 0 : hdr->count[0];
  const int count = hdr->count[args.expert];
  const int kblocks = (count + DW_BK - 1) / DW_BK;
  // token-order inputs: a row block of the set is one 128-row tile of the plan, whose record says
  // whether its rows are consecutive token rows (then tiled loads) or not (then four-row gathers
  // through the plan's permutation)
  const Tile* plan_tiles = reinterpret_cast<const Tile*>(args.ws + tiles_offset(args.T));
  const int32_t* perm = reinterpret_cast<const int32_t*>(args.ws + perm_offset());
  const int tile_first = args.expert == 0 ? 0 : (hdr->count[0] + kTileRows - 1) / kTileRows;
  const int m_tiles = args.N / BN, n_tiles = args.K / BN;
  const int total = m_tiles * n_tiles;
  const int items = args.split_from + 2 * (total - args.split_from);
  if (kblocks == 0) {
    // a set without rows: its gradient is zero
    const int64_t n4 = int64_t(args.N) * args.K / 4;
    float4* o = reinterpret_cast<float4*>(args.dw);
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x)
      o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int cluster = int(blockIdx.x >> 1), nclusters = int(gridDim.x >> 1);
  if (cluster >= items) return;  // uniform across the pair

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 2 * EPI_WARPS);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_d);
    tma_prefetch_desc(&tm_d_rows);
    tma_prefetch_desc(&tm_d16);
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_rows);
    tma_prefetch_desc(&tm_a16);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    // In token order the set's tiles form runs: consecutive tiles whose rows are consecutive token
    // rows at one offset from their plan positions (a full block is one tiled copy per box at plan
    // position + offset), or consecutive tiles that are not (read in 16-row groups, below). The
    // producer keeps the run of the block it reaches next in warp-uniform values (reductions
    // across the warp), so no block's copies wait on per-block data: a tile-record load, or even
    // a selection on one, per block costs the producer more than the MMA's time for the block. A
    // run is looked up when the loop leaves the last one, in the tile records read 32 at a time,
    // one per lane. In the plan's order the whole set is one run at offset 0.
    const int set_tiles = (count + kTileRows - 1) / kTileRows;
    int rec_chunk = -1, rec_cls = kGathered;  // the class of the set's tile 32 * rec_chunk + lane
    int run_lo = 0, run_hi = kblocks, run_off = 0;  // blocks [run_lo, run_hi) and their offset
    auto load_chunk = [&](int c) {
      if (c != rec_chunk) {
        rec_chunk = c;
        const int t = 32 * c + lane;
        const int r0 = t < set_tiles ? plan_tiles[tile_first + t].row0 : -1;
        rec_cls = r0 >= 0 ? r0 - (row_start + t * kTileRows) : kGathered;
      }
    };
    auto find_run = [&](int kb) {  // warp-collective: the run holding block kb, from kb on
      const int t0 = (kb * DW_BK) / kTileRows;
      load_chunk(t0 >> 5);
      const int cls = __reduce_max_sync(0xffffffffu, lane == (t0 & 31) ? rec_cls : kGathered);
      int end = set_tiles;
      for (int c = t0 >> 5; 32 * c < set_tiles; ++c) {
        load_chunk(c);
        const int t = 32 * c + lane;
        const int first = __reduce_min_sync(0xffffffffu, t > t0 && t < set_tiles && rec_cls != cls ? t : kNoTile);
        if (first != kNoTile) {
          end = first;
          break;
        }
      }
      run_lo = kb;
      run_hi = min(kblocks, end * (kTileRows / DW_BK));
      run_off = cls;
    };
    if (args.token_order) find_run(0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = cluster; it < items && ok; it += nclusters) {
      const DwItem w = dw_item(it, args.split_from, m_tiles);
      const int n0 = w.mt * BN + int(rank) * BN_HALF;  // this CTA's 128 rows of dW
      // this CTA's 128 (a half: 64) columns of the B' operand
      const int k0 = w.nt * BN + (w.split ? w.h * BN_HALF + int(rank) * 64 : int(rank) * BN_HALF);
      const uint32_t stage_tx = w.split ? 2 * (DW_A_BYTES + DW_B_BYTES / 2) : 2 * DW_STAGE_BYTES;
      for (int kb = 0; kb < kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err));
        if (!ok) break;
        const uint32_t fb = map_to_rank(smem_u32(&full[stage]), 0);
        const int row0 = row_start + kb * DW_BK;  // the block's first plan position
        const int valid = count - kb * DW_BK;
        const bool tiled = valid >= DW_BK && run_off != kGathered;
        const int y0 = tiled ? row0 + run_off : 0;  // its first input row
        const uint32_t da = smem_u32(sa + stage * DW_A_BYTES), db = smem_u32(sb + stage * DW_B_BYTES);
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full[stage]), stage_tx);
          if (tiled) {
            tma_load_2d_pair(da, &tm_d, n0, y0, fb);
            tma_load_2d_pair(da + DW_A_BYTES / 2, &tm_d, n0 + 64, y0, fb);
            tma_load_2d_pair(db, &tm_a, k0, y0, fb);
            if (!w.split) tma_load_2d_pair(db + DW_B_BYTES / 2, &tm_a, k0 + 64, y0, fb);
          }
        }
        __syncwarp();
        if (!tiled) {
          // Lane l holds the block's rows 4 l .. 4 l + 3 (rows past the set point outside the
          // tensor and read as zeros). The set's rows ascend in token order, so a 16-row group
          // (lanes 4 g .. 4 g + 3) whose last row is its first + 15 is 16 consecutive token rows:
          // one tiled copy per box from its group leader; any other group is four-row gathers
          // from each of its lanes (a half has no second B box). Same bytes either way.
          int r[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int p = lane * 4 + i;
            r[i] = p < valid ? (args.token_order ? perm[row0 + p] : row0 + p) : args.T;
          }
          const int g = lane >> 2;
          const int first = __shfl_sync(0xffffffffu, r[0], lane & ~3);
          const int last = __shfl_sync(0xffffffffu, r[3], lane | 3);
          const bool whole = 16 * g + 15 < valid && last - first == 15;
#pragma unroll
          for (int box = 0; box < 4; ++box) {
            if (w.split && box == 3) continue;
            const uint32_t base = (box < 2 ? da : db) + (box & 1) * (box < 2 ? DW_A_BYTES / 2 : DW_B_BYTES / 2);
            const int x = (box < 2 ? n0 : k0) + 64 * (box & 1);
            if (whole) {
              if ((lane & 3) == 0)
                tma_load_2d_pair(base + g * 2048, box < 2 ? &tm_d16 : &tm_a16, x, first, fb);
            } else {
              tma_gather4_pair(base + lane * 512,
                               box < 2 ? static_cast<const void*>(&tm_d_rows) : static_cast<const void*>(&tm_a_rows), x,
                               r[0], r[1], r[2], r[3], fb);
            }
          }
        }
        const int next_kb = kb + 1 < kblocks ? kb + 1 : 0;  // the next item starts at block 0
        if (args.token_order && (next_kb < run_lo || next_kb >= run_hi)) find_run(next_kb);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (ok) {
      for (int i = 0; i < STAGES; ++i) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err))) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader CTA only) ----------------
    if (rank == 0) {
      constexpr uint32_t idesc_full = idesc_bf16_f32(2 * BM, BN) | kIdescAMnMajor | kIdescBMnMajor;
      constexpr uint32_t idesc_half = idesc_bf16_f32(2 * BM, BN_HALF) | kIdescAMnMajor | kIdescBMnMajor;
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int it = cluster; it < items && ok; it += nclusters) {
        const uint32_t idesc = it < args.split_from ? idesc_full : idesc_half;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, args.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < kblocks; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a0 = smem_u32(sa + stage * DW_A_BYTES), b0 = smem_u32(sb + stage * DW_B_BYTES);
            // K16 steps up to the last 16-row group that holds a row of the set
            const int valid = count - kb * DW_BK;
            const int nk = valid >= DW_BK ? DW_BK / 16 : (valid + 15) / 16;
#pragma unroll
            for (int k = 0; k < DW_BK / 16; ++k)
              if (k < nk)
                mma_bf16_pair(d, smem_desc_mn_sw128(a0 + k * 2048, DW_A_BYTES / 2), smem_desc_mn_sw128(b0 + k * 2048, DW_B_BYTES / 2),
                              idesc, (kb | k) != 0);
            mma_commit_pair_multicast(smem_u32(&empty[stage]), 0x3);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) mma_commit_pair_multicast(smem_u32(&tfull[acc]), 0x3);
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (lane == 0) mma_commit_pair(smem_u32(drain));
      __syncwarp();
      mbar_drain(smem_u32(drain), 0);
    }
  } else {
    // ---------------- epilogue (both CTAs): fp32 rows of dW ----------------
    // Each lane writes its accumulator row's 32 columns per TMEM load as whole 32-byte sectors
    // (16-byte pieces when dw is only 16-byte aligned).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = cluster; it < items; it += nclusters) {
      const DwItem w = dw_item(it, args.split_from, m_tiles);
      const int n_row = w.mt * BN + int(rank) * BN_HALF + quarter * 32 + lane;  // this lane's dW row
      const int wcols = w.split ? 64 : 128;  // this warp's columns of the item
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, args.err))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * ACC_COLS + (uint32_t(quarter * 32) << 16) + half * wcols;
      float* drow = args.dw + int64_t(n_row) * args.K + w.nt * BN + w.h * BN_HALF + half * wcols;
#pragma unroll 1
      for (int c = 0; c < wcols / 32; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        if (args.st32) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(drow + c * 32 + 8 * i),
                         "f"(v[8 * i]), "f"(v[8 * i + 1]), "f"(v[8 * i + 2]), "f"(v[8 * i + 3]), "f"(v[8 * i + 4]),
                         "f"(v[8 * i + 5]), "f"(v[8 * i + 6]), "f"(v[8 * i + 7])
                         : "memory");
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(drow + c * 32 + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2],
                                                                            v[4 * i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(map_to_rank(smem_u32(&tempty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Clusters of the pair kernel that fit on the device at once (computed once per device).
template <int EPI, bool B_MN = false>
static int max_active_pairs(int dev) {
  static std::atomic<int> cache[kMaxDevices];
  int v = cache[dev].load();
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, routed_gemm_kernel<EPI, B_MN>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count(dev) / 2;
  }
  cache[dev].store(n);
  return n;
}

template <int EPI, bool B_MN = false>
static int launch(const void* a, const void* w, int T, int N, int K, const Args& args, int dev, cudaStream_t s) {
  CUtensorMap tm_a, tm_rows, tm_w;
  const bool w_ok = B_MN ? make_tmap_bf16(&tm_w, w, uint64_t(N), uint64_t(2) * K, 64, BK)
                         : make_tmap_bf16(&tm_w, w, uint64_t(K), uint64_t(2) * N, BK, BN_HALF);
  if (!make_tmap_bf16(&tm_a, a, uint64_t(K), uint64_t(T), BK, BM) ||
      !make_tmap_bf16(&tm_rows, a, uint64_t(K), uint64_t(T), BK, 1) || !w_ok)
    return MOT_ERR_CUDA;
  if (cudaFuncSetAttribute(routed_gemm_kernel<EPI, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(SMEM_BYTES)) != cudaSuccess)
    return MOT_ERR_CUDA;
  // upper bound of pair tiles: ceil(tiles0 / 2) + ceil(tiles1 / 2) <= (ceil(T / 128) + 1) / 2 + 1
  const int64_t pairs_max = ((int64_t(T) + BM - 1) / BM + 1) / 2 + 1;
  const int64_t work_max = pairs_max * int64_t(N / BN);
  const int64_t cap = max_active_pairs<EPI, B_MN>(dev);
  const int64_t clusters = work_max < cap ? work_max : cap;
  Args la = args;
  la.st32 = (reinterpret_cast<uintptr_t>(args.out) % 32 == 0 && (int64_t(args.ldo) * 2) % 32 == 0) ? 1 : 0;
  if (launch_dependent(routed_gemm_kernel<EPI, B_MN>, dim3(unsigned(2 * clusters)), dim3(THREADS), SMEM_BYTES, s,
                       tm_a, tm_rows, tm_w, la) != cudaSuccess) {
    cudaGetLastError();
    return MOT_ERR_CUDA;
  }
  return MOT_OK;
}

}  // namespace gemm
}  // namespace mot

using namespace mot;

// Shared by both RoPE profiles: validation, then one launch. table_bf16 / table_f32: the
// (cos, sin) table of the profile (the other is null).
static int routed_qkv_entry(const mot_bf16* x, const mot_bf16* w_qkv, const mot_bf16* b_qkv, const mot_bf16* q_norm_w,
                            const mot_bf16* k_norm_w, const int32_t* pos, const mot_bf16* table_bf16,
                            const float* table_f32, int P, int64_t T, int H, int Hq, int Hkv, int D, float eps,
                            void* ws, size_t ws_bytes, mot_bf16* qkv_out, void* stream) {
  const void* table = table_f32 ? static_cast<const void*>(table_f32) : static_cast<const void*>(table_bf16);
  if (!x || !w_qkv || !q_norm_w || !k_norm_w || !pos || !table || !ws || !qkv_out) return MOT_ERR_NULL;
  if (T < 1 || T > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (D != 64 && D != 128) return MOT_ERR_GEOMETRY;
  if (Hq < 1 || Hkv < 1 || Hq > 1024 || Hkv > 1024) return MOT_ERR_GEOMETRY;
  const int64_t N = int64_t(Hq + 2 * Hkv) * D;
  if (N % gemm::BN != 0 || N > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (H < gemm::BK || H % gemm::BK != 0 || H > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (P < 1 || P > MOT_MAX_TOKENS) return MOT_ERR_ARG;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return MOT_ERR_ARG;
  if (!aligned16(x) || !aligned16(w_qkv) || (b_qkv && !aligned16(b_qkv)) || !aligned16(q_norm_w) ||
      !aligned16(k_norm_w) || !aligned16(pos) || !aligned16(table) || !aligned16(ws) || !aligned16(qkv_out))
    return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {x, w_qkv, b_qkv, q_norm_w, k_norm_w, pos, table, ws, qkv_out};
  int dev = -1;
  int st = check_device(s, ptrs, 9, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  gemm::Args a{};
  a.ws = static_cast<const uint8_t*>(ws);
  a.err = &static_cast<PlanHeader*>(ws)->error;
  a.T = int(T);
  a.N = int(N);
  a.K = H;
  a.n_tiles = int(N / gemm::BN);
  a.out = qkv_out;
  a.ldo = int(N);
  a.bias = b_qkv;
  a.qn = q_norm_w;
  a.kn = k_norm_w;
  a.pos = pos;
  a.cs = table_bf16;
  a.cs32 = table_f32;
  a.P = P;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.eps = eps;
  if (table_f32) {
    if (D == 64) return gemm::launch<gemm::EPI_QKV64_F32>(x, w_qkv, int(T), int(N), H, a, dev, s);
    return gemm::launch<gemm::EPI_QKV128_F32>(x, w_qkv, int(T), int(N), H, a, dev, s);
  }
  if (D == 64) return gemm::launch<gemm::EPI_QKV64>(x, w_qkv, int(T), int(N), H, a, dev, s);
  return gemm::launch<gemm::EPI_QKV128>(x, w_qkv, int(T), int(N), H, a, dev, s);
}

extern "C" int mot_routed_qkv_norm_rope(const mot_bf16* x, const mot_bf16* w_qkv, const mot_bf16* b_qkv,
                                        const mot_bf16* q_norm_w, const mot_bf16* k_norm_w, const int32_t* pos,
                                        const mot_bf16* rope_cs, int P, int64_t T, int H, int Hq, int Hkv, int D,
                                        float eps, void* ws, size_t ws_bytes, mot_bf16* qkv_out, void* stream) {
  if (rope_cs == nullptr) return MOT_ERR_NULL;
  return routed_qkv_entry(x, w_qkv, b_qkv, q_norm_w, k_norm_w, pos, rope_cs, nullptr, P, T, H, Hq, Hkv, D, eps, ws,
                          ws_bytes, qkv_out, stream);
}

extern "C" int mot_routed_qkv_norm_rope_fp32(const mot_bf16* x, const mot_bf16* w_qkv, const mot_bf16* b_qkv,
                                             const mot_bf16* q_norm_w, const mot_bf16* k_norm_w, const int32_t* pos,
                                             const float* rope_cs_f32, int P, int64_t T, int H, int Hq, int Hkv,
                                             int D, float eps, void* ws, size_t ws_bytes, mot_bf16* qkv_out,
                                             void* stream) {
  if (rope_cs_f32 == nullptr) return MOT_ERR_NULL;
  return routed_qkv_entry(x, w_qkv, b_qkv, q_norm_w, k_norm_w, pos, nullptr, rope_cs_f32, P, T, H, Hq, Hkv, D, eps,
                          ws, ws_bytes, qkv_out, stream);
}

extern "C" int mot_routed_gemm_dx(const mot_bf16* dout, const mot_bf16* w, int64_t T, int N, int K, int flags,
                                  void* ws, size_t ws_bytes, mot_bf16* dx, void* stream) {
  if (!dout || !w || !ws || !dx) return MOT_ERR_NULL;
  if ((flags & ~(MOT_A_PLAN_ORDER | MOT_OUT_PLAN_ORDER)) != 0) return MOT_ERR_ARG;
  if (T < 1 || T > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  // the forward's K is the output width (tiles of 256), its N the reduction (blocks of 64)
  if (K < gemm::BN || K % gemm::BN != 0 || K > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (N < gemm::BK || N % gemm::BK != 0 || N > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (!aligned16(dout) || !aligned16(w) || !aligned16(ws) || !aligned16(dx)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {dout, w, ws, dx};
  int dev = -1;
  int st = check_device(s, ptrs, 4, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  gemm::Args a{};
  a.ws = static_cast<const uint8_t*>(ws);
  a.err = &static_cast<PlanHeader*>(ws)->error;
  a.T = int(T);
  a.N = K;
  a.K = N;
  a.n_tiles = K / gemm::BN;
  a.out = dx;
  a.ldo = K;
  a.a_plan_order = (flags & MOT_A_PLAN_ORDER) != 0;
  a.out_plan_order = (flags & MOT_OUT_PLAN_ORDER) != 0;
  return gemm::launch<gemm::EPI_CAST, true>(dout, w, int(T), K, N, a, dev, s);
}

extern "C" int mot_routed_gemm_dw(const mot_bf16* dout, const mot_bf16* a_in, int64_t T, int N, int K,
                                  int expert, int flags, void* ws, size_t ws_bytes, float* dw, void* stream) {
  if (!dout || !a_in || !ws || !dw) return MOT_ERR_NULL;
  if (expert != 0 && expert != 1) return MOT_ERR_ARG;
  if ((flags & ~MOT_A_PLAN_ORDER) != 0) return MOT_ERR_ARG;
  if (T < 1 || T > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (N < gemm::BN || N % gemm::BN != 0 || N > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (K < gemm::BN || K % gemm::BN != 0 || K > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (!aligned16(dout) || !aligned16(a_in) || !aligned16(ws) || !aligned16(dw)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {dout, a_in, ws, dw};
  int dev = -1;
  int st = check_device(s, ptrs, 4, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  CUtensorMap tm_d, tm_d_rows, tm_d16, tm_a, tm_a_rows, tm_a16;
  if (!make_tmap_bf16(&tm_d, dout, uint64_t(N), uint64_t(T), 64, gemm::DW_BK) ||
      !make_tmap_bf16(&tm_d_rows, dout, uint64_t(N), uint64_t(T), 64, 1) ||
      !make_tmap_bf16(&tm_d16, dout, uint64_t(N), uint64_t(T), 64, 16) ||
      !make_tmap_bf16(&tm_a16, a_in, uint64_t(K), uint64_t(T), 64, 16) ||
      !make_tmap_bf16(&tm_a, a_in, uint64_t(K), uint64_t(T), 64, gemm::DW_BK) ||
      !make_tmap_bf16(&tm_a_rows, a_in, uint64_t(K), uint64_t(T), 64, 1))
    return MOT_ERR_CUDA;
  if (cudaFuncSetAttribute(gemm::routed_gemm_dw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(gemm::kDwSmem)) != cudaSuccess)
    return MOT_ERR_CUDA;
  gemm::DwArgs a{};
  a.ws = static_cast<const uint8_t*>(ws);
  a.err = &static_cast<PlanHeader*>(ws)->error;
  a.T = int(T);
  a.N = N;
  a.K = K;
  a.expert = expert;
  a.dw = dw;
  a.st32 = reinterpret_cast<uintptr_t>(dw) % 32 == 0 ? 1 : 0;
  a.token_order = (flags & MOT_A_PLAN_ORDER) ? 0 : 1;
  const int64_t total = int64_t(N / gemm::BN) * (K / gemm::BN);
  // same threads and cluster shape as the routed kernel and more shared memory than half an
  // SM: one pair per two SMs, the same residency
  const int64_t cap = gemm::max_active_pairs<gemm::EPI_CAST, true>(dev);
  // the tiles of a last round that would leave at least half the clusters idle are split in
  // halves (all of them when the whole problem is such a round)
  const int64_t rem = total > cap ? total % cap : total;
  const int64_t split_from = rem > 0 && 2 * rem <= cap ? total - rem : total;
  const int64_t items = split_from + 2 * (total - split_from);
  if (items > INT32_MAX) return MOT_ERR_GEOMETRY;
  a.split_from = int(split_from);
  const int64_t clusters = items < cap ? items : cap;
  const cudaError_t e = launch_dependent(gemm::routed_gemm_dw_kernel, dim3(unsigned(2 * clusters)),
                                         dim3(gemm::THREADS), gemm::kDwSmem, s, tm_d, tm_d_rows, tm_d16, tm_a, tm_a_rows, tm_a16, a);
  return e == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}

extern "C" int mot_routed_gemm(const mot_bf16* a_in, const mot_bf16* w, int64_t T, int N, int K, int epilogue,
                               void* ws, size_t ws_bytes, mot_bf16* out, void* stream) {
  if (!a_in || !w || !ws || !out) return MOT_ERR_NULL;
  const int order_flags = epilogue & (MOT_A_PLAN_ORDER | MOT_OUT_PLAN_ORDER);
  epilogue &= ~(MOT_A_PLAN_ORDER | MOT_OUT_PLAN_ORDER);
  if (epilogue != MOT_EPI_CAST && epilogue != MOT_EPI_SWIGLU) return MOT_ERR_ARG;
  if (T < 1 || T > MOT_MAX_TOKENS) return MOT_ERR_GEOMETRY;
  if (N < gemm::BN || N % gemm::BN != 0 || N > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (K < gemm::BK || K % gemm::BK != 0 || K > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (!aligned16(a_in) || !aligned16(w) || !aligned16(ws) || !aligned16(out)) return MOT_ERR_ALIGN;
  if (ws_bytes < size_t(plan_bytes(T))) return MOT_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {a_in, w, ws, out};
  int dev = -1;
  int st = check_device(s, ptrs, 4, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  gemm::Args a{};
  a.ws = static_cast<const uint8_t*>(ws);
  a.err = &static_cast<PlanHeader*>(ws)->error;
  a.T = int(T);
  a.N = N;
  a.K = K;
  a.n_tiles = N / gemm::BN;
  a.out = out;
  a.ldo = epilogue == MOT_EPI_SWIGLU ? N / 2 : N;
  a.a_plan_order = (order_flags & MOT_A_PLAN_ORDER) != 0;
  a.out_plan_order = (order_flags & MOT_OUT_PLAN_ORDER) != 0;
  if (epilogue == MOT_EPI_SWIGLU) return gemm::launch<gemm::EPI_SWIGLU>(a_in, w, int(T), N, K, a, dev, s);
  return gemm::launch<gemm::EPI_CAST>(a_in, w, int(T), N, K, a, dev, s);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of mot_routed_gemm.
//
// Some callers cannot hand this library a workspace: engines that reserve all device
// memory once at start-up and forbid any later allocation, and plug-ins whose host
// framework owns the device memory and gives them no allocator. For them the routing plan
// lives in the file-scope array below, which every GPU that loads the library keeps until
// the process exits. Host code may not use the array's name as a device address (on the
// host it only stands in for the symbol); its device address is looked up once per device
// with cudaGetSymbolAddress while that device is current, on the first call made on that
// device. All calls on a device share the array and it keeps the last call's plan, so calls
// whose work overlaps on the GPU (other streams, or other host threads) race and must be
// serialized by the caller. Each call rebuilds the plan, which rewrites every field the
// GEMM reads and clears the error word first.
// ---------------------------------------------------------------------------
namespace mot {
namespace noalloc {

constexpr int64_t kMaxTokens = MOT_NOALLOC_MAX_TOKENS;
// the routing plan of kMaxTokens rows, laid out exactly as in a caller's workspace
constexpr size_t kScratchBytes = size_t(plan_bytes(kMaxTokens));
static_assert(kScratchBytes >= size_t(plan_bytes(kMaxTokens)), "the array must hold the largest plan");
static_assert(kScratchBytes <= (size_t(1) << 20), "the array stays a modest fixed size");

static __device__ __align__(256) uint8_t g_plan_scratch[kScratchBytes];

static std::mutex g_mu;
static void* g_scratch_addr[kMaxDevices];

// Device address of g_plan_scratch on `dev`, which must be the current device.
static int scratch_for(int dev, uint8_t** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOT_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
  return MOT_OK;
}

__global__ void copy_error_word(const uint8_t* scratch, uint32_t* flags) {
  *flags = reinterpret_cast<const PlanHeader*>(scratch)->error;
}

}  // namespace noalloc
}  // namespace mot

extern "C" int mot_routed_gemm_noalloc(const mot_bf16* a_in, const mot_bf16* w, const uint8_t* mod, int64_t T, int N,
                                       int K, int epilogue, mot_bf16* out, uint32_t* device_flags, void* stream) {
  if (!a_in || !w || !mod || !out) return MOT_ERR_NULL;
  if (epilogue != MOT_EPI_CAST && epilogue != MOT_EPI_SWIGLU) return MOT_ERR_ARG;
  if (T > noalloc::kMaxTokens) return MOT_ERR_NOALLOC_LIMIT;
  if (T < 1) return MOT_ERR_GEOMETRY;
  if (N < gemm::BN || N % gemm::BN != 0 || N > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (K < gemm::BK || K % gemm::BK != 0 || K > (1 << 20)) return MOT_ERR_GEOMETRY;
  if (!aligned16(a_in) || !aligned16(w) || !aligned16(out) || (reinterpret_cast<uintptr_t>(device_flags) & 3u))
    return MOT_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* ptrs[] = {a_in, w, mod, out, device_flags};
  int dev = -1;
  int st = check_device(s, ptrs, 5, &dev);
  if (st != MOT_OK) return st;
  DeviceGuard guard(dev);
  uint8_t* ws = nullptr;
  st = noalloc::scratch_for(dev, &ws);
  if (st != MOT_OK) return st;
  st = enqueue_route_plan(mod, int(T), ws, s);
  if (st != MOT_OK) return st;
  gemm::Args a{};
  a.ws = ws;
  a.err = &reinterpret_cast<PlanHeader*>(ws)->error;
  a.T = int(T);
  a.N = N;
  a.K = K;
  a.n_tiles = N / gemm::BN;
  a.out = out;
  a.ldo = epilogue == MOT_EPI_SWIGLU ? N / 2 : N;
  st = epilogue == MOT_EPI_SWIGLU ? gemm::launch<gemm::EPI_SWIGLU>(a_in, w, int(T), N, K, a, dev, s)
                                  : gemm::launch<gemm::EPI_CAST>(a_in, w, int(T), N, K, a, dev, s);
  if (st != MOT_OK || device_flags == nullptr) return st;
  noalloc::copy_error_word<<<1, 1, 0, s>>>(ws, device_flags);
  return cudaGetLastError() == cudaSuccess ? MOT_OK : MOT_ERR_CUDA;
}
