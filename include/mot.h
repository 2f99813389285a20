/*
 * mot.h -- C ABI of the Mixture-of-Transformers (MoT) token-routed dense projection
 * library for NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [RFC-435]  "[RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435"
 *   [PR-1402]  "[omni, model, ops, ckpt, config, docs] feat: support Bagel in SeedOmni - #1402"
 *   [PR-503]   "[WS1][CUDA][Qwen3-Next] MoE route/combine contract with a batch-invariant
 *               grouped expert GEMM (RFC #428 stack 5/8) - #503"
 *
 * The method ([RFC-435] §1 Motivation, item 1): a packed batch of T token rows; each row
 * uses one of two weight sets -- und (modality 0: text and ViT tokens) or gen (modality 1:
 * VAE-latent tokens) -- chosen by a fixed per-token index; every GEMM and norm picks its
 * weight set per row, and a row's output bytes must not depend on the modality mix, the
 * order or the size of the pack.
 *
 * Conventions for every entry point
 *   - Tensors are plain device pointers to dense row-major arrays; bf16 values are passed
 *     as raw 16-bit patterns (mot_bf16). Every bf16 tensor and the workspace must start on
 *     a 16-byte boundary. The caller owns all memory; the library allocates nothing and
 *     keeps no state between calls apart from per-device attribute caches and the fixed
 *     plan array of mot_routed_gemm_noalloc.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream of the current
 *     device). Every pointer must belong to the stream's device (the device guard of
 *     [PR-503]'s RMSNorm launcher commit); the launch runs on that device.
 *   - Calls are asynchronous on `stream`. A nonzero return is a host-detected error: no
 *     kernel was launched and no output was written (fail closed: [RFC-435] §3 Numerical
 *     contract). Errors found on the device (a modality other than 0/1, a position
 *     outside the RoPE table, a plan that does not match the call, a pipeline wait that
 *     timed out) set bits in the workspace's error word, read by mot_device_status.
 *     Outputs are defined only when both are clean.
 *   - Numerics ([RFC-435] §3): fixed fp32 accumulation and reduction order, no split-K,
 *     stream-K or atomics in any reduction, no TF32 or fast math, round-to-nearest-even
 *     casts only at the points each entry point declares.
 */
#ifndef MOT_H
#define MOT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOT_ABI_VERSION 4

/* host-detected status codes (return values) */
#define MOT_OK            0
#define MOT_ERR_NULL      1  /* a required pointer is NULL */
#define MOT_ERR_ALIGN     2  /* a pointer is not 16-byte aligned */
#define MOT_ERR_GEOMETRY  3  /* unsupported shape: see each entry point */
#define MOT_ERR_DEVICE    4  /* a pointer is not device memory of the stream's device */
#define MOT_ERR_WORKSPACE 5  /* workspace smaller than mot_workspace_bytes(T) */
#define MOT_ERR_ARCH      6  /* the stream's device is not compute capability 10.3 */
#define MOT_ERR_CUDA      7  /* a CUDA runtime call or a launch failed */
#define MOT_ERR_ARG       8  /* any other invalid argument (epilogue id, eps, P ...) */
#define MOT_ERR_NOALLOC_LIMIT 9  /* T above MOT_NOALLOC_MAX_TOKENS (mot_routed_gemm_noalloc) */

/* device-detected error bits, OR-ed into the workspace error word */
#define MOT_DEV_BAD_MODALITY  0x1u  /* a modality index other than 0 or 1 */
#define MOT_DEV_TIMEOUT       0x2u  /* a pipeline wait gave up after about one second */
#define MOT_DEV_PLAN_MISMATCH 0x4u  /* the workspace holds no plan for this T */
#define MOT_DEV_BAD_POSITION  0x8u  /* a RoPE position outside [0, P) (clamped to 0) */
#define MOT_DEV_BAD_SEQUENCE  0x10u /* an attention sequence descriptor out of range */
#define MOT_DEV_BAD_TIME      0x20u /* SDE step times outside 0 <= t_next < t_i <= 1 */

/* epilogues of mot_routed_gemm */
#define MOT_EPI_CAST   0  /* out = bf16(acc) */
#define MOT_EPI_SWIGLU 1  /* out = bf16(silu(bf16(acc_gate)) * bf16(acc_up)) */
/* row-order flags, OR-ed into mot_routed_gemm's epilogue argument. "Plan order" is the row
 * order of the routing plan: the und rows in ascending order, then the gen rows (the order
 * mot_gather_rows produces). The flags change where rows are read and written, never their
 * values. */
#define MOT_A_PLAN_ORDER   0x100  /* row i of `a` is the plan's i-th row */
#define MOT_OUT_PLAN_ORDER 0x200  /* row i of `out` is the plan's i-th row */

/* weight-set masks of the norm backward's partials and fold */
#define MOT_SET_UND  1
#define MOT_SET_GEN  2
#define MOT_SET_BOTH 3

/* largest packed batch the library accepts */
#define MOT_MAX_TOKENS (1 << 24)

/* largest packed batch of mot_routed_gemm_noalloc (its plan lives in a fixed device array) */
#define MOT_NOALLOC_MAX_TOKENS 65536

typedef uint16_t mot_bf16; /* raw bfloat16 bit pattern */

/* ABI version of the loaded library; a binding refuses to run against another one
 * (the stale-binding check of [PR-503]'s evidence-runner commit). */
int mot_abi_version(void);

/* Static, NUL-terminated description of a status code. */
const char* mot_status_string(int status);

/* Bytes of workspace needed for a pack of T rows (0 if T is out of range). The workspace
 * holds the routing plan and the device error word; the caller allocates it. */
size_t mot_workspace_bytes(int64_t T);

/*
 * mot_route_plan -- routing pre-pass ([RFC-435] §1 item 1: a fixed index set per token;
 * §6 Contribution notes: both weight sets always present).
 *   mod   [T] uint8 device array: 0 = und, 1 = gen.
 *   ws    device workspace of at least mot_workspace_bytes(T) bytes.
 * Writes into ws the row list of each expert in ascending row order and the table of
 * 128-row tiles that the routed GEMMs walk, and clears the error word. A modality other
 * than 0/1 sets MOT_DEV_BAD_MODALITY and leaves a plan with no tiles, so later GEMMs on
 * this workspace write nothing. The plan depends only on mod, so one plan serves every
 * routed GEMM of a layer.
 */
int mot_route_plan(const uint8_t* mod, int64_t T, void* ws, size_t ws_bytes, void* stream);

/*
 * mot_fused_add_rmsnorm -- residual add, then RMSNorm with the row's weight set
 * ([RFC-435] §5 claim order, item 2; RMSNorm convention of [PR-503]'s zero-centred
 * RMSNorm commit with offset 0; fixed 32-wide chunked reduction of its "On exactness
 * against vLLM" section).
 *   x, res    [T][H] bf16          inputs.
 *   w         [2][H] bf16          norm weight of und (row 0) and gen (row 1).
 *   mod       [T] uint8            modality of each row.
 *   eps       > 0 and finite       added to the mean square inside the square root.
 *   y         [T][H] bf16          normalized output.
 *   res_out   [T][H] bf16          new residual stream; may alias res (in place).
 *   ws        optional workspace   if not NULL (ws_bytes >= mot_workspace_bytes(T)), one extra
 *                                  CTA of the same launch writes the routing plan of mod into
 *                                  it, exactly as mot_route_plan does, so the layer's routed
 *                                  GEMMs need no separate pre-pass launch.
 * Per row: s = bf16(x + res) -> res_out; lane l of a 32-lane group owns columns
 * 256j + 8l + t; p_l = sequential fp32 sum of s^2 (j outer, t inner); partials combine
 * by an xor butterfly 16, 8, 4, 2, 1; rstd = 1 / sqrt(p / H + eps) with IEEE division and
 * square root; y = bf16((s * rstd) * w[mod]). A row with an invalid modality gets res_out
 * but no y (MOT_DEV_BAD_MODALITY in ws). Geometry: H a multiple of 256, 256 <= H <= 8192;
 * 1 <= T <= MOT_MAX_TOKENS.
 */
int mot_fused_add_rmsnorm(const mot_bf16* x, const mot_bf16* res, const mot_bf16* w,
                          const uint8_t* mod, int64_t T, int H, float eps,
                          mot_bf16* y, mot_bf16* res_out, void* ws, size_t ws_bytes, void* stream);

/*
 * mot_routed_qkv_norm_rope -- routed QKV projection with per-head QK RMSNorm in fp32 and
 * RoPE with Q/K in bf16 ([PR-1402] "What does this PR do?": MoT dual-branch routed Q/K/V
 * with fused qkv_proj_{und,gen} weights, per-head QK RMSNorm and packed RoPE; [RFC-435]
 * §2 Reference hazards: QK norm in FP32, then RoPE and Q/K in BF16).
 *   x         [T][H] bf16             normalized hidden states (mot_fused_add_rmsnorm's y).
 *   w_qkv     [2][N][H] bf16          fused weights, N = (Hq + 2 Hkv) D, rows ordered
 *                                     q heads, k heads, v heads (nn.Linear layout).
 *   b_qkv     [2][N] bf16 or NULL     optional bias, added in fp32 before the cast.
 *   q_norm_w, k_norm_w [2][D] bf16    per-expert QK-norm weights shared by all heads.
 *   pos       [T] int32               RoPE position of each row, 0 <= pos < P.
 *   rope_cs   [P][D/2][2] bf16        (cos, sin) table, see mot_rope_table_fill_host.
 *   ws        workspace holding the plan of mot_route_plan for this T (same stream).
 *   qkv_out   [T][N] bf16             output in the original row order.
 * Per row r with e = mod[r]: acc = sum_k x[r][k] W[e][n][k] in fp32 (tensor cores, fixed
 * K order); q = bf16(acc + b); for each Q/K head: rstd = 1/sqrt(ss/D + eps) with ss the
 * fixed chunk tree (32-wide sequential chunks, left fold); u = bf16((q * rstd) * g[e]);
 * out_i = bf16(bf16(u_i c) + bf16(partner_i s)) with partner -u_{i+D/2} (i < D/2) or
 * u_{i-D/2}; V heads: out = q. Geometry: D in {64, 128}; Hq, Hkv >= 1; N a multiple of
 * 256; H a multiple of 64; P >= 1.
 */
int mot_routed_qkv_norm_rope(const mot_bf16* x, const mot_bf16* w_qkv, const mot_bf16* b_qkv,
                             const mot_bf16* q_norm_w, const mot_bf16* k_norm_w,
                             const int32_t* pos, const mot_bf16* rope_cs, int P,
                             int64_t T, int H, int Hq, int Hkv, int D, float eps,
                             void* ws, size_t ws_bytes, mot_bf16* qkv_out, void* stream);

/*
 * mot_routed_qkv_norm_rope_fp32 -- the same projection with the FP32 RoPE profile
 * ([RFC-435] open question 4: keep the reference BF16 RoPE or define an FP32 profile; §3: a
 * profile change is a new numeric fingerprint). Arguments as mot_routed_qkv_norm_rope except
 *   rope_cs_f32  [P][D/2][2] fp32   (cos, sin) table, see mot_rope_table_fill_host_fp32.
 * Per Q/K head: u = (q * rstd) * g[e] in fp32 without a cast, then
 * out_i = bf16(fp32(u_i c) + fp32(partner_i s)): both products and the sum rounded to fp32,
 * one bf16 cast. q = bf16(acc + b), the statistics and V heads are those of the BF16 profile.
 * Errors and ownership as mot_routed_qkv_norm_rope; rope_cs_f32 must be 16-byte aligned.
 */
int mot_routed_qkv_norm_rope_fp32(const mot_bf16* x, const mot_bf16* w_qkv, const mot_bf16* b_qkv,
                                  const mot_bf16* q_norm_w, const mot_bf16* k_norm_w,
                                  const int32_t* pos, const float* rope_cs_f32, int P,
                                  int64_t T, int H, int Hq, int Hkv, int D, float eps,
                                  void* ws, size_t ws_bytes, mot_bf16* qkv_out, void* stream);

/*
 * mot_routed_gemm -- routed dense projection for the O, gate/up and down projections
 * ([RFC-435] §5 mot_routed_gemm and mot_swiglu_mlp; [PR-503] grouped expert GEMM commit:
 * one writer per row, grouped result equal to the per-expert GEMM).
 *   a    [T][K] bf16           input rows in the original order.
 *   w    [2][N][K] bf16        per-expert weights (nn.Linear layout).
 *   ws   workspace holding the plan of mot_route_plan for this T (same stream).
 *   epilogue MOT_EPI_CAST:    out [T][N]   = bf16(acc).
 *   epilogue MOT_EPI_SWIGLU:  w is the gate/up weight in the layout written by
 *                             mot_swiglu_interleave (N = 2 I); out [T][I] =
 *                             bf16(g / (1 + expf(-g)) * u), g = bf16(acc_gate),
 *                             u = bf16(acc_up), fp32 arithmetic.
 * With MOT_A_PLAN_ORDER every 128-row tile of `a` is contiguous and is read with one tiled
 * copy; without it, tiles whose rows are not consecutive are gathered four rows at a time.
 * Geometry: N a multiple of 256, K a multiple of 64.
 */
int mot_routed_gemm(const mot_bf16* a, const mot_bf16* w, int64_t T, int N, int K, int epilogue,
                    void* ws, size_t ws_bytes, mot_bf16* out, void* stream);

/*
 * mot_routed_gemm_noalloc -- mot_routed_gemm for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment variant of the entry point above.
 * Engines that reserve all device memory once at start-up, and plug-ins whose host framework
 * owns the device memory and offers them no allocator, cannot provide the workspace that
 * mot_routed_gemm needs. This call takes the modality index itself and keeps the routing plan
 * in a fixed array of the library's own device memory (about 264 KB, held by every GPU that
 * loads the library until the process exits), then runs the same routed GEMM. It calls no
 * allocator of any kind.
 *   a, w, epilogue, out   as for mot_routed_gemm (the same results, bit for bit).
 *   mod                   [T] uint8 device array: 0 = und, 1 = gen.
 *   device_flags          optional device uint32: receives the call's MOT_DEV_* bits once the
 *                         call's work has run on `stream` (NULL: not reported).
 * Limits: 1 <= T <= MOT_NOALLOC_MAX_TOKENS, else MOT_ERR_NOALLOC_LIMIT (above) or
 * MOT_ERR_GEOMETRY (below); other geometry as for mot_routed_gemm.
 * The first call on a device looks up the array's device address (once per device, under a
 * lock); make that first call before any stream capture. All calls on a device share the one
 * array: calls whose work can overlap on the GPU (different streams or host threads) race
 * and must be ordered by the caller.
 */
int mot_routed_gemm_noalloc(const mot_bf16* a, const mot_bf16* w, const uint8_t* mod, int64_t T, int N, int K,
                            int epilogue, mot_bf16* out, uint32_t* device_flags, void* stream);

/*
 * mot_gather_rows -- reorders the rows of a [T][K] bf16 tensor into plan order:
 * dst[i] = src[perm[i]], perm being the plan's row list (und rows ascending, then gen rows).
 * Feeding a routed GEMM with MOT_A_PLAN_ORDER this way reads each row once instead of
 * gathering it for every K block of every output tile when the modality is scattered.
 *   src, dst  [T][K] bf16 device arrays (distinct).   ws  workspace holding the plan for T.
 * Geometry: K a multiple of 8.
 */
int mot_gather_rows(const mot_bf16* src, int64_t T, int K, void* ws, size_t ws_bytes, mot_bf16* dst,
                    void* stream);

/*
 * mot_swiglu_interleave -- one-time layout step for the gate/up weights.
 *   w_gate, w_up  [2][I][K] bf16 device arrays.
 *   w_gu          [2][2I][K] bf16 device array: for each block b of 128 rows,
 *                 rows 256b .. 256b+127 are gate rows 128b .. and rows 256b+128 ..
 *                 256b+255 the matching up rows, so one 256-row GEMM tile holds
 *                 matching gate and up columns.
 * Geometry: I a multiple of 128, K a multiple of 8.
 */
int mot_swiglu_interleave(const mot_bf16* w_gate, const mot_bf16* w_up, int I, int K,
                          mot_bf16* w_gu, void* stream);

/*
 * mot_rope_table_fill_host -- host-side (cos, sin) table for positions 0 .. P-1.
 *   host_cs  host array of P * D/2 * 2 bf16: entry [p][i] = (cos, sin) of the angle
 *            fp32(p) * inv_i (an fp32 product), inv_i = theta^(-2i/D) built in fp64 and
 *            stored in fp32; cos and sin are evaluated in fp64, stored in fp32 and cast to
 *            bf16 ([RFC-435] §3: tables built in FP64, stored in FP32; §2: RoPE in BF16).
 * Geometry: D even, 2 <= D <= 1024; 1 <= P <= MOT_MAX_TOKENS; theta > 1.
 */
int mot_rope_table_fill_host(double theta, int D, int P, mot_bf16* host_cs);

/*
 * mot_rope_table_fill_host_fp32 -- the fp32 table of the FP32 RoPE profile: the same fp32
 * values as mot_rope_table_fill_host before its bf16 cast ([RFC-435] §3: tables built in
 * FP64, stored in FP32).
 *   host_cs  host array of P * D/2 * 2 floats, entry [p][i] = (cos, sin).
 * Geometry and errors as mot_rope_table_fill_host.
 */
int mot_rope_table_fill_host_fp32(double theta, int D, int P, float* host_cs);

/*
 * mot_joint_attention -- attention of packed sequences over the fused QKV output ([RFC-435]
 * §1 Motivation item 2: latent tokens query the prompt KV non-causally at every step; §2
 * Reference hazards: cached prefill needs a bottom-right causal mask; §3 Numerical contract:
 * no split-KV, fixed accumulation order).
 *   qkv   [T][(Hq + 2 Hkv) D] bf16   q heads, k heads, v heads per row (RoPE applied), the
 *                                    output of mot_routed_qkv_norm_rope.
 *   seqs  device int32 [n_seq][5] = (q_start, k_start, nq, nk, n_causal): queries are rows
 *         q_start .. q_start + nq - 1, keys rows k_start .. k_start + nk - 1; the queries are
 *         the last nq key positions (bottom-right alignment). Query row i < n_causal sees keys
 *         j <= nk - nq + i (a prompt row); the others see all nk keys (latent rows). Requires
 *         nk >= 1, 0 <= n_causal <= nq, nk >= nq when n_causal > 0, ranges inside [0, T) and
 *         query ranges of different sequences that do not overlap; otherwise
 *         MOT_DEV_BAD_SEQUENCE is set and the bad sequence's rows are not written.
 *   scale  softmax scale (1 / sqrt(D) for the standard attention), > 0.
 *   ws    at least 64 bytes (e.g. a routing plan); its error word receives device errors.
 *   out   [T][Hq D] bf16   out: rows that are some sequence's query; other rows untouched.
 * Query head h reads KV head h / (Hq / Hkv). Arithmetic: S = Q K^T in fp32 on the tensor
 * cores; per row, 128-key blocks in ascending order from the sequence's first key, with
 * c = scale * log2 e: the reference maximum m starts as the first block's maximum and moves
 * to a later block's maximum only when that exceeds m by more than 8 / c (so p <= 2^8);
 * p = 2^((S - m) c), the difference and the product each rounded to fp32, then CUDA's accurate
 * exp2f (no fused multiply-add, no approximate instruction); l = l alpha + the block's sum of p;
 * O = O alpha + bf16(p) V in fp32 with alpha = 2^((m_old - m) c); out = bf16(O r), r = 1 / l
 * rounded to fp32 once per row. The
 * result depends only on the row's own sequence, not on the other sequences in the pack.
 * D in {64, 128}, Hq a multiple of Hkv.
 */
int mot_joint_attention(const mot_bf16* qkv, int64_t T, int Hq, int Hkv, int D, const int32_t* seqs,
                        int n_seq, float scale, void* ws, size_t ws_bytes, mot_bf16* out, void* stream);

/*
 * mot_routed_gemm_dx -- input gradient of the routed GEMM out = a W[mod]^T through both
 * weight sets ([RFC-435] §3 BAGEL-specific rules: phase A trains only the gen set, but the
 * frozen und operators still need dX; §3 Numerical contract: fixed accumulation order).
 *   dout  [T][N] bf16        gradient of the forward output (rows in token order, or in the
 *                            plan's order with MOT_A_PLAN_ORDER).
 *   w     [2][N][K] bf16     the forward's weights, unchanged (nn.Linear layout).
 *   flags MOT_A_PLAN_ORDER | MOT_OUT_PLAN_ORDER or 0; no epilogue bits.
 *   ws    the routing plan of mod for this T.
 *   dx    [T][K] bf16        out: dx[r][k] = bf16(sum_n dout[r][n] W[mod[r]][n][k]), fp32
 *                            accumulation over n in ascending 64-wide blocks, one cast.
 * The weight is read as the MN-major operand of the same tensor-core pipeline, so no
 * transposed copy is made. Geometry: K a multiple of 256, N a multiple of 64. Errors as
 * mot_routed_gemm.
 */
int mot_routed_gemm_dx(const mot_bf16* dout, const mot_bf16* w, int64_t T, int N, int K, int flags,
                       void* ws, size_t ws_bytes, mot_bf16* dx, void* stream);

/*
 * mot_routed_gemm_dw -- gradient of one weight set of the routed GEMM out = a W[mod]^T
 * ([RFC-435] §3 BAGEL-specific rules: phase A trains the gen set; §3 Numerical contract:
 * fixed accumulation order, no split-K or atomics).
 *   dout      [T][N] bf16    gradient of the forward output: rows in token order, or in the
 *                            plan's order with MOT_A_PLAN_ORDER (mot_gather_rows, or a GEMM run
 *                            with MOT_OUT_PLAN_ORDER).
 *   a         [T][K] bf16    the forward GEMM's input, rows in the same order as dout.
 *   expert    0 (und) or 1 (gen): the weight set whose gradient is formed.
 *   flags     MOT_A_PLAN_ORDER or 0. In token order, each 128-row block of the set whose rows
 *             are consecutive token rows is read with tiled copies; any other block is read in
 *             16-row groups, tiled where the group's rows are consecutive, else by four-row
 *             gathers through the plan. The same bytes reach the tensor cores either way, so
 *             the result is the same bit for bit in both orders.
 *   ws        the routing plan of mod for this T.
 *   dw        [N][K] fp32    out: dw[n][k] = sum over the set's rows r of dout[r][n] a[r][k],
 *                            accumulated in fp32 on the tensor cores over the rows in
 *                            ascending order (blocks of 64, then 16), one accumulator per
 *                            output element, no cast; zeros for a set without rows.
 * Geometry: N and K multiples of 256. A plan for another T sets MOT_DEV_PLAN_MISMATCH; a plan
 * that failed (bad modality) leaves dw undefined. Other errors as mot_routed_gemm.
 */
int mot_routed_gemm_dw(const mot_bf16* dout, const mot_bf16* a, int64_t T, int N, int K,
                       int expert, int flags, void* ws, size_t ws_bytes, float* dw, void* stream);

/*
 * mot_add_rmsnorm_backward -- input gradient of mot_fused_add_rmsnorm ([RFC-435] §3
 * BAGEL-specific rules: the frozen und operators still need dX, so both weight sets take
 * part; [PR-503] gated-norm commit: the backward is assembled from deterministic pieces,
 * a dx kernel and the per-row weight-gradient partials).
 *   dy        [T][H] bf16      gradient of y.
 *   d_res_out [T][H] bf16      gradient reaching res_out (the residual stream), or NULL.
 *   s         [T][H] bf16      the forward's res_out (s = bf16(x + res)).
 *   w         [2][H] bf16      the forward's norm weights.
 *   ws        the routing plan of the forward's mod for this T (mot_route_plan, or the
 *             forward norm's); it selects each row's weight set, and its error word receives
 *             device errors (a plan for another T: MOT_DEV_PLAN_MISMATCH).
 *   dx        [T][H] bf16      out: the gradient of x and of res (s = x + res passes it to both).
 *   rstd      [T] fp32         out: each row's rstd (the forward's).
 *   dw_partials  [H/64][T][64] fp32, or NULL: out: the weight-gradient partials
 *             p[r][j] = dy[r][j] * (s[r][j] * rstd[r]) in blocks of 64 columns, rows in the
 *             plan's order: element (j / 64, i, j % 64) belongs to row perm[i] -- so each weight
 *             set's rows are one contiguous run in ascending order. mot_rmsnorm_dweight folds them.
 *   partial_sets  MOT_SET_UND, MOT_SET_GEN or MOT_SET_BOTH (ignored without dw_partials): the
 *             weight sets whose rows' partials are written; the other rows' entries are left as
 *             they are. Phase A of [RFC-435] §3 trains the gen set only: MOT_SET_GEN writes a
 *             quarter of the bytes on a layer of 3/4 und rows, and every row's dx is still formed.
 * Per row, every operation rounded on its own in fp32: rstd on the forward's fixed tree;
 * xh = s * rstd; g = dy * w[e]; dot = sum of g * xh on the same tree; c = dot / H;
 * dx = bf16(rstd * (g - xh * c) (+ d_res_out)). Geometry as mot_fused_add_rmsnorm; all
 * pointers 16-byte aligned device memory of the stream's device. A plan that failed (bad
 * modality) leaves every output undefined.
 */
int mot_add_rmsnorm_backward(const mot_bf16* dy, const mot_bf16* d_res_out, const mot_bf16* s,
                             const mot_bf16* w, int64_t T, int H, float eps, void* ws, size_t ws_bytes,
                             mot_bf16* dx, float* rstd, float* dw_partials, int partial_sets, void* stream);

/*
 * mot_rmsnorm_dweight -- gradient of the norm weight sets ([PR-503] gated-norm commit:
 * per-row fp32 partials, then the ascending-row fp32 left fold).
 *   dw_partials  [H/64][T][64] fp32  mot_add_rmsnorm_backward's partials (plan order), written
 *             for at least the sets folded here.
 *   sets      MOT_SET_UND, MOT_SET_GEN or MOT_SET_BOTH: the weight sets folded; any other value
 *             is MOT_ERR_ARG.
 *   ws        the same routing plan.
 *   dw        [2][H] fp32      out: dw[e][j] = ((p_r0 + p_r1) + p_r2) + ... over the rows
 *             r0 < r1 < ... of each folded set e; +0 for a set without rows; the rows of the
 *             sets not folded are left as they are.
 * Geometry: 256 <= H <= 8192, H a multiple of 256. Errors as mot_add_rmsnorm_backward.
 */
int mot_rmsnorm_dweight(const float* dw_partials, int64_t T, int H, int sets, void* ws, size_t ws_bytes,
                        float* dw, void* stream);

/*
 * mot_flow_schedule_host -- the sampler's n step times from 1 down to 0 ([RFC-435] §3
 * BAGEL-specific rules: the schedule is built in FP64 and stored in FP32 with the shift s).
 *   host_t  host array of n floats: t_i = float(s u / (1 + (s - 1) u)), u = 1 - i / (n - 1),
 *           evaluated in double; t_0 = 1, t_{n-1} = 0.
 * Geometry: 2 <= n <= 2^20, else MOT_ERR_GEOMETRY; shift finite and > 0, else MOT_ERR_ARG.
 */
int mot_flow_schedule_host(int n, double shift, float* host_t);

/*
 * mot_flow_workspace_bytes -- workspace bytes that mot_cfg_combine_renorm, mot_flow_sde_step
 * and mot_flow_cfg_sde_step need for n_req requests of N elements: the 64-byte header (its error
 * word), 8 bytes per request and segment of 8192 elements (rounded up to 16 bytes), and 4 more
 * per request and segment (rounded up to 16 bytes). 0 for a geometry those calls reject.
 */
size_t mot_flow_workspace_bytes(int n_req, int64_t N);

/*
 * mot_cfg_combine_renorm -- three-branch renormalised classifier-free guidance, per request
 * ([RFC-435] §1 Motivation item 3: up to three branches, two scales, a timestep window and a
 * norm-ratio rescale; §3 BAGEL-specific rules: the window is compared on FP32 t and the
 * renorm reduces over each request alone, never over the packed batch).
 *   v_c, v_tu  [n_req][N] bf16  the conditioned and the text-unconditioned velocities.
 *   v_iu       [n_req][N] bf16  the image-unconditioned velocity, or NULL for two branches.
 *   policy     device fp32 [n_req][6] = (t, s_text, s_img, t_lo, t_hi, renorm_min).
 *   ws         at least mot_flow_workspace_bytes(n_req, N) bytes; everything after its first
 *              64 bytes is scratch that the call overwrites (so not a routing plan in use).
 *   out        [n_req][N] fp32  out.
 * Per request, every operation rounded on its own in fp32: when t_lo <= t <= t_hi,
 * v1 = tu + s_text (c - tu), v2 = iu + s_img (v1 - iu) (v2 = v1 without iu); the sums of c c
 * and v2 v2 over the request on a fixed tree (the request cut into segments of 8192
 * elements; in each, chunks of 8 elements, thread k of 256 summing the chunks q with
 * q % 256 == k in ascending order, an xor butterfly 16, 8, 4, 2, 1 inside each warp and the 8
 * warps folded left to right; the segment sums folded left to right); r = sqrt(ss_c) /
 * sqrt(ss_g) (1 when ss_g is 0), r = min(max(r, renorm_min), 1); out = v2 r. Outside the
 * window out = c. Nothing depends on the other requests of the batch.
 * Geometry: 1 <= n_req <= 65535, N a multiple of 8, 8 <= N <= 2^24, else MOT_ERR_GEOMETRY;
 * all pointers 16-byte aligned device memory of the stream's device.
 */
int mot_cfg_combine_renorm(const mot_bf16* v_c, const mot_bf16* v_tu, const mot_bf16* v_iu, int n_req, int64_t N,
                           const float* policy, void* ws, size_t ws_bytes, float* out, void* stream);

/*
 * mot_flow_sde_step -- one reverse-SDE step of the flow sampler and the log-probability of
 * the transition, per request ([RFC-435] §1 Motivation item 2: the policy log-probability is
 * the ODE-to-SDE transition density; §3 BAGEL-specific rules: FP32, sigma = t,
 * dt = t_i - t_{i+1} > 0, logp summed over all latent elements in a fixed order; §2: training
 * and rollout must produce exactly equal logp).
 *   x, v    [n_req][N] fp32   the latent at t_i and the guided velocity there.
 *   z       [n_req][N] fp32   the step's standard normal noise (drawn by the caller), or NULL
 *                             to score a given x_next instead of sampling one.
 *   x_next  [n_req][N] fp32   out (z given): the latent at t_next; in (z NULL).
 *   times   device fp32 [n_req][2] = (t_i, t_next).
 *   ws      at least mot_flow_workspace_bytes(n_req, N) bytes, scratch after the first 64 as
 *           for mot_cfg_combine_renorm; its error word receives MOT_DEV_BAD_TIME for a request
 *           whose times are not 0 <= t_next < t_i <= 1 (fp32 dt <= 0 included); that
 *           request's outputs are then not written.
 *   logp    device fp32 [n_req]  out.
 * Per element, every operation rounded on its own in fp32: dt = t - t_next, k = (t t) / (2 t),
 * e = x + (1 - t) v, mu = x - dt (v + k e), std = t sqrt(dt), x_next = mu + std z; then
 * d = x_next - mu and ss = the sum of d d on the tree of mot_cfg_combine_renorm;
 * logp = -(ss / (2 (std std))) - N (logf(std) + log sqrt(2 pi)). Scoring the x_next that a
 * sampling call wrote returns that call's logp bit for bit.
 * Geometry: 1 <= n_req <= 65535, N a multiple of 8, 8 <= N <= 2^24, else MOT_ERR_GEOMETRY;
 * all pointers 16-byte aligned device memory of the stream's device.
 */
int mot_flow_sde_step(const float* x, const float* v, const float* z, float* x_next, int n_req, int64_t N,
                      const float* times, void* ws, size_t ws_bytes, float* logp, void* stream);

/*
 * mot_flow_cfg_sde_step -- mot_cfg_combine_renorm followed by mot_flow_sde_step on its output,
 * in one call that does not write the guided velocity to memory and read it back ([RFC-435] §1
 * Motivation items 2 and 3; §3 BAGEL-specific rules as for the two calls: window on FP32 t,
 * renorm per request, SDE and logp in FP32 in a fixed order).
 *   v_c, v_tu, v_iu, policy   as for mot_cfg_combine_renorm (v_iu may be NULL).
 *   x, z, x_next, times       as for mot_flow_sde_step (z NULL: x_next is scored, not sampled).
 *   ws       at least mot_flow_workspace_bytes(n_req, N) bytes, scratch after the first 64; its
 *            error word receives MOT_DEV_BAD_TIME as for mot_flow_sde_step.
 *   v_out    [n_req][N] fp32  out: the guided velocity, or NULL not to write it.
 *   logp     device fp32 [n_req]  out.
 * x_next, logp and v_out are bit for bit those of the two calls in sequence on the same inputs
 * (the same trees, the same order of every fp32 operation). Geometry and alignment as for the
 * two calls; every pointer 16-byte aligned device memory of the stream's device.
 */
int mot_flow_cfg_sde_step(const mot_bf16* v_c, const mot_bf16* v_tu, const mot_bf16* v_iu, const float* policy,
                          const float* x, const float* z, float* x_next, int n_req, int64_t N, const float* times,
                          void* ws, size_t ws_bytes, float* v_out, float* logp, void* stream);

/*
 * mot_flow_noise -- the per-sample standard normal noise of one sampler step ([RFC-435] §3
 * BAGEL-specific rules: initial and transition noise from an explicit per-sample generator with
 * a fixed device, dtype and consumption order).
 *   seeds   device uint64 [n_req]   one seed per request (sample).
 *   step    the step index k (any value; each step draws its own stream).
 *   z       [n_req][N] fp32         out: element 4b + m of request r is word m of the
 *           Philox4x64-10 block (Salmon et al., SC 2011) with counter (b, k, 0, 0) and key
 *           (seeds[r], 0x4D6F54466C6F77), mapped to u = ((x >> 41) + 0.5) 2^-23 (exact fp32 in
 *           (0, 1)); pairs (u_2p, u_2p+1) give z_2p = sqrt(-2 logf(u_2p)) cos(2 pi u_2p+1) and
 *           z_2p+1 = the same radius times sin(2 pi u_2p+1) (sincospif), fp32.
 * A request's noise depends only on its seed, the step and the element index, never on the
 * batch. Geometry: 1 <= n_req <= 65535, N a multiple of 8, 8 <= N <= 2^24; seeds and z 16-byte
 * aligned device memory of the stream's device.
 */
int mot_flow_noise(const uint64_t* seeds, uint64_t step, int n_req, int64_t N, float* z, void* stream);

/*
 * mot_selftest_wait_timeout -- exercises the bounded wait that every pipeline wait of the
 * library uses ([RFC-435] §3: fail closed instead of hanging). One thread waits on an mbarrier
 * that nothing signals; after about one second the wait gives up, MOT_DEV_TIMEOUT is OR-ed into
 * the workspace error word (read it with mot_device_status) and the kernel returns normally,
 * leaving the context usable. No fault, trap or unbounded wait is involved.
 *   ws   device workspace of at least 64 bytes (its error word receives the bit).
 */
int mot_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/*
 * mot_device_status -- synchronizes `stream` and copies the workspace error word
 * (MOT_DEV_* bits, 0 = clean) to *flags.
 */
int mot_device_status(const void* ws, uint32_t* flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOT_H */
