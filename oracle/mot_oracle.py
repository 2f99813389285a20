"""CPU oracle for the Mixture-of-Transformers (MoT) token-routed dense projection.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or executes this
module: only the tests, the smoke check of ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` (including its ``--impl reference`` arm) may use it. It shares no code
with the CUDA library and never reads a value produced by it, except where a function
below says it takes the GPU's own bf16 GEMM output as input ("teacher-forced" stage
checks of the epilogue, which no CPU can reproduce bit for bit after a tensor-core
accumulation).

Sources (web pages; cited by title and section):
  [RFC-435]  "[RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap and integration plan #435"
  [PR-1402]  "[omni, model, ops, ckpt, config, docs] feat: support Bagel in SeedOmni - #1402"
  [PR-503]   "[WS1][CUDA][Qwen3-Next] MoE route/combine contract with a batch-invariant
              grouped expert GEMM (RFC #428 stack 5/8) - #503"

What the path computes ([RFC-435] §1 Motivation, item 1): every GEMM and norm of a packed
batch picks, per token, one of two weight sets -- und (text and ViT tokens, modality 0)
or gen (VAE-latent tokens, modality 1) -- by a fixed index, with no learned router.

Two programs:
  G  -- the fp64 golden. Every quantity is computed in float64; the declared bf16 cast
        points ([RFC-435] §3 Numerical contract: "casts only at declared boundaries") are
        emulated by a direct round-to-nearest-even to bf16. Reductions use any order.
  E  -- the fp32 contract emulator. It restates, in float32 with every operation rounded
        separately (no fused multiply-add), the fixed non-GEMM arithmetic of the kernels:
        the fixed 32-wide chunked reduction trees, the IEEE division and square root, and
        the cast points. It is what the CUDA kernels must match bit for bit.

Inputs are numpy arrays. Floating-point tensors are float64 (G) or float32 (E) arrays
that hold bf16 values exactly; ``mod`` is a uint8 array of 0/1; ``pos`` an int array.
``eps`` is the float32 parameter the kernels receive; both programs use its exact value.

Parity status: every function here is pinned by tests/test_oracle_pins.py (closed forms,
brute force on integer-valued inputs, invariants, hand-derived values in tests/golden/).
"""

from __future__ import annotations

import numpy as np

F32 = np.float32

# Largest finite bf16 value: (2 - 2^-7) * 2^127.
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


# ---------------------------------------------------------------------------
# rounding to bf16
# ---------------------------------------------------------------------------

def bf16(x) -> np.ndarray:
    """Round each value to the nearest bf16 number, ties to even, in one step.

    bf16 keeps 8 significant bits and the float32 exponent range, so the spacing of
    bf16 numbers near |x| in [2^(e-1), 2^e) is 2^(e-8); below the smallest normal
    2^-126 the spacing stays 2^-133. Dividing by that power of two is exact, and numpy's
    ``round`` takes halves to even. Values past the largest finite bf16 after rounding
    become infinities ([PR-503] RMSNorm commit: one round-to-nearest cast at the store).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                                  # x = m * 2^e, 0.5 <= |m| < 1
    quantum = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.round(x / quantum) * quantum
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, x), r)


def bf16_f32(x) -> np.ndarray:
    """bf16 rounding of float32 values, returned as float32 (E's cast)."""
    return bf16(np.asarray(x, dtype=np.float32).astype(np.float64)).astype(F32)


def _eps32(eps: float) -> float:
    return float(F32(eps))


def _check_mod(mod) -> np.ndarray:
    mod = np.asarray(mod)
    if mod.size and (mod.min() < 0 or mod.max() > 1):
        raise ValueError("modality index must be 0 (und) or 1 (gen)")
    return mod.astype(np.int64)


# ---------------------------------------------------------------------------
# G: fp64 golden
# ---------------------------------------------------------------------------

def g_fused_add_rmsnorm(x, res, w, mod, eps):
    """Residual add, then RMSNorm with the row's own weight set.

    [RFC-435] §5 claim order names mot_fused_add_rmsnorm; §1 item 1: the norm picks its
    weight set per token. The RMSNorm convention is the one of [PR-503]'s zero-centred
    RMSNorm commit with offset 0: statistics in fp32 (here fp64), y = x * rstd * w with
    the weight multiply after the upcast and one trailing cast.
      s      = bf16(x + res)                 (the new residual stream, res_out)
      rstd   = 1 / sqrt(sum_j s_j^2 / H + eps)
      y_pre  = s * rstd * w[mod[r]]
      y      = bf16(y_pre)
    Returns a dict with y, y_pre (before the final cast), res_out and rstd.
    """
    mod = _check_mod(mod)
    x = np.asarray(x, np.float64)
    res = np.asarray(res, np.float64)
    w = np.asarray(w, np.float64)
    H = x.shape[1]
    s = bf16(x + res)
    ms = np.sum(s * s, axis=1) / H
    rstd = 1.0 / np.sqrt(ms + _eps32(eps))
    y_pre = s * rstd[:, None] * w[mod]
    return {"y": bf16(y_pre), "y_pre": y_pre, "res_out": s, "rstd": rstd}


def g_routed_matmul(a, w, mod):
    """acc[r, n] = sum_k a[r, k] * w[mod[r], n, k], in float64.

    The routed dense projection: each row is multiplied by the weight set its modality
    selects ([RFC-435] §1 item 1); w is [2][N][K] in the nn.Linear (out, in) layout.
    Each expert's rows go through one plain matmul, so a row's result is by definition
    the dense layer of its own expert ([PR-503] grouped expert GEMM commit: the grouped
    result equals the per-expert GEMM loop).
    """
    mod = _check_mod(mod)
    a = np.asarray(a, np.float64)
    w = np.asarray(w, np.float64)
    acc = np.zeros((a.shape[0], w.shape[1]), np.float64)
    for e in (0, 1):
        rows = np.nonzero(mod == e)[0]
        if rows.size:
            acc[rows] = a[rows] @ w[e].T
    return acc


def g_routed_gemm_cast(a, w, mod):
    """Plain routed projection (O and down projections): out = bf16(acc).

    [PR-1402] "What does this PR do?": MoT routes the O projection per branch (und/gen);
    [RFC-435] §5 names mot_routed_gemm.
    """
    acc = g_routed_matmul(a, w, mod)
    return {"out": bf16(acc), "out_pre": acc}


def rope_inv_freq(theta: float, D: int) -> np.ndarray:
    """inv_i = theta^(-2i/D) for i < D/2, built in fp64 and stored in fp32.

    [RFC-435] §3 BAGEL-specific rules: tables built in FP64, stored in FP32.
    """
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / D).astype(F32)


def rope_cos_sin_f32(theta: float, D: int, pos) -> tuple[np.ndarray, np.ndarray]:
    """fp32 cos/sin of the angle pos * inv_i, for each position and i < D/2.

    The angle is the fp32 product of the position and inv_i; cos and sin are evaluated
    in fp64 of that fp32 angle and stored in fp32 ([RFC-435] §3 BAGEL-specific rules:
    tables built in FP64, stored in FP32). Returns float64 arrays [len(pos)][D/2] holding
    fp32 values.
    """
    inv = rope_inv_freq(theta, D)
    ang = np.asarray(pos).astype(F32)[:, None] * inv[None, :]
    ang64 = ang.astype(np.float64)
    return np.cos(ang64).astype(F32).astype(np.float64), np.sin(ang64).astype(F32).astype(np.float64)


def rope_cos_sin(theta: float, D: int, pos) -> tuple[np.ndarray, np.ndarray]:
    """bf16 cos/sin for the BF16 RoPE profile: the fp32 table values of rope_cos_sin_f32,
    cast to bf16 at the RoPE boundary ([RFC-435] §2 Reference hazards: "QK norm runs in
    FP32, then RoPE and Q/K in BF16"). Returns float64 arrays [len(pos)][D/2] holding bf16
    values.
    """
    c, s = rope_cos_sin_f32(theta, D, pos)
    return bf16(c), bf16(s)


def g_rope_bf16(u, c, s):
    """RoPE in BF16 on a head u[..., D] with the half-split (rotate-half) pairing.

    Element i < D/2 pairs with i + D/2: the rotation partner of element i is -u_{i+D/2}
    for i < D/2 and u_{i-D/2} for i >= D/2; each product and the sum are rounded to bf16
    in turn ([RFC-435] §2 Reference hazards: RoPE and Q/K in BF16).
      out_i = bf16( bf16(u_i * c_i') + bf16(partner_i * s_i') ),  i' = i mod D/2
    Returns (out, pre) with pre the value before the final cast.
    """
    h = u.shape[-1] // 2
    u1, u2 = u[..., :h], u[..., h:]
    pre1 = bf16(u1 * c) + bf16(-u2 * s)
    pre2 = bf16(u2 * c) + bf16(u1 * s)
    pre = np.concatenate([pre1, pre2], axis=-1)
    return bf16(pre), pre


def g_rope_f32(u, c, s):
    """RoPE of the FP32 profile on a head u[..., D]: the rotation of g_rope_bf16 (same
    half-split pairing and direction) evaluated exactly on the unrounded normalized head
    and the fp32 table values, then one bf16 cast.

    [RFC-435] open question 4 (keep the reference BF16 RoPE, or define an FP32 profile):
    the FP32 profile rotates the fp32 normalized q/k and casts once.
      out_i = bf16( u_i * c_i' + partner_i * s_i' ),  i' = i mod D/2
    Returns (out, pre) with pre the value before the cast.
    """
    h = u.shape[-1] // 2
    u1, u2 = u[..., :h], u[..., h:]
    pre = np.concatenate([u1 * c - u2 * s, u2 * c + u1 * s], axis=-1)
    return bf16(pre), pre


def g_rope_exact(u, pos, theta: float, D: int):
    """Cast-free RoPE in fp64 (same pairing and direction as g_rope_bf16).

    Used only by the pins on the rotation itself (norm preservation, relative
    position, complex-multiplication form).
    """
    i = np.arange(D // 2, dtype=np.float64)
    ang = np.asarray(pos, np.float64)[:, None] * np.power(float(theta), -2.0 * i / D)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    h = D // 2
    u1, u2 = u[..., :h], u[..., h:]
    return np.concatenate([u1 * c - u2 * s, u2 * c + u1 * s], axis=-1)


ROPE_PROFILES = ("bf16", "fp32")


def g_qk_norm_rope(q, q_norm, k_norm, pos, mod, Hq, Hkv, D, eps, theta, rope_profile: str = "bf16"):
    """Per-head QK RMSNorm and RoPE on the bf16 GEMM output q (fp64 statistics).

    [RFC-435] §2 Reference hazards: QK norm in FP32 (here fp64), then RoPE and Q/K in BF16.
      Q, K heads:  rstd_head = 1/sqrt(sum q^2 / D + eps)
                   BF16 profile (the reference):  u = bf16(q * rstd_head * g[mod]),
                                                  out = RoPE_bf16(u, bf16 cos, sin of pos)
                   FP32 profile ([RFC-435] open question 4):  u = q * rstd_head * g[mod],
                                                  out = bf16(rotation of u by the fp32 cos, sin)
      V heads:     out = q
    The per-head norm weight g is q_norm or k_norm, [2][D], one vector per expert shared by
    all heads of that kind. Returns out, out_pre (value before the final cast) and u, the
    normalized heads [T][Hq+Hkv][D].
    """
    if rope_profile not in ROPE_PROFILES:
        raise ValueError(f"rope_profile must be one of {ROPE_PROFILES}")
    mod = _check_mod(mod)
    eps = _eps32(eps)
    q = np.asarray(q, np.float64)
    out = q.copy()
    out_pre = q.copy()
    if rope_profile == "bf16":
        c, s = rope_cos_sin(theta, D, pos)
    else:
        c, s = rope_cos_sin_f32(theta, D, pos)
    q_norm = np.asarray(q_norm, np.float64)
    k_norm = np.asarray(k_norm, np.float64)
    us = np.zeros((q.shape[0], Hq + Hkv, D))
    for h in range(Hq + Hkv):
        g = q_norm if h < Hq else k_norm
        cols = slice(h * D, (h + 1) * D)
        qh = q[:, cols]
        ms = np.sum(qh * qh, axis=1) / D
        rstd = 1.0 / np.sqrt(ms + eps)
        if rope_profile == "bf16":
            u = bf16(qh * rstd[:, None] * g[mod])
            o, pre = g_rope_bf16(u, c, s)
        else:
            u = qh * rstd[:, None] * g[mod]
            o, pre = g_rope_f32(u, c, s)
        out[:, cols] = o
        out_pre[:, cols] = pre
        us[:, h] = u
    return {"out": out, "out_pre": out_pre, "u": us}


def g_qkv_norm_rope(y, w_qkv, b_qkv, q_norm, k_norm, pos, mod, Hq, Hkv, D, eps, theta, rope_profile: str = "bf16"):
    """Routed QKV projection, per-head QK RMSNorm in fp32, RoPE and Q/K in BF16.

    [PR-1402] "What does this PR do?": MoT dual-branch routed Q/K/V projections with
    fused qkv_proj_{und,gen} weights, per-head QK RMSNorm and packed RoPE.
      acc  = routed(y, w_qkv) (+ b_qkv[mod] if given)       columns ordered q, k, v heads
      q    = bf16(acc)                                      (GEMM output boundary)
      out  = g_qk_norm_rope(q)                              (BF16 or FP32 RoPE profile)
    For V columns the value before the final cast is acc itself. Returns out, out_pre, q,
    acc and u (the normalized Q/K heads).
    """
    mod = _check_mod(mod)
    acc = g_routed_matmul(y, w_qkv, mod)
    if b_qkv is not None:
        acc = acc + np.asarray(b_qkv, np.float64)[mod]
    q = bf16(acc)
    r = g_qk_norm_rope(q, q_norm, k_norm, pos, mod, Hq, Hkv, D, eps, theta, rope_profile)
    out_pre = r["out_pre"]
    v0 = (Hq + Hkv) * D
    out_pre[:, v0:] = acc[:, v0:]
    return {"out": r["out"], "out_pre": out_pre, "q": q, "acc": acc, "u": r["u"]}


def g_swiglu(acc_gate, acc_up):
    """SiLU(gate) * up with the gate and up GEMM outputs cast to bf16 first.

    [PR-503] grouped expert GEMM commit: gate_up GEMM, then SwiGLU in FP32, one BF16
    cast; the gated-norm commit: SiLU uses the accurate exponential.
      g = bf16(acc_gate), u = bf16(acc_up), h = bf16( g / (1 + exp(-g)) * u )
    """
    g = bf16(acc_gate)
    u = bf16(acc_up)
    pre = g / (1.0 + np.exp(-g)) * u
    return {"h": bf16(pre), "h_pre": pre, "g": g, "u": u}


def g_routed_swiglu(a, w_gate, w_up, mod):
    """Routed gate/up projections followed by the SwiGLU epilogue ([RFC-435] §5 mot_swiglu_mlp)."""
    return g_swiglu(g_routed_matmul(a, w_gate, mod), g_routed_matmul(a, w_up, mod))


def g_layer(x, res, w_norm, w_qkv, b_qkv, q_norm, k_norm, pos, mod, Hq, Hkv, D, eps, theta,
            rope_profile: str = "bf16"):
    """The whole projection step: fused add-RMSNorm, then the routed QKV with norm and RoPE."""
    n = g_fused_add_rmsnorm(x, res, w_norm, mod, eps)
    r = g_qkv_norm_rope(n["y"], w_qkv, b_qkv, q_norm, k_norm, pos, mod, Hq, Hkv, D, eps, theta, rope_profile)
    r.update({"y": n["y"], "y_pre": n["y_pre"], "res_out": n["res_out"]})
    return r


# ---------------------------------------------------------------------------
# E: fp32 contract emulator
# ---------------------------------------------------------------------------

def e_row_tree_sum(terms):
    """Row sums of fp32 terms [T][H] over the fixed 32-wide chunked tree of the add-RMSNorm.

    ([PR-503] zero-centred RMSNorm commit, "On exactness against vLLM": the fixed 32-wide
    chunked sum is what buys batch invariance), defined here as:
      lane l in [0, 32) owns columns 256*j + 8*l + t, j = 0 .. H/256-1, t = 0 .. 7;
      p_l = sequential fp32 sum of its terms from 0.0, j outer, t inner;
      the 32 partials combine by an xor butterfly with offsets 16, 8, 4, 2, 1,
      each step p_l <- p_l + p_(l xor off)  (every lane ends with the same value).
    Returns (sums [T], lane partials after the butterfly [T][32]).
    """
    terms = np.asarray(terms, F32)
    T, H = terms.shape
    if H % 256:
        raise ValueError("the reduction tree is defined for H a multiple of 256")
    lanes = np.arange(32)
    p = np.zeros((T, 32), F32)
    for j in range(H // 256):
        for t in range(8):
            p = p + terms[:, 256 * j + 8 * lanes + t]
    for off in (16, 8, 4, 2, 1):
        p = p + p[:, lanes ^ off]
    return p[:, 0], p


def e_fused_add_rmsnorm(x, res, w, mod, eps, return_stats: bool = False):
    """fp32 restatement of the fused add-RMSNorm with its fixed reduction tree.

    The sum of s^2 runs over e_row_tree_sum's fixed tree. Then ms = p / H (IEEE division),
    rstd = 1 / sqrt(ms + eps) (IEEE sqrt and division), y = bf16((s * rstd) * w[mod]) left
    to right, each operation rounded on its own.
    """
    mod = _check_mod(mod)
    x32 = np.asarray(x, np.float64).astype(F32)
    r32 = np.asarray(res, np.float64).astype(F32)
    w32 = np.asarray(w, np.float64).astype(F32)
    T, H = x32.shape
    if H % 256:
        raise ValueError("the reduction tree is defined for H a multiple of 256")
    s = bf16_f32(x32 + r32)
    ss, p = e_row_tree_sum(s * s)
    ms = ss / F32(H)
    rstd = F32(1.0) / np.sqrt(ms + F32(eps))
    y = bf16_f32((s * rstd[:, None]) * w32[mod])
    out = {"y": y, "res_out": s}
    if return_stats:
        out.update({"ss": ss, "rstd": rstd, "lane_partials": p})
    return out


def e_head_rstd(qh, eps):
    """rstd of one head in fp32 with the head's fixed chunk tree.

    The D values split into 32-wide chunks; each chunk is a sequential fp32 sum of q^2
    from 0.0; the chunk partials are folded left to right ((c0 + c1) + c2) + c3.
    ms = ss / D, rstd = 1 / sqrt(ms + eps).
    """
    T, D = qh.shape
    chunks = []
    for c in range(D // 32):
        acc = np.zeros(T, F32)
        for t in range(32):
            v = qh[:, 32 * c + t]
            acc = acc + v * v
        chunks.append(acc)
    ss = chunks[0]
    for c in chunks[1:]:
        ss = ss + c
    ms = ss / F32(D)
    return F32(1.0) / np.sqrt(ms + F32(eps)), ss


def e_rope_bf16(u, c, s):
    """fp32 restatement of g_rope_bf16 (each product and the sum rounded to bf16)."""
    h = u.shape[-1] // 2
    u1, u2 = u[..., :h], u[..., h:]
    o1 = bf16_f32(bf16_f32(u1 * c) + bf16_f32(-u2 * s))
    o2 = bf16_f32(bf16_f32(u2 * c) + bf16_f32(u1 * s))
    return np.concatenate([o1, o2], axis=-1)


def e_rope_f32(u, c, s):
    """fp32 restatement of g_rope_f32: each product and the sum rounded to fp32 (no fused
    multiply-add), then one bf16 cast.
      out_i = bf16( fp32( fp32(u_i * c) + fp32(partner_i * s) ) )
    """
    h = u.shape[-1] // 2
    u1, u2 = u[..., :h], u[..., h:]
    o1 = bf16_f32((u1 * c) + (-u2 * s))
    o2 = bf16_f32((u2 * c) + (u1 * s))
    return np.concatenate([o1, o2], axis=-1)


def e_qk_norm_rope(q, q_norm, k_norm, cos, sin, mod, Hq, Hkv, D, eps, return_stats: bool = False,
                   rope_profile: str = "bf16"):
    """Teacher-forced epilogue check: per-head QK RMSNorm and RoPE on a given q.

    q is the bf16 GEMM output (float values), [T][(Hq+2Hkv)*D]; cos and sin are the table
    rows of each token's position, [T][D/2] (bf16 values for the BF16 profile, fp32 values
    for the FP32 profile). Q and K heads become RoPE_bf16(bf16((q * rstd) * g[mod])) in the
    BF16 profile and e_rope_f32((q * rstd) * g[mod]) in the FP32 profile; V heads pass
    through unchanged.
    """
    if rope_profile not in ROPE_PROFILES:
        raise ValueError(f"rope_profile must be one of {ROPE_PROFILES}")
    mod = _check_mod(mod)
    q32 = np.asarray(q, np.float64).astype(F32)
    c32 = np.asarray(cos, np.float64).astype(F32)
    s32 = np.asarray(sin, np.float64).astype(F32)
    gq = np.asarray(q_norm, np.float64).astype(F32)
    gk = np.asarray(k_norm, np.float64).astype(F32)
    out = q32.copy()
    stats = []
    us = np.zeros((q32.shape[0], Hq + Hkv, D), F32)
    for h in range(Hq + Hkv):
        g = gq if h < Hq else gk
        cols = slice(h * D, (h + 1) * D)
        qh = q32[:, cols]
        rstd, ss = e_head_rstd(qh, eps)
        if rope_profile == "bf16":
            u = bf16_f32((qh * rstd[:, None]) * g[mod])
            out[:, cols] = e_rope_bf16(u, c32, s32)
        else:
            u = (qh * rstd[:, None]) * g[mod]
            out[:, cols] = e_rope_f32(u, c32, s32)
        stats.append(ss)
        us[:, h] = u
    if return_stats:
        return out, np.stack(stats, axis=1), us
    return out


def e_swiglu(g, u):
    """fp32 SwiGLU on bf16 gate/up values: h = bf16((g / (1 + exp(-g))) * u).

    exp is the host's float32 exponential, so this matches a GPU's expf only to within
    an ulp or two; comparisons against it use a tolerance.
    """
    g32 = np.asarray(g, np.float64).astype(F32)
    u32 = np.asarray(u, np.float64).astype(F32)
    silu = g32 / (F32(1.0) + np.exp(-g32))
    return bf16_f32(silu * u32)


# ---------------------------------------------------------------------------
# Backward of the routed projection path
# ---------------------------------------------------------------------------
#
# [RFC-435] §3 BAGEL-specific rules: phase A trains only the gen expert, but the frozen und
# operators still need dX for marker rows, so dX runs through both weight sets while the
# weight gradient is needed for the gen set. [PR-503] gated-norm commit: the backward is
# assembled from deterministic pieces -- a dx kernel and a weight gradient taken as per-row
# fp32 partials folded in ascending row order. The cast of a forward output to bf16 is
# treated as the identity when differentiating (its gradient is the incoming gradient).

def g_routed_gemm_dx(dout, w, mod):
    """Input gradient of the routed GEMM out = a W[mod]^T, in float64, then one bf16 cast.

      dA[r, k] = sum_n dout[r, n] * w[mod[r], n, k]
    Both weight sets take part (each row through its own). Returns dx and dx_pre.
    """
    mod = _check_mod(mod)
    dout = np.asarray(dout, np.float64)
    w = np.asarray(w, np.float64)
    acc = np.zeros((dout.shape[0], w.shape[2]), np.float64)
    for e in (0, 1):
        rows = np.nonzero(mod == e)[0]
        if rows.size:
            acc[rows] = dout[rows] @ w[e]
    return {"dx": bf16(acc), "dx_pre": acc}


def g_routed_gemm_dw(dout, a, mod, expert: int):
    """Weight gradient of one weight set of the routed GEMM, in float64 (no cast).

      dW[n, k] = sum over rows r with mod[r] = expert of dout[r, n] * a[r, k]
    Rows of the other weight set do not contribute.
    """
    mod = _check_mod(mod)
    dout = np.asarray(dout, np.float64)
    a = np.asarray(a, np.float64)
    rows = np.nonzero(mod == expert)[0]
    return dout[rows].T @ a[rows]


def g_add_rmsnorm_backward(dy, s, w, mod, eps, d_res_out=None):
    """Gradient of the fused add-RMSNorm, in float64.

    Forward (g_fused_add_rmsnorm): s = bf16(x + res), rstd = 1/sqrt(mean(s^2) + eps),
    y_pre = s * rstd * w[mod]. With xh = s * rstd and g = dy * w[mod]:
      ds  = rstd * (g - xh * mean(g * xh))  (+ d_res_out, the gradient reaching res_out)
      dx  = dres = bf16(ds)                 (s = x + res passes ds to both inputs)
      dw[e, j] = sum over rows r with mod[r] = e of dy[r, j] * xh[r, j]
    Returns dx, dx_pre, dw [2][H] and rstd.
    """
    mod = _check_mod(mod)
    dy = np.asarray(dy, np.float64)
    s = np.asarray(s, np.float64)
    w = np.asarray(w, np.float64)
    H = s.shape[1]
    rstd = 1.0 / np.sqrt(np.sum(s * s, axis=1) / H + _eps32(eps))
    xh = s * rstd[:, None]
    g = dy * w[mod]
    c = np.sum(g * xh, axis=1) / H
    ds = rstd[:, None] * (g - xh * c[:, None])
    if d_res_out is not None:
        ds = ds + np.asarray(d_res_out, np.float64)
    dw = np.zeros((2, H))
    for e in (0, 1):
        rows = np.nonzero(mod == e)[0]
        dw[e] = np.sum(dy[rows] * xh[rows], axis=0)
    return {"dx": bf16(ds), "dx_pre": ds, "dw": dw, "rstd": rstd}


def e_left_fold_rows(partials, mod, expert: int):
    """Ascending-row fp32 left fold of per-row partials [T][H] over the rows of one weight
    set ([PR-503] gated-norm commit: per-row fp32 dweight rows, then an ascending-row fp32
    left fold): ((p_r0 + p_r1) + p_r2) + ... for r0 < r1 < r2 < ... with mod[r] = expert.
    The fold starts from the first row's partial; no rows give zeros.
    """
    mod = _check_mod(mod)
    partials = np.asarray(partials, F32)
    rows = np.nonzero(mod == expert)[0]
    if rows.size == 0:
        return np.zeros(partials.shape[1], F32)
    acc = partials[rows[0]].copy()
    for r in rows[1:]:
        acc = acc + partials[r]
    return acc


def e_add_rmsnorm_backward(dy, s, w, mod, eps, d_res_out=None):
    """fp32 restatement of g_add_rmsnorm_backward, every operation rounded on its own.

      rstd   as in the forward (e_row_tree_sum of s^2, IEEE division and square root)
      xh_j   = s_j * rstd
      g_j    = dy_j * w[mod]_j
      dot    = e_row_tree_sum of g_j * xh_j      (the forward's fixed tree)
      c      = dot / H
      ds_j   = rstd * (g_j - xh_j * c)           (+ d_res_out_j)
      dx_j   = bf16(ds_j)
      p_r[j] = dy_j * xh_j,  dw[e] = e_left_fold_rows(p, mod, e)
    Returns dx, dw [2][H] (fp32), rstd and dot.
    """
    mod = _check_mod(mod)
    dy32 = np.asarray(dy, np.float64).astype(F32)
    s32 = np.asarray(s, np.float64).astype(F32)
    w32 = np.asarray(w, np.float64).astype(F32)
    T, H = s32.shape
    ss, _ = e_row_tree_sum(s32 * s32)
    rstd = F32(1.0) / np.sqrt(ss / F32(H) + F32(eps))
    xh = s32 * rstd[:, None]
    g = dy32 * w32[mod]
    dot, _ = e_row_tree_sum(g * xh)
    c = dot / F32(H)
    ds = rstd[:, None] * (g - xh * c[:, None])
    if d_res_out is not None:
        ds = ds + np.asarray(d_res_out, np.float64).astype(F32)
    p = dy32 * xh
    dw = np.stack([e_left_fold_rows(p, mod, 0), e_left_fold_rows(p, mod, 1)])
    return {"dx": bf16_f32(ds), "dw": dw, "rstd": rstd, "dot": dot}


# ---------------------------------------------------------------------------
# Joint attention of the packed sequences
# ---------------------------------------------------------------------------
#
# [RFC-435] §1 Motivation item 2: latent tokens query the prompt KV non-causally at every
# step; §2 Reference hazards: cached prefill needs a bottom-right causal mask (a top-left
# aligned causal mask is wrong when the queries are the last rows of a longer key range);
# §3 Numerical contract: no split-KV. The pages give no formula beyond that; the attention
# is the textbook scaled dot-product softmax attention with grouped KV heads.

def g_joint_attention(qkv, seqs, Hq: int, Hkv: int, D: int, scale: float | None = None):
    """Attention over packed sequences, in float64, one bf16 cast.

    qkv   [T][(Hq + 2 Hkv) D]: per row the q heads, then k heads, then v heads (the fused QKV
          output after QK-norm and RoPE). Query head h reads KV head h // (Hq / Hkv).
    seqs  rows (q_start, k_start, nq, nk, n_causal): the sequence's queries are rows
          q_start .. q_start + nq - 1 and its keys rows k_start .. k_start + nk - 1; the
          queries are the last nq key positions (bottom-right alignment), so query i sits at
          key position nk - nq + i. Query rows i < n_causal are causal: they see keys
          j <= nk - nq + i. The other query rows see all nk keys (latent rows).
    scale defaults to 1 / sqrt(D).
    Returns out [T][Hq D] (bf16 values; rows that are no sequence's query are 0) and out_pre.
    """
    qkv = np.asarray(qkv, np.float64)
    T = qkv.shape[0]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    grp = Hq // Hkv
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    out = np.zeros((T, Hq * D))
    for q0, k0, nq, nk, nc in np.asarray(seqs, np.int64):
        if nq < 0 or nk < 1 or not 0 <= nc <= nq or (nc > 0 and nk < nq):
            raise ValueError("bad sequence descriptor")
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        allowed = np.where(i < nc, j <= nk - nq + i, True)
        for h in range(Hq):
            g = h // grp
            q = qkv[q0:q0 + nq, h * D:(h + 1) * D]
            k = qkv[k0:k0 + nk, (Hq + g) * D:(Hq + g + 1) * D]
            v = qkv[k0:k0 + nk, (Hq + Hkv + g) * D:(Hq + Hkv + g + 1) * D]
            s = (q @ k.T) * sc
            s = np.where(allowed, s, -np.inf)
            m = np.max(s, axis=1, keepdims=True)
            p = np.exp(s - m)
            p = p / np.sum(p, axis=1, keepdims=True)
            out[q0:q0 + nq, h * D:(h + 1) * D] = p @ v
    return {"out": bf16(out), "out_pre": out}


# ---------------------------------------------------------------------------
# Flow-matching sampler pieces: schedule, three-branch renormalised CFG, SDE step and logp
# ---------------------------------------------------------------------------
#
# [RFC-435] §1 Motivation items 2 and 3 (the policy log-probability is the ODE-to-SDE transition
# density; three-branch renormalised CFG with two scales, a timestep window and a norm-ratio
# rescale) and §3 BAGEL-specific rules (schedule built in FP64 and stored in FP32 with the shift
# s; SDE step and logp in FP32 with sigma = t and dt = t_i - t_{i+1} > 0; logp summed over all
# latent elements in a fixed order; the CFG window compared on FP32 t; renorm per request).
# The pages give no formulas: the readings are the rectified-flow path x_t = (1 - t) x_0 + t eps
# (t = 1 is noise), velocity v = eps - x_0, the marginal-preserving reverse SDE, and CFG as
# successive interpolations; each is stated in its docstring.

LOG_SQRT_2PI = 0.5 * np.log(2.0 * np.pi)


def flow_schedule(n: int, shift: float) -> np.ndarray:
    """n times from 1 to 0 (n - 1 steps): t_i = s u / (1 + (s - 1) u) with u = 1 - i/(n-1),
    built in float64 and stored in float32 ([RFC-435] §3: schedule built in FP64, stored and
    traced in FP32; the shift s comes from the run config)."""
    u = 1.0 - np.arange(n, dtype=np.float64) / (n - 1)
    return (shift * u / (1.0 + (shift - 1.0) * u)).astype(F32)


def cfg_guided(t, t_lo, t_hi) -> bool:
    """Whether step time t lies in the CFG window, compared on fp32 values."""
    return bool(F32(t_lo) <= F32(t) <= F32(t_hi))


def g_cfg_combine_renorm(v_c, v_tu, v_iu, t, s_text, s_img, t_lo, t_hi, renorm_min):
    """Three-branch renormalised CFG of one request, in float64.

    v_c: the fully conditioned velocity; v_tu: text-unconditioned; v_iu: image-unconditioned
    or None (two branches). Inside the window:
      v1 = v_tu + s_text (v_c - v_tu);  v2 = v_iu + s_img (v1 - v_iu) (or v1);
      r  = clamp(||v_c|| / ||v2||, renorm_min, 1) over all the request's elements (1 if v2 = 0);
      v  = v2 r.
    Outside the window v = v_c.
    """
    v_c = np.asarray(v_c, np.float64)
    if not cfg_guided(t, t_lo, t_hi):
        return v_c.copy()
    v1 = np.asarray(v_tu, np.float64) + float(F32(s_text)) * (v_c - np.asarray(v_tu, np.float64))
    if v_iu is not None:
        v_iu = np.asarray(v_iu, np.float64)
        v2 = v_iu + float(F32(s_img)) * (v1 - v_iu)
    else:
        v2 = v1
    ng = np.sqrt(np.sum(v2 * v2))
    r = 1.0 if ng == 0 else np.sqrt(np.sum(v_c * v_c)) / ng
    r = min(max(r, float(F32(renorm_min))), 1.0)
    return v2 * r


def g_flow_sde_step(x, v, z, t_i, t_next, x_next=None):
    """One SDE step from t_i down to t_next and its log-probability, in float64.

    sigma = t_i, dt = t_i - t_next > 0. With eps_hat = x + (1 - t) v (the noise the velocity
    implies) and the score -eps_hat / t, the reverse SDE that keeps the marginals of
    dx/dt = v steps to
      mu = x - dt (v + sigma^2 / (2 t) eps_hat),   std = sigma sqrt(dt),   x_next = mu + std z,
    and logp = sum over the latent elements of log N(x_next; mu, std^2).
    With z None the step is evaluated, not taken: x_next is given (the latent a rollout stored)
    and only logp depends on it, so training scores the rollout's transition.
    """
    t = float(F32(t_i))
    dt = t - float(F32(t_next))
    if not dt > 0:
        raise ValueError("dt must be positive")
    x = np.asarray(x, np.float64)
    v = np.asarray(v, np.float64)
    sigma = t
    eps_hat = x + (1.0 - t) * v
    mu = x - dt * (v + sigma * sigma / (2.0 * t) * eps_hat)
    std = sigma * np.sqrt(dt)
    if z is None:
        x_next = np.asarray(x_next, np.float64)
    else:
        x_next = mu + std * np.asarray(z, np.float64)
    d = x_next - mu
    logp = -np.sum(d * d) / (2.0 * std * std) - x.size * (np.log(std) + LOG_SQRT_2PI)
    return {"x_next": x_next, "mu": mu, "std": std, "logp": logp}


FLOW_SEGMENT = 8192  # elements per segment of the request tree


def e_request_tree_sum(terms):
    """Sum of the fp32 terms of one request on the fixed tree of the flow kernels. The request's
    elements are cut into segments of FLOW_SEGMENT (the last may be shorter); each segment is
    summed on its own: elements in chunks of 8, thread tau of 256 owns the segment's chunks q
    with q % 256 == tau, summing them in ascending order (the chunk's 8 elements in order) from
    0.0; within each warp of 32 threads an xor butterfly with offsets 16, 8, 4, 2, 1; then the 8
    warps' sums folded left to right. The segment sums are then folded left to right. The order
    depends only on the request's own length, never on the batch around it."""
    terms = np.asarray(terms, F32).reshape(-1)
    if terms.size % 8 or terms.size == 0:
        raise ValueError("the tree is defined for a positive multiple of 8 elements")
    lanes = np.arange(32)
    seg_sums = []
    for s0 in range(0, terms.size, FLOW_SEGMENT):
        chunks = terms[s0:s0 + FLOW_SEGMENT].reshape(-1, 8)
        p = np.zeros(256, F32)
        for q in range(chunks.shape[0]):
            tau = q % 256
            for u in range(8):
                p[tau] = p[tau] + chunks[q, u]
        w = p.reshape(8, 32)
        for off in (16, 8, 4, 2, 1):
            w = w + w[:, lanes ^ off]
        acc = w[0, 0]
        for k in range(1, 8):
            acc = acc + w[k, 0]
        seg_sums.append(F32(acc))
    total = seg_sums[0]
    for v in seg_sums[1:]:
        total = total + v
    return F32(total)


def e_cfg_combine_renorm(v_c, v_tu, v_iu, t, s_text, s_img, t_lo, t_hi, renorm_min):
    """fp32 restatement of g_cfg_combine_renorm, each operation rounded on its own:
    v1 = tu + s_text (c - tu), v2 = iu + s_img (v1 - iu); the sums of squares of c and v2 on
    e_request_tree_sum; r = sqrt(ss_c) / sqrt(ss_g) (1 if ss_g is 0), then max with renorm_min
    and min with 1; v = v2 r. Outside the window v = c."""
    c = np.asarray(v_c, np.float64).astype(F32)
    if not cfg_guided(t, t_lo, t_hi):
        return c.copy()
    tu = np.asarray(v_tu, np.float64).astype(F32)
    v1 = tu + F32(s_text) * (c - tu)
    if v_iu is not None:
        iu = np.asarray(v_iu, np.float64).astype(F32)
        v2 = iu + F32(s_img) * (v1 - iu)
    else:
        v2 = v1
    ss_c = e_request_tree_sum(c * c)
    ss_g = e_request_tree_sum(v2 * v2)
    r = F32(1.0) if ss_g == 0 else np.sqrt(ss_c) / np.sqrt(ss_g)
    r = min(max(r, F32(renorm_min)), F32(1.0))
    return v2 * F32(r)


def e_flow_sde_step(x, v, z, t_i, t_next, x_next=None):
    """fp32 restatement of g_flow_sde_step, each operation rounded on its own:
    dt = t - t_next, k = (sigma sigma) / (2 t), e = x + (1 - t) v, mu = x - dt (v + k e),
    std = sigma sqrt(dt), x_next = mu + std z (or the given x_next when z is None);
    d = x_next - mu, ss = e_request_tree_sum(d d),
    logp = -(ss / (2 std std)) - N (log(std) + log sqrt(2 pi)) with the host's fp32 log (the
    GPU's logf may differ in the last bit, so logp is compared within a tolerance)."""
    t = F32(t_i)
    dt = t - F32(t_next)
    sigma = t
    k = (sigma * sigma) / (F32(2.0) * t)
    x32 = np.asarray(x, np.float64).astype(F32)
    v32 = np.asarray(v, np.float64).astype(F32)
    e = x32 + (F32(1.0) - t) * v32
    mu = x32 - dt * (v32 + k * e)
    std = sigma * np.sqrt(dt)
    if z is None:
        x_next = np.asarray(x_next, np.float64).astype(F32)
    else:
        x_next = mu + std * np.asarray(z, np.float64).astype(F32)
    d = x_next - mu
    ss = e_request_tree_sum(d * d)
    a = ss / (F32(2.0) * (std * std))
    logp = -a - F32(x32.size) * (np.log(std) + F32(LOG_SQRT_2PI))
    return {"x_next": x_next, "mu": mu, "std": std, "logp": F32(logp)}


# ---------------------------------------------------------------------------
# Per-sample transition noise: a counter-based generator (Philox4x64-10) and Box-Muller
# ---------------------------------------------------------------------------
#
# [RFC-435] §3 BAGEL-specific rules: initial and transition noise come from an explicit
# per-sample generator with a fixed device, dtype and consumption order. Reading: the noise of
# request r at step k is a pure function of (seed_r, k, element index), so it does not depend on
# the batch, the device count or the order of the calls. The generator is Philox4x64-10 as
# published by Salmon, Moraes, Dror and Shaw ("Parallel random numbers: as easy as 1, 2, 3",
# SC 2011): ten rounds of two 64 x 64 -> 128-bit products with the round keys bumped by the
# Weyl constants; the normal deviates come from the Box-Muller transform.

PHILOX_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)   # round multipliers
PHILOX_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)   # key increments (golden ratio, sqrt(3) - 1)
NOISE_DOMAIN = 0x4D6F54466C6F77                       # second key word: "MoTFlow" in ASCII
_M64 = (1 << 64) - 1


def philox4x64_10(ctr, key):
    """One Philox4x64 block with 10 rounds: counter (x0, x1, x2, x3) and key (k0, k1) are
    64-bit integers. Each round multiplies x0 and x2 by the two multipliers into 128-bit
    products and forms (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)); the key
    words then grow by the two Weyl constants (mod 2^64)."""
    x0, x1, x2, x3 = (int(v) & _M64 for v in ctr)
    k0, k1 = (int(v) & _M64 for v in key)
    for _ in range(10):
        p0 = PHILOX_M[0] * x0
        p1 = PHILOX_M[1] * x2
        x0, x1, x2, x3 = (p1 >> 64) ^ x1 ^ k0, p1 & _M64, (p0 >> 64) ^ x3 ^ k1, p0 & _M64
        k0 = (k0 + PHILOX_W[0]) & _M64
        k1 = (k1 + PHILOX_W[1]) & _M64
    return (x0, x1, x2, x3)


def noise_uniform(x):
    """The top 23 bits of a 64-bit word as a uniform in (0, 1): ((x >> 41) + 0.5) 2^-23, exact
    in fp32 (at most 24 significant bits) and never 0 or 1."""
    return F32(((int(x) >> 41) + 0.5) * 2.0 ** -23)


def flow_noise_uniforms(seed, step, N):
    """The N uniforms of one request at one step, fp32: element 4b + m takes word m of
    philox4x64_10(counter = (b, step, 0, 0), key = (seed, NOISE_DOMAIN))."""
    if N % 4:
        raise ValueError("N must be a multiple of 4")
    u = np.empty(N, F32)
    for b in range(N // 4):
        words = philox4x64_10((b, step, 0, 0), (seed, NOISE_DOMAIN))
        for m in range(4):
            u[4 * b + m] = noise_uniform(words[m])
    return u


def g_flow_noise(seeds, step, N):
    """Standard normal transition noise z [n_req][N], fp64: Box-Muller on the uniforms of each
    request, pairs (u_{2p}, u_{2p+1}) giving z_{2p} = sqrt(-2 ln u_{2p}) cos(2 pi u_{2p+1}) and
    z_{2p+1} = sqrt(-2 ln u_{2p}) sin(2 pi u_{2p+1})."""
    out = np.empty((len(seeds), N), np.float64)
    for r, seed in enumerate(seeds):
        u = flow_noise_uniforms(int(seed), int(step), N).astype(np.float64)
        rad = np.sqrt(-2.0 * np.log(u[0::2]))
        ang = 2.0 * np.pi * u[1::2]
        out[r, 0::2] = rad * np.cos(ang)
        out[r, 1::2] = rad * np.sin(ang)
    return out

