"""Pins of the CPU oracle against facts outside itself (no GPU).

Each test checks the oracle against something it does not compute itself: a library
routine for bf16 rounding, hand-derived values (tests/golden/hand_values.json), closed
forms, brute force on integer-valued inputs where every sum is exact, and invariants
of the mathematics (scale invariance of RMSNorm, RoPE as a complex rotation). The
inputs are chosen so that a plausible slip in the oracle -- a dropped term, a wrong
sign or index, a transposed operand, a wrong expert, a different reduction order --
fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mot_oracle as O

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_values.json")))
F32 = np.float32


def _hex(s):
    return float("inf") if s == "inf" else float.fromhex(s)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def test_bf16_hand_cases():
    for c in GOLDEN["bf16_round"]["cases"]:
        got = O.bf16(np.array([_hex(c["x"])]))[0]
        exp = _hex(c["expected"])
        assert got == exp, (c, got)
        assert math.copysign(1.0, got) == math.copysign(1.0, exp)


def test_bf16_matches_torch_on_float32_values():
    # torch's float32 -> bf16 conversion is an independent round-to-nearest-even.
    rng = np.random.default_rng(7)
    a = rng.standard_normal(200_000).astype(F32) * F32(3.0)
    b = np.ldexp(rng.standard_normal(20_000).astype(F32), rng.integers(-140, 120, 20_000)).astype(F32)
    bits = rng.integers(0, 2**16, 20_000).astype(np.uint32)
    ties = ((bits << 16) | 0x8000).view(F32)              # exact half-way cases
    ties = ties[np.isfinite(ties)]
    v = np.concatenate([a, b, ties, np.array([0.0, -0.0, 1e-45, -1e-45], F32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.bf16(v.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


# ---------------------------------------------------------------------------
# fused add-RMSNorm
# ---------------------------------------------------------------------------

def test_add_rmsnorm_constant_row_closed_form():
    gd = GOLDEN["add_rmsnorm_constant_row"]
    H = gd["H"]
    eps = _hex(gd["eps"])
    assert eps == float(F32(1e-6))
    w = np.stack([np.full(H, 0.75), np.full(H, 1.25)])
    for case in gd["cases"]:
        c = _hex(case["c"])
        ratio = _hex(case["c_over_rms"])
        x = np.full((2, H), c)
        res = np.zeros((2, H))
        mod = np.array([0, 1])
        g = O.g_fused_add_rmsnorm(x, res, w, mod, 1e-6)
        np.testing.assert_allclose(g["y_pre"][0], 0.75 * ratio, rtol=1e-15)
        np.testing.assert_allclose(g["y_pre"][1], 1.25 * ratio, rtol=1e-15)
        np.testing.assert_array_equal(g["res_out"], x)
        e = O.e_fused_add_rmsnorm(x, res, w, mod, 1e-6)
        # fp32 statistics: within one bf16 step of the closed form
        for r, wr in ((0, 0.75), (1, 1.25)):
            step = 2.0 ** (math.frexp(wr * ratio)[1] - 8)
            assert np.all(np.abs(e["y"][r] - wr * ratio) <= step), (c, e["y"][r][:4])


def test_add_rmsnorm_residual_is_rounded_sum():
    # res_out = bf16(x + res): 1 + 2^-9 is a tie that rounds to 1, 1 + 3*2^-9 rounds up.
    H = 256
    x = np.zeros((1, H))
    res = np.zeros((1, H))
    x[0, 0], res[0, 0] = 1.0, 2.0 ** -9
    x[0, 1], res[0, 1] = 1.0, 3 * 2.0 ** -9
    x[0, 2], res[0, 2] = 0.5, 0.25
    w = np.ones((2, H))
    for out in (O.g_fused_add_rmsnorm(x, res, w, [0], 1e-6), O.e_fused_add_rmsnorm(x, res, w, [0], 1e-6)):
        assert out["res_out"][0, 0] == 1.0
        assert out["res_out"][0, 1] == 1.0 + 2.0 ** -7
        assert out["res_out"][0, 2] == 0.75


def test_add_rmsnorm_scale_invariance_bitwise():
    # With eps = 0, scaling a row by a power of two leaves RMSNorm unchanged, exactly.
    rng = np.random.default_rng(3)
    T, H = 8, 512
    s = O.bf16(rng.standard_normal((T, H)))
    w = O.bf16(1.0 + 0.1 * rng.standard_normal((2, H)))
    mod = np.array([0, 1] * 4)
    zero = np.zeros((T, H))
    for k in (-6, 3, 9):
        for fn in (O.g_fused_add_rmsnorm, O.e_fused_add_rmsnorm):
            a = fn(s, zero, w, mod, 0.0)["y"]
            b = fn(s * 2.0 ** k, zero, w, mod, 0.0)["y"]
            np.testing.assert_array_equal(a, b)


def test_add_rmsnorm_routes_weight_set_per_row():
    # Expert weights 1 and 2: gen rows are exactly twice the und rows (x2 is exact in bf16).
    rng = np.random.default_rng(4)
    H = 256
    s = O.bf16(rng.standard_normal((1, H)))
    x = np.repeat(s, 4, axis=0)
    w = np.stack([np.ones(H), 2 * np.ones(H)])
    mod = np.array([1, 0, 0, 1])
    for fn in (O.g_fused_add_rmsnorm, O.e_fused_add_rmsnorm):
        y = fn(x, np.zeros_like(x), w, mod, 1e-6)["y"]
        np.testing.assert_array_equal(y[0], 2 * y[1])
        np.testing.assert_array_equal(y[3], 2 * y[2])
        np.testing.assert_array_equal(y[1], y[2])


def test_add_rmsnorm_e_tree_order_hand_values():
    gd = GOLDEN["add_rmsnorm_tree_sum"]
    H = 512
    x = np.zeros((2, H))
    x[0, 0] = 4096.0
    x[0, 1:8] = 1.0
    for lane in range(1, 32):
        x[0, 8 * lane] = 1.0
    x[1, 0:8] = 1.0
    x[1, 256] = 4096.0
    e = O.e_fused_add_rmsnorm(x, np.zeros_like(x), np.ones((2, H)), [0, 0], 1e-6, return_stats=True)
    assert e["ss"][0] == gd["row_A_sum_of_squares"]
    assert e["ss"][1] == gd["row_B_sum_of_squares"]
    # every lane of the butterfly holds the same total
    assert np.all(e["lane_partials"][0] == e["lane_partials"][0, 0])


def test_add_rmsnorm_e_within_half_step_of_g():
    rng = np.random.default_rng(5)
    T, H = 64, 768
    x = O.bf16(rng.standard_normal((T, H)))
    res = O.bf16(rng.standard_normal((T, H)))
    w = O.bf16(1 + 0.1 * rng.standard_normal((2, H)))
    mod = rng.integers(0, 2, T)
    g = O.g_fused_add_rmsnorm(x, res, w, mod, 1e-6)
    e = O.e_fused_add_rmsnorm(x, res, w, mod, 1e-6)
    np.testing.assert_array_equal(e["res_out"], g["res_out"])
    _, ex = np.frexp(g["y_pre"])
    half = np.ldexp(1.0, ex - 9)
    assert np.all(np.abs(e["y"] - g["y_pre"]) <= half * (1 + 1e-5) + 1e-30)


# ---------------------------------------------------------------------------
# routed GEMM
# ---------------------------------------------------------------------------

def _brute_routed(a, w, mod):
    T, K = a.shape
    N = w.shape[1]
    out = [[0 for _ in range(N)] for _ in range(T)]
    for r in range(T):
        for n in range(N):
            acc = 0
            for k in range(K):
                acc += int(a[r][k]) * int(w[mod[r]][n][k])
            out[r][n] = acc
    return np.array(out, dtype=np.float64)


def test_routed_matmul_brute_force_integers():
    # Integer values: every product and sum is exact, so the result is unique.
    rng = np.random.default_rng(11)
    T, K, N = 7, 5, 3                 # non-square: a transposed operand cannot pass
    a = rng.integers(-4, 5, (T, K))
    w = rng.integers(-3, 4, (2, N, K))
    mod = np.array([0, 1, 1, 0, 1, 0, 0])
    np.testing.assert_array_equal(O.g_routed_matmul(a, w, mod), _brute_routed(a, w, mod))
    out = O.g_routed_gemm_cast(a, w, mod)
    np.testing.assert_array_equal(out["out"], _brute_routed(a, w, mod))


def test_routed_matmul_single_modality_is_dense():
    rng = np.random.default_rng(12)
    a = rng.integers(-4, 5, (6, 4))
    w = rng.integers(-3, 4, (2, 5, 4))
    for e in (0, 1):
        mod = np.full(6, e)
        dense = np.array([[sum(int(a[r, k]) * int(w[e, n, k]) for k in range(4)) for n in range(5)]
                          for r in range(6)], dtype=np.float64)
        np.testing.assert_array_equal(O.g_routed_matmul(a, w, mod), dense)


def test_routed_rows_depend_only_on_themselves():
    rng = np.random.default_rng(13)
    a = rng.integers(-50, 51, (9, 8)).astype(np.float64)      # exact sums in any order
    w = rng.integers(-50, 51, (2, 6, 8)).astype(np.float64)
    mod = rng.integers(0, 2, 9)
    full = O.g_routed_matmul(a, w, mod)
    for r in range(9):
        one = O.g_routed_matmul(a[r:r + 1], w, mod[r:r + 1])
        np.testing.assert_array_equal(one[0], full[r])


def test_modality_out_of_range_rejected():
    with pytest.raises(ValueError):
        O.g_routed_matmul(np.ones((2, 2)), np.ones((2, 2, 2)), [0, 2])


# ---------------------------------------------------------------------------
# QK norm and RoPE
# ---------------------------------------------------------------------------

def _onehot_qkv(c_q, c_k, Hq, Hkv, D):
    """y = e_0 and W[:, n, 0] = c: the GEMM output of every Q (K) column is exactly c_q (c_k)."""
    N = (Hq + 2 * Hkv) * D
    w = np.zeros((2, N, 64))
    w[:, : Hq * D, 0] = c_q
    w[:, Hq * D: (Hq + Hkv) * D, 0] = c_k
    w[:, (Hq + Hkv) * D:, 0] = 0.5
    y = np.zeros((2, 64))
    y[:, 0] = 1.0
    return y, w


@pytest.mark.parametrize("profile", ["bf16", "fp32"])
@pytest.mark.parametrize("c_q,c_k", [(1.5, -3.0), (2.0 ** -10, -(2.0 ** -11))])
def test_qk_norm_constant_head_closed_form_at_position_zero(c_q, c_k, profile):
    # A head of equal values c normalizes to g * c / sqrt(c^2 + eps); small c makes eps visible.
    Hq, Hkv, D = 2, 1, 128
    eps = float(F32(1e-6))
    y, w = _onehot_qkv(c_q, c_k, Hq, Hkv, D)
    qn = np.stack([np.full(D, 0.75), np.full(D, 1.25)])
    kn = np.stack([np.full(D, 1.5), np.full(D, 0.5)])
    mod = np.array([0, 1])
    g = O.g_qkv_norm_rope(y, w, None, qn, kn, np.array([0, 0]), mod, Hq, Hkv, D, 1e-6, 1e6, rope_profile=profile)
    table = O.rope_cos_sin if profile == "bf16" else O.rope_cos_sin_f32
    c, s = table(1e6, D, np.array([0, 0]))
    e_out = O.e_qk_norm_rope(g["q"], qn, kn, c, s, mod, Hq, Hkv, D, 1e-6, rope_profile=profile)
    for r, e in ((0, 0), (1, 1)):
        qv = O.bf16(qn[e, 0] * c_q / math.sqrt(c_q * c_q + eps))
        kv = O.bf16(kn[e, 0] * c_k / math.sqrt(c_k * c_k + eps))
        for out in (g["out"], e_out):
            assert np.all(out[r, : Hq * D] == qv)
            assert np.all(out[r, Hq * D: (Hq + Hkv) * D] == kv)
            assert np.all(out[r, (Hq + Hkv) * D:] == 0.5)       # V passes through


def test_qk_norm_scale_invariance_and_bias():
    rng = np.random.default_rng(21)
    Hq, Hkv, D, T = 2, 1, 64, 6
    N = (Hq + 2 * Hkv) * D
    y = O.bf16(rng.standard_normal((T, 128)))
    w = O.bf16(0.05 * rng.standard_normal((2, N, 128)))
    qn = O.bf16(1 + 0.1 * rng.standard_normal((2, D)))
    kn = O.bf16(1 + 0.1 * rng.standard_normal((2, D)))
    mod = rng.integers(0, 2, T)
    pos = rng.integers(0, 1000, T)
    a = O.g_qkv_norm_rope(y, w, None, qn, kn, pos, mod, Hq, Hkv, D, 0.0, 1e6)
    b = O.g_qkv_norm_rope(y * 8.0, w, None, qn, kn, pos, mod, Hq, Hkv, D, 0.0, 1e6)
    np.testing.assert_array_equal(a["out"][:, : (Hq + Hkv) * D], b["out"][:, : (Hq + Hkv) * D])
    np.testing.assert_array_equal(a["out"][:, (Hq + Hkv) * D:] * 8.0, b["out"][:, (Hq + Hkv) * D:])
    # a bias of the row's own expert is added before the cast
    bias = O.bf16(rng.standard_normal((2, N)))
    c = O.g_qkv_norm_rope(y, w, bias, qn, kn, pos, mod, Hq, Hkv, D, 1e-6, 1e6)
    np.testing.assert_array_equal(c["acc"], a["acc"] + bias[mod])


def test_qk_head_tree_order_hand_value():
    gd = GOLDEN["qk_head_tree_sum"]
    D = 128
    q = np.zeros((1, 3 * D))
    q[0, 0] = 4096.0
    q[0, 1:32] = 1.0
    q[0, 32] = 1.0
    q[0, 64] = 1.0
    q[0, 96:98] = 1.0
    cs = np.ones((1, D // 2)), np.zeros((1, D // 2))
    _, ss, _ = O.e_qk_norm_rope(q, np.ones((2, D)), np.ones((2, D)), cs[0], cs[1], [0], 1, 1, D, 1e-6,
                                return_stats=True)
    assert ss[0, 0] == gd["sum_of_squares"]


def test_rope_table_hand_values():
    gd = GOLDEN["rope"]
    c, s = O.rope_cos_sin(1e6, 128, np.array([0, 1]))
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    assert c[1, 0] == gd["pos1_i0_cos"] and s[1, 0] == gd["pos1_i0_sin"]
    inv = O.rope_inv_freq(1e6, 128)
    assert inv[0] == 1.0
    # successive frequencies shrink by theta^(2/D), to fp32 rounding
    np.testing.assert_allclose(inv[:-1] / inv[1:], 1e6 ** (2 / 128), rtol=3e-7)


def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(31)
    D = 128
    u = O.bf16(rng.standard_normal((5, D)))
    u[u == 0] = 1.0
    c, s = O.rope_cos_sin(1e6, D, np.zeros(5, np.int64))
    out, _ = O.g_rope_bf16(u, c, s)
    np.testing.assert_array_equal(out, u)
    np.testing.assert_array_equal(O.e_rope_bf16(u.astype(F32), c.astype(F32), s.astype(F32)), u.astype(F32))


def test_rope_is_complex_rotation():
    # (out_i + j out_{i+D/2}) = (u_i + j u_{i+D/2}) * exp(j * pos * theta^(-2i/D))
    rng = np.random.default_rng(32)
    D, theta = 64, 1e6
    u = rng.standard_normal((7, D))
    pos = rng.integers(0, 5000, 7)
    out = O.g_rope_exact(u, pos, theta, D)
    i = np.arange(D // 2)
    z = (u[:, : D // 2] + 1j * u[:, D // 2:]) * np.exp(1j * pos[:, None] * theta ** (-2.0 * i / D))
    np.testing.assert_allclose(out[:, : D // 2], z.real, atol=1e-12)
    np.testing.assert_allclose(out[:, D // 2:], z.imag, atol=1e-12)
    # direction (hand value): e_0 at position 1 sends +sin(1) to element D/2
    e0 = np.zeros((1, D))
    e0[0, 0] = 1.0
    r = O.g_rope_exact(e0, np.array([1]), theta, D)
    assert abs(r[0, 0] - math.cos(1.0)) < 1e-15 and abs(r[0, D // 2] - math.sin(1.0)) < 1e-15


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(33)
    D = 128
    q = rng.standard_normal((1, D))
    k = rng.standard_normal((1, D))
    h = D // 2
    r = O.g_rope_exact(q, np.array([37]), 1e6, D)
    np.testing.assert_allclose(r[:, :h] ** 2 + r[:, h:] ** 2, q[:, :h] ** 2 + q[:, h:] ** 2, rtol=1e-12)
    dots = []
    for m, n in ((40, 15), (1040, 1015), (25, 0)):
        dots.append(float(np.sum(O.g_rope_exact(q, np.array([m]), 1e6, D) * O.g_rope_exact(k, np.array([n]), 1e6, D))))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


def test_rope_bf16_agrees_with_exact_rotation():
    # BF16 RoPE stays within a few bf16 steps of the exact rotation of the same u.
    rng = np.random.default_rng(34)
    D = 128
    u = O.bf16(rng.standard_normal((32, D)))
    pos = rng.integers(0, 4096, 32)
    c, s = O.rope_cos_sin(1e6, D, pos)
    out, _ = O.g_rope_bf16(u, c, s)
    assert np.max(np.abs(out - O.g_rope_exact(u, pos, 1e6, D))) < 0.08


def test_e_qk_epilogue_matches_g_on_same_q():
    rng = np.random.default_rng(35)
    Hq, Hkv, D, T = 4, 2, 64, 40
    N = (Hq + 2 * Hkv) * D
    y = O.bf16(rng.standard_normal((T, 256)))
    w = O.bf16(0.02 * rng.standard_normal((2, N, 256)))
    qn = O.bf16(1 + 0.1 * rng.standard_normal((2, D)))
    kn = O.bf16(1 + 0.1 * rng.standard_normal((2, D)))
    mod = rng.integers(0, 2, T)
    pos = np.arange(T)
    g = O.g_qkv_norm_rope(y, w, None, qn, kn, pos, mod, Hq, Hkv, D, 1e-6, 1e6)
    c, s = O.rope_cos_sin(1e6, D, pos)
    e = O.e_qk_norm_rope(g["q"], qn, kn, c, s, mod, Hq, Hkv, D, 1e-6)
    # same q in: E and G differ only by fp32 vs fp64 statistics -> rare one-step flips
    _, ex = np.frexp(np.maximum(np.abs(g["out"]), 2.0 ** -100))
    step = np.ldexp(1.0, ex - 8)
    diff = np.abs(e - g["out"])
    assert np.all(diff <= 2 * step)
    assert np.mean(diff > 0) < 0.01


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

# ---------------------------------------------------------------------------
# FP32 RoPE profile
# ---------------------------------------------------------------------------

def test_rope_f32_table_hand_values():
    gd = GOLDEN["rope_fp32"]
    c, s = O.rope_cos_sin_f32(1e6, 128, np.array([0, 1]))
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    assert c[1, 0] == _hex(gd["pos1_i0_cos"]) and s[1, 0] == _hex(gd["pos1_i0_sin"])
    # the angle is the fp32 product of the position and the fp32 frequency
    a = gd["angle_case"]
    assert O.rope_inv_freq(a["theta"], a["D"])[1] == _hex(a["inv_1"])
    _, s3 = O.rope_cos_sin_f32(a["theta"], a["D"], np.array([a["pos"]]))
    assert s3[0, 1] == _hex(a["sin_1"])


def test_rope_f32_single_cast_and_fp32_sum_hand_values():
    # G rounds the exact rotation once; E rounds the fp32 sum, which lands on a bf16 tie.
    gd = GOLDEN["rope_fp32"]
    D = 4
    u = np.array([[_hex(gd["u_i"]), 0.0, _hex(gd["u_partner"]), 0.0]])
    c = np.ones((1, D // 2))
    s = np.ones((1, D // 2))
    out, pre = O.g_rope_f32(u, c, s)
    assert out[0, 0] == _hex(gd["exact_profile_out"]) and out[0, 2] == _hex(gd["partner_out"])
    assert out[0, 1] == 0.0 and out[0, 3] == 0.0
    e = O.e_rope_f32(u.astype(F32), c.astype(F32), s.astype(F32))
    assert e[0, 0] == _hex(gd["fp32_sum_out"]) and e[0, 2] == _hex(gd["partner_out"])


def _table_bound(u, pos, theta, D):
    """Bound on |rotation with the fp32 table - exact rotation| per element: the fp32 angle
    (two roundings of pos * theta^(-2i/D), relative 2^-23 together) and the fp32 rounding
    of cos and sin (2^-24 each), times |u_i| + |u_partner|."""
    h = D // 2
    i = np.arange(h)
    ang = np.asarray(pos, np.float64)[:, None] * np.power(float(theta), -2.0 * i / D)[None, :]
    per = 1.01 * ang * 2.0 ** -23 + 2.0 ** -23
    mag = np.abs(u[..., :h]) + np.abs(u[..., h:])
    b = mag * per
    return np.concatenate([b, b], axis=-1)


def _complex_rotation(u, pos, theta, D):
    h = D // 2
    i = np.arange(h)
    z = (u[:, :h] + 1j * u[:, h:]) * np.exp(1j * np.asarray(pos)[:, None] * theta ** (-2.0 * i / D))
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_f32_is_rotation_within_table_error():
    rng = np.random.default_rng(36)
    D, theta = 128, 1e6
    u = rng.standard_normal((64, D))
    pos = rng.integers(0, 4096, 64)
    c, s = O.rope_cos_sin_f32(theta, D, pos)
    out, pre = O.g_rope_f32(u, c, s)
    exact = _complex_rotation(u, pos, theta, D)
    assert np.all(np.abs(pre - exact) <= _table_bound(u, pos, theta, D) + 1e-15)
    h = D // 2
    np.testing.assert_allclose(pre[:, :h] ** 2 + pre[:, h:] ** 2, u[:, :h] ** 2 + u[:, h:] ** 2, rtol=2.0 ** -21)


def _half_step(v):
    _, ex = np.frexp(np.maximum(np.abs(v), 2.0 ** -126))
    return np.ldexp(1.0, ex - 9)


@pytest.mark.parametrize("c_q,c_k", [(1.5, -3.0), (0.25, 7.0)])
def test_rope_f32_profile_on_constant_heads_is_one_rounding(c_q, c_k):
    # A constant head c normalizes to g * c / sqrt(c^2 + eps) (closed form); the FP32
    # profile then rotates it with the fp32 table and rounds once, so every output lies
    # within half a bf16 step (plus the table error) of the exact rotation of that closed
    # form. The BF16 profile rounds u, both products and the sum, and misses this bound.
    Hq, Hkv, D, theta = 2, 1, 128, 1e6
    eps = float(F32(1e-6))
    y, w = _onehot_qkv(c_q, c_k, Hq, Hkv, D)
    rng = np.random.default_rng(37)
    qn = O.bf16(1 + 0.2 * rng.standard_normal((2, D)))
    kn = O.bf16(1 + 0.2 * rng.standard_normal((2, D)))
    mod = np.array([0, 1])
    pos = np.array([1234, 3001])
    outs = {}
    for profile in ("fp32", "bf16"):
        outs[profile] = O.g_qkv_norm_rope(y, w, None, qn, kn, pos, mod, Hq, Hkv, D, 1e-6, theta,
                                          rope_profile=profile)["out"]
    c32, s32 = O.rope_cos_sin_f32(theta, D, pos)
    e32 = O.e_qk_norm_rope(O.bf16(np.einsum("tk,tnk->tn", y, w[mod])), qn, kn, c32, s32, mod, Hq, Hkv, D, 1e-6,
                           rope_profile="fp32")
    miss_bf16 = 0
    for h in range(Hq + Hkv):
        cv = c_q if h < Hq else c_k
        g = (qn if h < Hq else kn)[mod]
        u = g * (cv / math.sqrt(cv * cv + eps))
        exact = _complex_rotation(u, pos, theta, D)
        bound = _half_step(exact) + _table_bound(u, pos, theta, D) + 1e-12
        cols = slice(h * D, (h + 1) * D)
        assert np.all(np.abs(outs["fp32"][:, cols] - exact) <= bound)
        # E: fp32 u, products and sum add a few fp32 roundings before the one cast
        e_bound = bound + 8 * 2.0 ** -24 * (np.abs(u) + np.abs(np.roll(u, D // 2, axis=1)))
        e_diff = np.abs(e32[:, cols] - exact)
        assert np.all((e_diff <= e_bound) | (e_diff <= 2 * _half_step(exact)))
        miss_bf16 += int(np.sum(np.abs(outs["bf16"][:, cols] - exact) > bound))
    assert miss_bf16 > 0


def test_e_qk_epilogue_fp32_profile_matches_g_on_same_q():
    rng = np.random.default_rng(38)
    Hq, Hkv, D, T = 4, 2, 64, 40
    N = (Hq + 2 * Hkv) * D
    y = O.bf16(rng.standard_normal((T, 256)))
    w = O.bf16(0.02 * rng.standard_normal((2, N, 256)))
    qn = O.bf16(1 + 0.1 * rng.standard_normal((2, D)))
    kn = O.bf16(1 + 0.1 * rng.standard_normal((2, D)))
    mod = rng.integers(0, 2, T)
    pos = rng.integers(0, 4096, T)
    g = O.g_qkv_norm_rope(y, w, None, qn, kn, pos, mod, Hq, Hkv, D, 1e-6, 1e6, rope_profile="fp32")
    c, s = O.rope_cos_sin_f32(1e6, D, pos)
    e = O.e_qk_norm_rope(g["q"], qn, kn, c, s, mod, Hq, Hkv, D, 1e-6, rope_profile="fp32")
    # same q in: one cast on each side, so they differ by at most one step, rarely
    _, ex = np.frexp(np.maximum(np.abs(g["out"]), 2.0 ** -100))
    step = np.ldexp(1.0, ex - 8)
    diff = np.abs(e - g["out"])
    assert np.all(diff <= step)
    assert np.mean(diff > 0) < 0.01
    # the two profiles are different fingerprints of the same rotation
    gb = O.g_qkv_norm_rope(y, w, None, qn, kn, pos, mod, Hq, Hkv, D, 1e-6, 1e6)
    assert np.any(gb["out"] != g["out"])
    assert np.max(np.abs(gb["out"] - g["out"])) < 0.1


def test_swiglu_hand_values():
    for c in GOLDEN["swiglu"]["cases"]:
        g = O.g_swiglu(np.array([c["g"]]), np.array([c["u"]]))
        assert g["h"][0] == c["h"]
        e = O.e_swiglu(np.array([c["g"]]), np.array([c["u"]]))
        assert e[0] == c["h"]


def test_swiglu_limits_and_e_agreement():
    g = O.g_swiglu(np.array([30.0, -30.0]), np.array([1.0, 1.0]))
    assert g["h"][0] == 30.0 and abs(g["h"][1]) < 1e-11
    rng = np.random.default_rng(41)
    ag = rng.standard_normal(5000) * 3
    au = rng.standard_normal(5000) * 3
    ref = O.g_swiglu(ag, au)
    e = O.e_swiglu(ref["g"], ref["u"])
    _, ex = np.frexp(np.maximum(np.abs(ref["h_pre"]), 2.0 ** -100))
    assert np.all(np.abs(e - ref["h_pre"]) <= np.ldexp(1.0, ex - 8))


def test_layer_composition():
    # the layer is the norm followed by the projection on the norm's bf16 output
    from mixture_transformers_token_gb300 import workloads as W
    shape, inp = W.tiny_layer(seed=2)
    f = {k: (v.float().numpy().astype(np.float64) if isinstance(v, torch.Tensor) and v.is_floating_point() else
             (v.numpy() if isinstance(v, torch.Tensor) else v)) for k, v in inp.items()}
    lay = O.g_layer(f["x"], f["res"], f["w_norm"], f["w_qkv"], None, f["q_norm"], f["k_norm"], f["pos"],
                    f["mod"], shape.Hq, shape.Hkv, shape.D, shape.eps, shape.theta)
    n = O.g_fused_add_rmsnorm(f["x"], f["res"], f["w_norm"], f["mod"], shape.eps)
    q = O.g_qkv_norm_rope(n["y"], f["w_qkv"], None, f["q_norm"], f["k_norm"], f["pos"], f["mod"],
                          shape.Hq, shape.Hkv, shape.D, shape.eps, shape.theta)
    np.testing.assert_array_equal(lay["out"], q["out"])
    assert np.isfinite(lay["out"]).all()


# ---------------------------------------------------------------------------
# backward: routed GEMM dX / dW, add-RMSNorm dx / dw
# ---------------------------------------------------------------------------

def test_routed_dx_dw_brute_force_integers():
    rng = np.random.default_rng(41)
    T, N, K = 7, 5, 3
    dout = rng.integers(-3, 4, (T, N)).astype(np.float64)
    a = rng.integers(-3, 4, (T, K)).astype(np.float64)
    w = rng.integers(-3, 4, (2, N, K)).astype(np.float64)
    mod = np.array([0, 1, 1, 0, 1, 0, 0])
    dx = O.g_routed_gemm_dx(dout, w, mod)["dx_pre"]
    for r in range(T):
        for k in range(K):
            assert dx[r, k] == sum(dout[r, n] * w[mod[r], n, k] for n in range(N))
    for e in (0, 1):
        dw = O.g_routed_gemm_dw(dout, a, mod, e)
        for n in range(N):
            for k in range(K):
                assert dw[n, k] == sum(dout[r, n] * a[r, k] for r in range(T) if mod[r] == e)


def test_routed_dx_dw_adjoint_identities():
    # <dout, routed(a, W)> = <dA, a> = sum_e <dW_e, W_e>  (the backward is the adjoint of the forward)
    rng = np.random.default_rng(42)
    T, N, K = 40, 24, 16
    dout = rng.standard_normal((T, N))
    a = rng.standard_normal((T, K))
    w = rng.standard_normal((2, N, K))
    mod = rng.integers(0, 2, T)
    lhs = float(np.sum(dout * O.g_routed_matmul(a, w, mod)))
    via_dx = float(np.sum(O.g_routed_gemm_dx(dout, w, mod)["dx_pre"] * a))
    via_dw = sum(float(np.sum(O.g_routed_gemm_dw(dout, a, mod, e) * w[e])) for e in (0, 1))
    assert abs(via_dw - lhs) <= 1e-9 * (1 + abs(lhs))
    assert abs(via_dx - lhs) <= 1e-9 * (1 + abs(lhs))
    # a weight set's gradient ignores the other set's rows
    d2 = dout.copy()
    d2[mod == 1] = rng.standard_normal((int(np.sum(mod == 1)), N))
    np.testing.assert_array_equal(O.g_routed_gemm_dw(d2, a, mod, 0), O.g_routed_gemm_dw(dout, a, mod, 0))


def _norm_forward_pre(s, w, mod, eps):
    """The cast-free add-RMSNorm forward as a function of the residual sum s (for finite differences)."""
    rstd = 1.0 / np.sqrt(np.mean(s * s, axis=1) + eps)
    return s * rstd[:, None] * w[mod]


def test_norm_backward_is_the_gradient():
    # directional derivatives by central differences of F(s, w) = <dy, y_pre(s, w)> + <dro, s>
    rng = np.random.default_rng(43)
    T, H = 6, 256
    eps = float(F32(1e-6))
    s = rng.standard_normal((T, H))
    s[2] *= 1e-3                                       # a row where eps matters
    w = 1 + 0.1 * rng.standard_normal((2, H))
    dy = rng.standard_normal((T, H))
    dro = rng.standard_normal((T, H))
    mod = np.array([0, 1, 1, 0, 1, 0])
    g = O.g_add_rmsnorm_backward(dy, s, w, mod, 1e-6, d_res_out=dro)

    def F(s_, w_):
        return float(np.sum(dy * _norm_forward_pre(s_, w_, mod, eps)) + np.sum(dro * s_))

    h = 1e-6
    for seed in range(3):
        v = np.random.default_rng(100 + seed).standard_normal((T, H))
        num = (F(s + h * v, w) - F(s - h * v, w)) / (2 * h)
        assert abs(num - float(np.sum(g["dx_pre"] * v))) <= 1e-5 * (1 + abs(num))
        V = np.random.default_rng(200 + seed).standard_normal((2, H))
        num_w = (F(s, w + h * V) - F(s, w - h * V)) / (2 * h)
        assert abs(num_w - float(np.sum(g["dw"] * V))) <= 1e-5 * (1 + abs(num_w))


def test_left_fold_hand_value():
    gd = GOLDEN["dweight_left_fold"]
    p = np.array(gd["partials"], F32)[:, None]
    mod = np.array(gd["mod"])
    assert O.e_left_fold_rows(p, mod, 1)[0] == gd["dw_gen"]
    assert O.e_left_fold_rows(p, mod, 0)[0] == gd["dw_und"]
    assert O.e_left_fold_rows(p[:0], mod[:0], 0).shape == (1,)


def test_norm_backward_e_dot_uses_the_forward_tree():
    # s = 1, w = 1, eps = 0: rstd = 1 and xh = 1, so the dot's terms are dy itself; dy set to
    # row A of the forward tree fixture (2^24 at column 0, 1 at columns 1..7 and at 8l) sums
    # to the fixture's hand value on the fixed tree
    gd = GOLDEN["add_rmsnorm_tree_sum"]
    H = 512
    dy = np.zeros((1, H))
    dy[0, 0] = 2.0 ** 24
    dy[0, 1:8] = 1.0
    dy[0, 8 * np.arange(1, 32)] = 1.0
    e = O.e_add_rmsnorm_backward(dy, np.ones((1, H)), np.ones((2, H)), np.array([0]), 0.0)
    assert e["rstd"][0] == 1.0
    assert e["dot"][0] == gd["row_A_sum_of_squares"]


def test_norm_backward_e_matches_g():
    rng = np.random.default_rng(44)
    T, H = 48, 512
    s = O.bf16(rng.standard_normal((T, H)))
    dy = O.bf16(rng.standard_normal((T, H)))
    dro = O.bf16(rng.standard_normal((T, H)))
    w = O.bf16(1 + 0.1 * rng.standard_normal((2, H)))
    mod = rng.integers(0, 2, T)
    for d_res in (None, dro):
        g = O.g_add_rmsnorm_backward(dy, s, w, mod, 1e-6, d_res_out=d_res)
        e = O.e_add_rmsnorm_backward(dy, s, w, mod, 1e-6, d_res_out=d_res)
        # one cast on each side: equal or one bf16 step apart, rarely
        _, ex = np.frexp(np.maximum(np.abs(g["dx"]), 2.0 ** -100))
        step = np.ldexp(1.0, ex - 8)
        diff = np.abs(e["dx"] - g["dx"])
        assert np.all(diff <= step) and np.mean(diff > 0) < 0.02
        np.testing.assert_allclose(e["dw"], g["dw"], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(e["rstd"], g["rstd"], rtol=1e-6)


# ---------------------------------------------------------------------------
# joint attention
# ---------------------------------------------------------------------------

def _qkv_rows(q, k, v):
    """Pack per-row q [T][Hq][D], k and v [T][Hkv][D] into the fused QKV layout."""
    T = q.shape[0]
    return np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], axis=1)


def test_joint_attention_scale_and_softmax_hand_value():
    gd = GOLDEN["joint_attention"]
    D = 4
    q = np.zeros((2, 1, D))
    k = np.zeros((2, 1, D))
    v = np.zeros((2, 1, D))
    q[1, 0, 0] = 2.0          # the query is row 1; rows 0 and 1 are the keys
    k[1, 0, 0] = 1.0
    v[1, 0, :] = 1.0
    r = O.g_joint_attention(_qkv_rows(q, k, v), [(1, 0, 1, 2, 0)], 1, 1, D)
    assert np.allclose(r["out_pre"][1], gd["sigmoid_1"], rtol=0, atol=1e-15)
    assert np.all(r["out"][1] == gd["sigmoid_1_bf16"])
    assert np.all(r["out"][0] == 0.0)        # not a query row of any sequence


def test_joint_attention_bottom_right_alignment_and_closed_forms():
    rng = np.random.default_rng(51)
    D, nk = 8, 3
    v = O.bf16(rng.standard_normal((nk, 1, D)))
    qkv = _qkv_rows(np.zeros((nk, 1, D)), O.bf16(rng.standard_normal((nk, 1, D))), v)
    # one causal query at the bottom right sees all three keys; q = 0 gives their mean
    r = O.g_joint_attention(qkv, [(2, 0, 1, nk, 1)], 1, 1, D)
    np.testing.assert_allclose(r["out_pre"][2], v[:, 0].mean(axis=0), rtol=0, atol=1e-15)
    # the first causal row of a full-length sequence sees key 0 only: out = v0 exactly
    qkv2 = _qkv_rows(O.bf16(rng.standard_normal((nk, 1, D))), O.bf16(rng.standard_normal((nk, 1, D))), v)
    r2 = O.g_joint_attention(qkv2, [(0, 0, nk, nk, nk)], 1, 1, D)
    np.testing.assert_array_equal(r2["out"][0], v[0, 0])
    # q = 0: a causal row i averages v_0..v_i, a latent row averages all values
    r3 = O.g_joint_attention(qkv, [(0, 0, nk, nk, 2)], 1, 1, D)
    np.testing.assert_allclose(r3["out_pre"][1], v[:2, 0].mean(axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(r3["out_pre"][2], v[:, 0].mean(axis=0), rtol=0, atol=1e-15)


def test_joint_attention_grouped_heads():
    # query heads 0, 1 read KV head 0 (values 1); heads 2, 3 read KV head 1 (values 2)
    rng = np.random.default_rng(52)
    T, D, Hq, Hkv = 5, 8, 4, 2
    q = rng.standard_normal((T, Hq, D))
    k = rng.standard_normal((T, Hkv, D))
    v = np.zeros((T, Hkv, D))
    v[:, 0] = 1.0
    v[:, 1] = 2.0
    r = O.g_joint_attention(_qkv_rows(q, k, v), [(0, 0, T, T, 3)], Hq, Hkv, D)
    out = r["out_pre"].reshape(T, Hq, D)
    np.testing.assert_allclose(out[:, :2], 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[:, 2:], 2.0, rtol=0, atol=1e-12)


def test_joint_attention_brute_force_and_sequence_independence():
    rng = np.random.default_rng(53)
    Hq, Hkv, D = 4, 2, 8
    T = 13
    qkv = O.bf16(rng.standard_normal((T, (Hq + 2 * Hkv) * D)))
    seqs = [(0, 0, 6, 6, 4), (6, 6, 3, 7, 3), (10, 6, 3, 7, 0)]  # the last two share keys (cached prefix)
    r = O.g_joint_attention(qkv, seqs, Hq, Hkv, D)
    for q0, k0, nq, nk, nc in seqs:
        for i in range(nq):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                qv = qkv[q0 + i, h * D:(h + 1) * D]
                keys = [j for j in range(nk) if i >= nc or j <= nk - nq + i]
                sc = [math.fsum(qv[d] * qkv[k0 + j, (Hq + g) * D + d] for d in range(D)) / math.sqrt(D) for j in keys]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = math.fsum(w)
                for d in range(D):
                    want = math.fsum(w[n] * qkv[k0 + j, (Hq + Hkv + g) * D + d] for n, j in enumerate(keys)) / tot
                    assert abs(r["out_pre"][q0 + i, h * D + d] - want) <= 1e-12
    # changing another sequence's rows leaves a sequence's output bit for bit
    qkv2 = qkv.copy()
    qkv2[:6] = O.bf16(rng.standard_normal((6, qkv.shape[1])))
    r2 = O.g_joint_attention(qkv2, seqs, Hq, Hkv, D)
    np.testing.assert_array_equal(r2["out_pre"][6:], r["out_pre"][6:])


# ---------------------------------------------------------------------------
# flow schedule, CFG combine with renorm, SDE step and logp
# ---------------------------------------------------------------------------

def test_flow_schedule_reproduces_the_printed_guided_step_counts():
    gd = GOLDEN["flow_schedule_guided_steps"]
    lo, hi = gd["window"]
    for shift, want in gd["guided"].items():
        ts = O.flow_schedule(gd["n"], float(shift))
        assert sum(O.cfg_guided(ts[i], lo, hi) for i in range(gd["n"] - 1)) == want
    ts = O.flow_schedule(5, 3.0)
    assert ts.dtype == np.float32 and ts[0] == 1.0 and ts[-1] == 0.0
    assert ts[2] == F32(0.75)                                  # u = 1/2: 1.5 / 2
    np.testing.assert_array_equal(O.flow_schedule(5, 1.0), np.array([1, 0.75, 0.5, 0.25, 0], F32))


def test_request_tree_sum_hand_values():
    gd = GOLDEN["request_tree_sum"]
    a = np.zeros(16, F32)
    a[0] = 2.0 ** 24
    a[1:] = 1.0
    assert O.e_request_tree_sum(a) == gd["chunks_sum"]
    b = np.zeros(65 * 8, F32)
    b[0] = 2.0 ** 24
    b[32 * 8] = 1.0
    b[64 * 8] = 1.0
    assert O.e_request_tree_sum(b) == gd["warps_sum"]
    c = np.zeros(2 * O.FLOW_SEGMENT + 8, F32)
    c[0] = 2.0 ** 24
    c[O.FLOW_SEGMENT] = 1.0
    c[2 * O.FLOW_SEGMENT] = 1.0
    assert O.e_request_tree_sum(c) == gd["segments_sum"]
    # a small-magnitude sum is the exact sum (every partial sum is representable)
    rng = np.random.default_rng(64)
    d = rng.integers(-1000, 1000, 3 * O.FLOW_SEGMENT + 40).astype(F32)
    assert O.e_request_tree_sum(d) == float(np.sum(d.astype(np.int64)))


def test_cfg_combine_identities_window_and_renorm():
    rng = np.random.default_rng(61)
    N = 512
    c, tu, iu = (rng.standard_normal(N) for _ in range(3))
    # outside the window: the conditioned velocity itself
    np.testing.assert_array_equal(O.g_cfg_combine_renorm(c, tu, iu, 0.2, 4.0, 2.0, 0.4, 1.0, 0.0), c)
    # text scale 1 without an image branch: v1 = c, r = 1
    np.testing.assert_allclose(O.g_cfg_combine_renorm(c, tu, None, 0.5, 1.0, 1.0, 0.4, 1.0, 0.0), c, atol=1e-15)
    # equal branches leave c unchanged for any scales
    np.testing.assert_allclose(O.g_cfg_combine_renorm(c, c, c, 0.5, 4.0, 2.0, 0.0, 1.0, 0.0), c, atol=1e-12)
    # the two interpolations by hand, and the rescale to ||c|| when the guided norm is larger
    v = O.g_cfg_combine_renorm(c, tu, iu, 0.5, 4.0, 2.0, 0.4, 1.0, 0.0)
    v1 = tu + 4.0 * (c - tu)
    v2 = iu + 2.0 * (v1 - iu)
    assert np.linalg.norm(v2) > np.linalg.norm(c)
    np.testing.assert_allclose(v, v2 * np.linalg.norm(c) / np.linalg.norm(v2), rtol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(v), np.linalg.norm(c), rtol=1e-13)
    # the clamp from below
    v_min = O.g_cfg_combine_renorm(c, tu, iu, 0.5, 4.0, 2.0, 0.4, 1.0, 0.9)
    np.testing.assert_allclose(v_min, float(F32(0.9)) * v2, rtol=1e-13)   # the policy values are fp32
    # the guided norm below ||c||: r would exceed 1 and is clamped to it (v = v2)
    np.testing.assert_allclose(O.g_cfg_combine_renorm(c, np.zeros(N), None, 0.5, 0.5, 1.0, 0.4, 1.0, 0.0), 0.5 * c,
                               rtol=1e-15)
    # the window includes both ends (compared on fp32 t)
    assert O.cfg_guided(F32(0.4), 0.4, 1.0) and O.cfg_guided(1.0, 0.4, 1.0)
    assert not O.cfg_guided(np.nextafter(F32(0.4), F32(0)), 0.4, 1.0)
    # E follows G
    e = O.e_cfg_combine_renorm(c, tu, iu, 0.5, 4.0, 2.0, 0.4, 1.0, 0.0)
    np.testing.assert_allclose(e, v, rtol=2e-5, atol=2e-5)


def test_sde_step_closed_forms_and_logp():
    pytest.importorskip("scipy")
    from scipy.stats import norm
    rng = np.random.default_rng(62)
    N = 256
    x, v, z = (rng.standard_normal(N) for _ in range(3))
    # t = 1 (the first step): eps_hat = x, mu = x - dt (v + x / 2), std = sqrt(dt)
    r = O.g_flow_sde_step(x, v, np.zeros(N), 1.0, 0.75)
    np.testing.assert_allclose(r["mu"], x - 0.25 * (v + 0.5 * x), rtol=1e-14)
    assert abs(r["std"] - 0.5) < 1e-15
    np.testing.assert_array_equal(r["x_next"], r["mu"])
    assert abs(r["logp"] - N * norm.logpdf(0.0, scale=0.5)) < 1e-9
    # logp of a noisy step against the library's Gaussian log-density
    t, tn = float(F32(0.3)), float(F32(0.28))
    r = O.g_flow_sde_step(x, v, z, t, tn)
    assert abs(r["logp"] - np.sum(norm.logpdf(r["x_next"], loc=r["mu"], scale=r["std"]))) < 1e-8
    # E follows G
    e = O.e_flow_sde_step(x, v, z, t, tn)
    np.testing.assert_allclose(e["x_next"], r["x_next"], rtol=1e-5, atol=1e-6)
    assert abs(e["logp"] - r["logp"]) < 1e-4 * abs(r["logp"])


def test_sde_step_keeps_the_gaussian_marginals():
    # data x0 ~ N(0, a^2), eps ~ N(0, 1): x_t ~ N(0, s_t^2), s_t^2 = (1-t)^2 a^2 + t^2, and the exact
    # velocity is v = beta x with beta = (t - (1-t) a^2) / s_t^2. One step of the reverse SDE must
    # carry the variance s_t^2 to s_{t-dt}^2 up to O(dt^2); a wrong sign or factor on the score term
    # leaves an O(dt) error.
    a2, t = 0.7, 0.6
    s2 = lambda tt: (1 - tt) ** 2 * a2 + tt * tt
    errs = []
    for dt in (1e-2, 5e-3, 2.5e-3):
        beta = (t - (1 - t) * a2) / s2(t)
        # the step is linear in x and z: x_next = A x + std z
        A = O.g_flow_sde_step(np.array([1.0]), np.array([beta]), np.array([0.0]), t, t - dt)["mu"][0]
        std = O.g_flow_sde_step(np.array([0.0]), np.array([0.0]), np.array([0.0]), t, t - dt)["std"]
        var = A * A * s2(t) + std * std
        errs.append(abs(var - s2(t - dt)))
    assert errs[0] < 1e-3
    assert errs[1] < errs[0] / 3 and errs[2] < errs[1] / 3     # quadratic convergence


def test_sde_logp_of_a_given_latent():
    # Training scores the latent a rollout stored: with the same x, v and times, evaluating the
    # step at the rollout's x_next returns the rollout's logp exactly, and for any other latent
    # it is the library's Gaussian log-density around mu.
    pytest.importorskip("scipy")
    from scipy.stats import norm
    rng = np.random.default_rng(63)
    N = 4096
    x, v, z = (rng.standard_normal(N) for _ in range(3))
    t, tn = float(F32(0.55)), float(F32(0.5))
    roll = O.e_flow_sde_step(x, v, z, t, tn)
    score = O.e_flow_sde_step(x, v, None, t, tn, x_next=roll["x_next"])
    assert score["logp"] == roll["logp"]
    np.testing.assert_array_equal(score["x_next"], roll["x_next"])
    y = rng.standard_normal(N)
    g = O.g_flow_sde_step(x, v, None, t, tn, x_next=y)
    assert abs(g["logp"] - np.sum(norm.logpdf(y, loc=g["mu"], scale=g["std"]))) < 1e-7
    e = O.e_flow_sde_step(x, v, None, t, tn, x_next=y)
    assert abs(e["logp"] - g["logp"]) < 1e-4 * abs(g["logp"])


def test_philox_matches_numpy_bit_generator():
    # numpy's Philox bit generator is Philox4x64-10; it advances the counter before each block
    for ctr, key in (((0, 0, 0, 0), (0, 0)), ((5, 7, 0, 3), (11, 13)),
                     ((2 ** 64 - 1, 2 ** 64 - 1, 2 ** 64 - 1, 2 ** 64 - 2), (2 ** 64 - 1, 2 ** 63)),
                     ((123456789, 42, 0, 0), (987654321, O.NOISE_DOMAIN))):
        bg = np.random.Philox(counter=list(ctr), key=list(key))
        got = [int(v) for v in bg.random_raw(4)]
        c = list(ctr)
        c[0] = (c[0] + 1) % 2 ** 64
        if c[0] == 0:
            c[1] = (c[1] + 1) % 2 ** 64
            if c[1] == 0:
                c[2] = (c[2] + 1) % 2 ** 64
                if c[2] == 0:
                    c[3] = (c[3] + 1) % 2 ** 64
        assert list(O.philox4x64_10(c, key)) == got


def test_noise_uniform_mapping_and_box_muller():
    # the mapping's ends and exactness
    assert O.noise_uniform(0) == F32(0.5 * 2.0 ** -23)
    assert O.noise_uniform(2 ** 64 - 1) == F32(1.0 - 2.0 ** -24)
    assert O.noise_uniform(1 << 41) == F32(1.5 * 2.0 ** -23)
    # Box-Muller identities: the pair's squared radius is -2 ln u_even and its angle 2 pi u_odd
    N = 64
    u = O.flow_noise_uniforms(7, 3, N).astype(np.float64)
    z = O.g_flow_noise([7], 3, N)[0]
    np.testing.assert_allclose(z[0::2] ** 2 + z[1::2] ** 2, -2.0 * np.log(u[0::2]), rtol=1e-12)
    ang = np.mod(np.arctan2(z[1::2], z[0::2]), 2 * np.pi)
    np.testing.assert_allclose(ang, 2 * np.pi * u[1::2], rtol=1e-9, atol=1e-12)
    # a different seed, step or element block gives different deviates
    assert not np.array_equal(O.g_flow_noise([8], 3, N)[0], z)
    assert not np.array_equal(O.g_flow_noise([7], 4, N)[0], z)


def test_noise_is_standard_normal():
    pytest.importorskip("scipy")
    from scipy import stats
    z = O.g_flow_noise([2024, 7], 11, 8192).reshape(-1)
    assert abs(z.mean()) < 0.03 and abs(z.var() - 1.0) < 0.04
    assert stats.kstest(z, "norm").pvalue > 1e-3

