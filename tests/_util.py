"""Shared helpers of the GPU tests: conversions, the tolerance gate, plan decoding."""

import numpy as np
import pytest
import torch

# Tolerance on bf16 outputs against the fp64 golden's value before its final cast:
# max |diff| <= 2e-2 (or half a bf16 step where |value| >= 8) and relative L2 <= 4e-3.
MAX_ABS = 2e-2
MAX_REL_L2 = 4e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy().astype(np.float64)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def np_bits(a: np.ndarray) -> np.ndarray:
    """int16 bit patterns of float values that are exact bf16 numbers."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy()


def half_bf16_step(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |v|: the error of a correctly rounded bf16 value."""
    _, ex = np.frexp(np.maximum(np.abs(v), 2.0 ** -126))
    return np.ldexp(1.0, ex - 9)


def allowed_abs(ref: np.ndarray, acc_err=None) -> np.ndarray:
    """max |diff| bound per element: 2e-2, or -- where |ref| >= 8, since no bf16 number lies
    within 2e-2 of an exact value there -- half a bf16 step (a correctly rounded result) plus
    the accumulation error that can carry an fp32 sum across the rounding tie, capped at half a
    step so that only the other neighbour of the exact value is admitted. acc_err is that error
    bound per element when the caller has it (2 K 2^-24 sum|a||w| for a K-long fp32 dot
    product); otherwise 1e-5 |ref|."""
    h = half_bf16_step(ref)
    slack = 1e-5 * np.abs(ref) if acc_err is None else np.minimum(acc_err, h)
    return np.maximum(MAX_ABS, h + slack)


def gemm_acc_err(K: int, acc_abs: np.ndarray) -> np.ndarray:
    """Bound on the fp32 accumulation error of K-long dot products whose absolute terms sum to
    acc_abs (the products of bf16 numbers are exact; each of at most K additions rounds by at
    most one fp32 unit, counted twice for a non-nearest rounding of the accumulator)."""
    return 2.0 * K * 2.0 ** -24 * acc_abs


def tol_report(gpu: np.ndarray, ref: np.ndarray, acc_err=None) -> tuple[float, float, int]:
    d = np.abs(gpu - ref)
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    return float(d.max()) if d.size else 0.0, rel, int(np.sum(d > allowed_abs(ref, acc_err)))


def assert_tolerance(gpu: np.ndarray, ref: np.ndarray, what: str, acc_err=None) -> None:
    maxd, rel, nbad = tol_report(gpu, ref, acc_err)
    if nbad:
        idx = np.argwhere(np.abs(gpu - ref) > allowed_abs(ref, acc_err))[:10]
        detail = [(tuple(int(v) for v in i), float(gpu[tuple(i)]), float(ref[tuple(i)])) for i in idx]
    else:
        detail = []
    assert nbad == 0 and rel <= MAX_REL_L2, f"{what}: max|diff| {maxd:.3e} rel-L2 {rel:.3e} {detail}"


def assert_bitwise(a: torch.Tensor | np.ndarray, b: torch.Tensor | np.ndarray, what: str) -> None:
    ba = bits(a) if isinstance(a, torch.Tensor) else a
    bb = bits(b) if isinstance(b, torch.Tensor) else b
    if not np.array_equal(ba, bb):
        bad = np.argwhere(ba != bb)
        raise AssertionError(f"{what}: {len(bad)} elements differ, first {bad[:5].tolist()}")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mixture_transformers_token_gb300 import build
    build.build()


def decode_plan(ws: torch.Tensor, T: int):
    raw = ws.cpu().numpy()
    hdr = raw[:64].view(np.int32)
    perm = raw[64:64 + 4 * T].view(np.int32)
    toff = 64 + ((4 * T + 15) // 16) * 16
    ntiles = int(hdr[3])
    tiles = raw[toff:toff + 16 * ntiles].view(np.int32).reshape(ntiles, 4)
    return {"T": int(hdr[0]), "count": (int(hdr[1]), int(hdr[2])), "num_m_tiles": ntiles,
            "error": int(raw[16:20].view(np.uint32)[0]), "magic": int(raw[20:24].view(np.uint32)[0]),
            "perm": perm, "tiles": tiles}


def bf16_step(v):
    """Spacing of bf16 numbers at |v| (2^-133 below the normal range)."""
    _, ex = np.frexp(np.maximum(np.abs(v), 2.0 ** -126))
    return np.ldexp(1.0, ex - 8)


def _rope_pre_of_u(u, c, s, profile):
    """The value of the emulator's output before its final bf16 cast, from its own normalized
    heads u [T][heads][D]: in the BF16 profile bf16(u_i c) + bf16(partner_i s), exact in fp64
    (products of two bf16 numbers and the sum of two are exact there); in the FP32 profile the
    fp32 products and sum, each rounded to fp32."""
    if profile == "bf16":
        from oracle import mot_oracle as O

        return O.g_rope_bf16(u, c[:, None, :], s[:, None, :])[1]
    u32 = u.astype(np.float32)
    c32 = c.astype(np.float32)[:, None, :]
    s32 = s.astype(np.float32)[:, None, :]
    h = u.shape[-1] // 2
    u1, u2 = u32[..., :h], u32[..., h:]
    return np.concatenate([(u1 * c32) + (-u2 * s32), (u2 * c32) + (u1 * s32)], axis=-1).astype(np.float64)


def check_end_to_end(out, g, q_gpu, u_e, acc_abs, shape, what, profile, epi):
    """End to end against the fp64 golden chain G, with a cause proven for every element
    beyond the tolerance.

    The pages declare bf16 casts after the GEMM (q = bf16(acc), u in the BF16 profile, each
    RoPE product and the sum), so a legitimate one-step difference at one of them can grow
    past 2e-2 downstream. The check:
      0. rel-L2 <= 4e-3 over the whole output; every GEMM output q_gpu lies within half a bf16
         step plus the fp32 accumulation bound 2 K 2^-24 sum|a||w| (acc_abs) of the exact
         accumulation (a legitimate fixed-order fp32 sum, rounded once).
      1. G_tf = G's fp64 epilogue applied to the GPU's own q_gpu (teacher forcing). An element
         beyond the bound of G but within it of G_tf is caused by the GEMM's rounding of q
         (G and G_tf differ only in q), which step 0 bounds.
      2. An element beyond the bound of G_tf too is accepted only if the emulator's u (fp32
         statistics, which the GPU matches bit for bit) and G_tf's u differ at the element or
         at its rotation partner (BF16 profile), and the output is the final cast of the
         emulator's rotation of its u: |out - pre_E| <= half a bf16 step. In the FP32 profile
         u is not rounded; the emulator's pre-cast value must lie within the fp32 rounding of
         u, both products and the sum of G_tf's, and the output within half a step of it.
    Anything else fails. `epi` holds the epilogue's inputs: q_norm, k_norm, pos, mod, eps,
    theta (float64 / integer arrays). Returns the counts of each cause.
    """
    from oracle import mot_oracle as O

    D, nqk = shape.D, shape.Hq + shape.Hkv
    ref = g["out_pre"]
    d = np.abs(out - ref)
    rel = float(np.linalg.norm(out - ref) / np.linalg.norm(ref))
    assert rel <= MAX_REL_L2, f"{what}: rel-L2 {rel:.3e}"
    K = shape.H
    gemm_err = np.abs(q_gpu - g["acc"])
    allowed = 0.5 * bf16_step(q_gpu) + gemm_acc_err(K, acc_abs)
    assert np.all(gemm_err <= allowed), f"{what}: GEMM output outside half a step plus the accumulation bound"
    q_flips = int(np.sum(q_gpu != g["q"]))
    bad = d > allowed_abs(ref)
    n_bad = int(bad.sum())
    n_gemm = n_stats = 0
    if n_bad:
        rows = np.unique(np.nonzero(bad)[0])
        g_tf = O.g_qk_norm_rope(q_gpu[rows], epi["q_norm"], epi["k_norm"], epi["pos"][rows], epi["mod"][rows],
                                shape.Hq, shape.Hkv, D, shape.eps, shape.theta, rope_profile=profile)
        o, b = out[rows], bad[rows]
        tf_ok = np.abs(o - g_tf["out_pre"]) <= allowed_abs(g_tf["out_pre"])
        n_gemm = int(np.sum(b & tf_ok))
        rest = b & ~tf_ok
        unexplained = []
        if rest.any():
            table = O.rope_cos_sin if profile == "bf16" else O.rope_cos_sin_f32
            c, s = table(shape.theta, D, epi["pos"][rows])
            ue = u_e[rows]
            pre_e = _rope_pre_of_u(ue, c, s, profile).reshape(len(rows), nqk * D)
            utf = g_tf["u"]
            for rr, col in np.argwhere(rest):
                h, i = divmod(int(col), D)
                r = int(rows[rr])
                if h >= nqk:
                    unexplained.append((r, int(col), float(o[rr, col]), float(ref[r, col]), "V column"))
                    continue
                j = (i + D // 2) % D
                cast_only = abs(o[rr, col] - pre_e[rr, col]) <= 0.5 * bf16_step(o[rr, col]) * (1 + 1e-9)
                if profile == "bf16":
                    # u differs by at most one bf16 step at i or its partner j, and the rotations
                    # of the two u differ by no more than that flip times (cos, sin) plus the
                    # rounding of each side's two products
                    f = i % (D // 2)
                    du_i, du_j = abs(ue[rr, h, i] - utf[rr, h, i]), abs(ue[rr, h, j] - utf[rr, h, j])
                    one_step = (du_i <= bf16_step(max(abs(ue[rr, h, i]), abs(utf[rr, h, i]))) and
                                du_j <= bf16_step(max(abs(ue[rr, h, j]), abs(utf[rr, h, j]))))
                    cf, sf = abs(c[rr, f]), abs(s[rr, f])
                    prop = (du_i * cf + du_j * sf + bf16_step(abs(utf[rr, h, i]) * cf) +
                            bf16_step(abs(utf[rr, h, j]) * sf))
                    ok = (du_i > 0 or du_j > 0) and one_step and cast_only and \
                        abs(pre_e[rr, col] - g_tf["out_pre"][rr, col]) <= prop * (1 + 1e-9)
                else:
                    slack = 16 * 2.0 ** -24 * (abs(utf[rr, h, i]) + abs(utf[rr, h, j]))
                    ok = cast_only and abs(pre_e[rr, col] - g_tf["out_pre"][rr, col]) <= slack
                if ok:
                    n_stats += 1
                else:
                    unexplained.append((r, int(col), float(o[rr, col]), float(ref[r, col]),
                                        float(g_tf["out_pre"][rr, col])))
        assert not unexplained, f"{what}: |diff| beyond the bound with no proven cause (row, col, out, G, G_tf): " \
                                f"{unexplained[:10]}"
    print(f"{what}: max|diff| {d.max():.3e}, rel-L2 {rel:.2e}; q flips at the GEMM cast: {q_flips}; "
          f"{n_bad} of {d.size} elements beyond the bound of G: {n_gemm} within it of the teacher-forced "
          f"golden (GEMM rounding of q), {n_stats} from an fp32-statistics flip of u and the final cast")
    return {"max_abs": float(d.max()), "rel_l2": rel, "beyond": n_bad, "q_flips": q_flips, "gemm_cause": n_gemm,
            "stats_cause": n_stats}
