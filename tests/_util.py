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


def allowed_abs(ref: np.ndarray) -> np.ndarray:
    """max |diff| bound per element: 2e-2, or -- where |ref| >= 8, since no bf16 number lies
    within 2e-2 of an exact value there -- half a bf16 step plus 1e-5 |ref| for the fp32
    accumulation rounding that can put a value just past a rounding tie."""
    return np.maximum(MAX_ABS, half_bf16_step(ref) + 1e-5 * np.abs(ref))


def tol_report(gpu: np.ndarray, ref: np.ndarray) -> tuple[float, float, int]:
    d = np.abs(gpu - ref)
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    return float(d.max()) if d.size else 0.0, rel, int(np.sum(d > allowed_abs(ref)))


def assert_tolerance(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    maxd, rel, nbad = tol_report(gpu, ref)
    if nbad:
        idx = np.argwhere(np.abs(gpu - ref) > allowed_abs(ref))[:10]
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


def check_end_to_end(out, g, q_gpu, u_e, acc_abs, shape, what, profile="bf16"):
    """End to end against the fp64 golden chain.

    The relative-L2 bound holds for the whole output. An element may exceed 2e-2 only when a
    legitimate one-step difference at a declared bf16 cast explains it: the GEMM's fp32
    accumulation rounding q to the other bf16 neighbour of the exact value (anywhere in the
    element's head, which moves rstd), the fp32 statistics rounding u the other way at the
    element or its rotation partner (BF16 profile; the FP32 profile does not round u), or the
    final cast alone -- within half a step, plus in the FP32 profile the fp32 rounding of u,
    both products and the sum, which can carry a value across the cast's rounding tie. Every q
    itself must lie within half a bf16 step plus the fp32 accumulation error bound
    2 K 2^-24 sum|a||w| (acc_abs) of the exact accumulation.
    """
    D, nqk = shape.D, shape.Hq + shape.Hkv
    ref = g["out_pre"]
    d = np.abs(out - ref)
    rel = float(np.linalg.norm(out - ref) / np.linalg.norm(ref))
    assert rel <= 4e-3, f"{what}: rel-L2 {rel:.3e}"
    K = shape.H
    gemm_err = np.abs(q_gpu - g["acc"])
    allowed = 0.5 * bf16_step(q_gpu) + 2.0 * K * 2.0 ** -24 * acc_abs
    assert np.all(gemm_err <= allowed), f"{what}: GEMM output outside half a step plus the accumulation bound"
    flips = q_gpu != g["q"]
    bad = np.argwhere(d > allowed_abs(ref))
    unexplained = []
    for r, c in bad:
        h, i = divmod(int(c), D)
        j = (i + D // 2) % D
        slack = 0.0
        if profile == "fp32" and h < nqk:
            slack = 16 * 2.0 ** -24 * (abs(g["u"][r, h, i]) + abs(g["u"][r, h, j]))
        final_cast = d[r, c] <= 0.5 * bf16_step(out[r, c]) * (1 + 1e-9) + slack
        q_flip = bool(np.any(flips[r, h * D:(h + 1) * D]))
        u_flip = profile == "bf16" and h < nqk and (u_e[r, h, i] != g["u"][r, h, i] or u_e[r, h, j] != g["u"][r, h, j])
        if not (final_cast or q_flip or u_flip):
            unexplained.append((int(r), int(c), float(out[r, c]), float(ref[r, c])))
    assert not unexplained, f"{what}: unexplained |diff| > 2e-2 at {unexplained[:10]}"
    # scale-aware sanity bound on Q/K columns: a few bf16 steps of the rotated pair (u_i, u_j)
    cols = np.arange(nqk * D)
    hh, ii = cols // D, cols % D
    jj = (ii + D // 2) % D
    scale = np.maximum(np.abs(g["u"][:, hh, ii]), np.abs(g["u"][:, hh, jj]))
    # plus what the GEMM's own cast output carries in: q_gpu may sit several bf16 steps from the
    # golden q where the accumulation cancels (the fp32 bound above is absolute), and the head's
    # norm scales that difference by rstd * g, bounded here by twice the head's |u| / |q| ratio
    dq = np.abs(q_gpu[:, : nqk * D] - g["q"][:, : nqk * D]).reshape(-1, nqk, D)
    qh = np.sqrt(np.sum(g["q"][:, : nqk * D].reshape(-1, nqk, D) ** 2, axis=2))
    uh = np.sqrt(np.sum(g["u"] ** 2, axis=2))
    factor = 2.0 * uh / np.maximum(qh, 1e-300)
    prop = (factor[:, hh] * (dq[:, hh, ii] + dq[:, hh, jj]))
    lim = 3 * bf16_step(scale) + bf16_step(ref[:, : nqk * D]) + prop
    over = np.argwhere(d[:, : nqk * D] > lim)
    detail = [(int(r), int(c), float(out[r, c]), float(ref[r, c]), float(g["u"][r, c // D, c % D]),
               float(g["u"][r, c // D, (c % D + D // 2) % D]), float(q_gpu[r, c]), float(g["q"][r, c]))
              for r, c in over[:8]]
    assert over.size == 0, f"{what}: {len(over)} errors beyond 3 bf16 steps of the rotated pair " \
                           f"(row, col, out, ref, u_i, u_partner, q_gpu, q_golden): {detail}"
    print(f"{what}: max|diff| {d.max():.3e}, rel-L2 {rel:.2e}, {len(bad)} of {d.size} elements beyond 2e-2, "
          f"each explained by a one-step flip at a bf16 cast; q flips at the GEMM cast: {int(flips.sum())}; "
          f"elements beyond 2e-2 at (row, column): {[tuple(int(v) for v in x) for x in bad[:20]]}")
    return {"max_abs": float(d.max()), "rel_l2": rel, "beyond": int(len(bad)), "q_flips": int(flips.sum())}
