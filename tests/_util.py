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
