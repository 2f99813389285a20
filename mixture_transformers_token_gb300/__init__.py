"""MoT token-routed dense projection for GB300 (sm_103a): Python binding of libmot.so.

Argument marshalling only. Every step of the path -- routing pre-pass, fused add-RMSNorm,
routed GEMMs and their epilogues -- runs in the CUDA kernels of libmot.so, whose C ABI is
declared in include/mot.h. PyTorch provides device memory and streams. There is no CPU
fallback: a missing or stale library raises, and every nonzero status raises MotError.

Functions keep the C names. Tensors are contiguous CUDA tensors: bf16 for activations and
weights, uint8 for the modality index (0 = und, 1 = gen), int32 for positions, uint8 for
the workspace.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "MotError", "load_library", "library_path", "ABI_VERSION", "EPI_CAST", "EPI_SWIGLU",
    "DEV_BAD_MODALITY", "DEV_TIMEOUT", "DEV_PLAN_MISMATCH", "DEV_BAD_POSITION",
    "mot_abi_version", "mot_status_string", "mot_workspace_bytes", "mot_route_plan",
    "mot_fused_add_rmsnorm", "mot_routed_qkv_norm_rope", "mot_routed_gemm",
    "mot_swiglu_interleave", "mot_rope_table_fill_host", "mot_device_status", "mot_routed_gemm_noalloc",
    "mot_routed_qkv_norm_rope_fp32", "mot_rope_table_fill_host_fp32", "mot_add_rmsnorm_backward",
    "mot_rmsnorm_dweight", "mot_routed_gemm_dx", "mot_routed_gemm_dw", "mot_joint_attention", "DEV_BAD_SEQUENCE",
    "NOALLOC_MAX_TOKENS", "A_PLAN_ORDER", "OUT_PLAN_ORDER", "SET_UND", "SET_GEN", "SET_BOTH", "mot_gather_rows",
    "mot_selftest_wait_timeout",
    "DEV_BAD_TIME", "mot_flow_workspace_bytes", "mot_flow_schedule_host", "mot_cfg_combine_renorm",
    "mot_flow_sde_step", "mot_flow_cfg_sde_step", "mot_flow_noise",
]

ABI_VERSION = 4
EPI_CAST = 0
EPI_SWIGLU = 1
A_PLAN_ORDER = 0x100
OUT_PLAN_ORDER = 0x200
SET_UND, SET_GEN, SET_BOTH = 1, 2, 3  # weight-set masks of the norm backward's partials and fold
DEV_BAD_MODALITY = 0x1
DEV_TIMEOUT = 0x2
DEV_PLAN_MISMATCH = 0x4
DEV_BAD_POSITION = 0x8
DEV_BAD_SEQUENCE = 0x10
DEV_BAD_TIME = 0x20
NOALLOC_MAX_TOKENS = 65536

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None

_c_p = ctypes.c_void_p
_c_i64 = ctypes.c_int64
_c_i = ctypes.c_int
_c_f = ctypes.c_float
_c_sz = ctypes.c_size_t

_SIGNATURES = {
    "mot_abi_version": (_c_i, []),
    "mot_status_string": (ctypes.c_char_p, [_c_i]),
    "mot_workspace_bytes": (_c_sz, [_c_i64]),
    "mot_route_plan": (_c_i, [_c_p, _c_i64, _c_p, _c_sz, _c_p]),
    "mot_fused_add_rmsnorm": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i, _c_f, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "mot_routed_qkv_norm_rope": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i64, _c_i, _c_i, _c_i,
                                        _c_i, _c_f, _c_p, _c_sz, _c_p, _c_p]),
    "mot_routed_qkv_norm_rope_fp32": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i64, _c_i, _c_i,
                                             _c_i, _c_i, _c_f, _c_p, _c_sz, _c_p, _c_p]),
    "mot_routed_gemm": (_c_i, [_c_p, _c_p, _c_i64, _c_i, _c_i, _c_i, _c_p, _c_sz, _c_p, _c_p]),
    "mot_routed_gemm_noalloc": (_c_i, [_c_p, _c_p, _c_p, _c_i64, _c_i, _c_i, _c_i, _c_p, _c_p, _c_p]),
    "mot_swiglu_interleave": (_c_i, [_c_p, _c_p, _c_i, _c_i, _c_p, _c_p]),
    "mot_gather_rows": (_c_i, [_c_p, _c_i64, _c_i, _c_p, _c_sz, _c_p, _c_p]),
    "mot_selftest_wait_timeout": (_c_i, [_c_p, _c_sz, _c_p]),
    "mot_rope_table_fill_host": (_c_i, [ctypes.c_double, _c_i, _c_i, _c_p]),
    "mot_rope_table_fill_host_fp32": (_c_i, [ctypes.c_double, _c_i, _c_i, _c_p]),
    "mot_add_rmsnorm_backward": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i, _c_f, _c_p, _c_sz, _c_p, _c_p, _c_p,
                                        _c_i, _c_p]),
    "mot_rmsnorm_dweight": (_c_i, [_c_p, _c_i64, _c_i, _c_i, _c_p, _c_sz, _c_p, _c_p]),
    "mot_routed_gemm_dx": (_c_i, [_c_p, _c_p, _c_i64, _c_i, _c_i, _c_i, _c_p, _c_sz, _c_p, _c_p]),
    "mot_routed_gemm_dw": (_c_i, [_c_p, _c_p, _c_i64, _c_i, _c_i, _c_i, _c_i, _c_p, _c_sz, _c_p, _c_p]),
    "mot_joint_attention": (_c_i, [_c_p, _c_i64, _c_i, _c_i, _c_i, _c_p, _c_i, _c_f, _c_p, _c_sz, _c_p, _c_p]),
    "mot_flow_workspace_bytes": (_c_sz, [_c_i, _c_i64]),
    "mot_flow_schedule_host": (_c_i, [_c_i, ctypes.c_double, _c_p]),
    "mot_cfg_combine_renorm": (_c_i, [_c_p, _c_p, _c_p, _c_i, _c_i64, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "mot_flow_sde_step": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_i, _c_i64, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "mot_flow_cfg_sde_step": (_c_i, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i64, _c_p, _c_p, _c_sz,
                                     _c_p, _c_p, _c_p]),
    "mot_flow_noise": (_c_i, [_c_p, ctypes.c_uint64, _c_i, _c_i64, _c_p, _c_p]),
    "mot_device_status": (_c_i, [_c_p, ctypes.POINTER(ctypes.c_uint32), _c_p]),
}


class MotError(RuntimeError):
    """A nonzero status returned by libmot.so."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed with status {status}: {_lib().mot_status_string(status).decode()}")


def library_path() -> str:
    return os.environ.get("MOT_LIBRARY", os.path.join(_PKG, "libmot.so"))


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads libmot.so and declares its C signatures; raises if it is missing or stale."""
    path = path or library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -m mixture_transformers_token_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.mot_abi_version() != ABI_VERSION:
        raise ImportError(f"{path} has ABI {lib.mot_abi_version()}, the binding expects {ABI_VERSION}")
    return lib


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MotError(fn, status)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int | None = None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")
    return t.data_ptr()


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def mot_abi_version() -> int:
    return _lib().mot_abi_version()


def mot_status_string(status: int) -> str:
    return _lib().mot_status_string(status).decode()


def mot_workspace_bytes(T: int) -> int:
    return int(_lib().mot_workspace_bytes(T))


def mot_route_plan(mod: torch.Tensor, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Builds the routing plan of `mod` in `ws` (allocated if None) and returns ws."""
    T = mod.numel()
    _dev(mod, "mod", torch.uint8, 1)
    if ws is None:
        ws = torch.empty(max(mot_workspace_bytes(T), 16), dtype=torch.uint8, device=mod.device)
    _dev(ws, "ws", torch.uint8, 1)
    _check("mot_route_plan", _lib().mot_route_plan(mod.data_ptr(), T, ws.data_ptr(), ws.numel(), _stream(mod, stream)))
    return ws


def mot_fused_add_rmsnorm(x, res, w, mod, eps: float, y=None, res_out=None, ws=None, stream=None):
    """Residual add and routed RMSNorm; returns (y, res_out). res_out may be res (in place).
    If `ws` is given, the same launch also writes the routing plan of `mod` into it."""
    T, H = x.shape
    if y is None:
        y = torch.empty_like(x)
    if res_out is None:
        res_out = torch.empty_like(res)
    for t, n in ((x, "x"), (res, "res"), (y, "y"), (res_out, "res_out")):
        _dev(t, n, torch.bfloat16, 2)
        if tuple(t.shape) != (T, H):
            raise ValueError(f"{n} must be [{T}, {H}]")
    _dev(w, "w", torch.bfloat16, 2)
    _dev(mod, "mod", torch.uint8, 1)
    if tuple(w.shape) != (2, H) or mod.numel() != T:
        raise ValueError("w must be [2, H] and mod [T]")
    wsp = _dev(ws, "ws", torch.uint8, 1) if ws is not None else None
    wsb = ws.numel() if ws is not None else 0
    _check("mot_fused_add_rmsnorm", _lib().mot_fused_add_rmsnorm(
        x.data_ptr(), res.data_ptr(), w.data_ptr(), mod.data_ptr(), T, H, eps, y.data_ptr(), res_out.data_ptr(),
        wsp, wsb, _stream(x, stream)))
    return y, res_out


def mot_routed_qkv_norm_rope(x, w_qkv, q_norm_w, k_norm_w, pos, rope_cs, Hq: int, Hkv: int, D: int, eps: float,
                             ws, b_qkv=None, out=None, stream=None):
    """Routed QKV GEMM + per-head QK RMSNorm + RoPE; `ws` must hold the plan for T rows.
    A bf16 `rope_cs` selects the BF16 RoPE profile (mot_routed_qkv_norm_rope), an fp32 one
    the FP32 profile (mot_routed_qkv_norm_rope_fp32)."""
    T, H = x.shape
    N = (Hq + 2 * Hkv) * D
    _dev(x, "x", torch.bfloat16, 2)
    _dev(w_qkv, "w_qkv", torch.bfloat16, 3)
    _dev(q_norm_w, "q_norm_w", torch.bfloat16, 2)
    _dev(k_norm_w, "k_norm_w", torch.bfloat16, 2)
    _dev(pos, "pos", torch.int32, 1)
    fp32 = rope_cs.dtype == torch.float32
    _dev(rope_cs, "rope_cs", torch.float32 if fp32 else torch.bfloat16, 3)
    _dev(ws, "ws", torch.uint8, 1)
    if tuple(w_qkv.shape) != (2, N, H):
        raise ValueError(f"w_qkv must be [2, {N}, {H}]")
    if tuple(q_norm_w.shape) != (2, D) or tuple(k_norm_w.shape) != (2, D) or pos.numel() != T:
        raise ValueError("q_norm_w/k_norm_w must be [2, D] and pos [T]")
    if rope_cs.shape[1:] != (D // 2, 2):
        raise ValueError("rope_cs must be [P, D/2, 2]")
    bp = None
    if b_qkv is not None:
        bp = _dev(b_qkv, "b_qkv", torch.bfloat16, 2)
        if tuple(b_qkv.shape) != (2, N):
            raise ValueError(f"b_qkv must be [2, {N}]")
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    _dev(out, "out", torch.bfloat16, 2)
    name = "mot_routed_qkv_norm_rope_fp32" if fp32 else "mot_routed_qkv_norm_rope"
    _check(name, getattr(_lib(), name)(
        x.data_ptr(), w_qkv.data_ptr(), bp, q_norm_w.data_ptr(), k_norm_w.data_ptr(), pos.data_ptr(),
        rope_cs.data_ptr(), rope_cs.shape[0], T, H, Hq, Hkv, D, eps, ws.data_ptr(), ws.numel(), out.data_ptr(),
        _stream(x, stream)))
    return out


def mot_routed_qkv_norm_rope_fp32(x, w_qkv, q_norm_w, k_norm_w, pos, rope_cs_f32, Hq: int, Hkv: int, D: int,
                                  eps: float, ws, b_qkv=None, out=None, stream=None):
    """The FP32 RoPE profile of mot_routed_qkv_norm_rope; `rope_cs_f32` is the fp32 table."""
    if rope_cs_f32.dtype != torch.float32:
        raise TypeError("rope_cs_f32 must be float32 (mot_rope_table_fill_host_fp32)")
    return mot_routed_qkv_norm_rope(x, w_qkv, q_norm_w, k_norm_w, pos, rope_cs_f32, Hq, Hkv, D, eps, ws,
                                    b_qkv=b_qkv, out=out, stream=stream)


def mot_routed_gemm(a, w, ws, epilogue: int = EPI_CAST, out=None, stream=None):
    """Routed GEMM: out[T][N] = bf16(a W^T) (cast) or out[T][N/2] = SwiGLU (interleaved gate/up w).
    `epilogue` may carry A_PLAN_ORDER / OUT_PLAN_ORDER (rows of a / out in the plan's order)."""
    T, K = a.shape
    _dev(a, "a", torch.bfloat16, 2)
    _dev(w, "w", torch.bfloat16, 3)
    _dev(ws, "ws", torch.uint8, 1)
    if w.shape[0] != 2 or w.shape[2] != K:
        raise ValueError("w must be [2, N, K]")
    N = w.shape[1]
    ncols = N // 2 if (epilogue & 0xFF) == EPI_SWIGLU else N
    if out is None:
        out = torch.empty((T, ncols), dtype=torch.bfloat16, device=a.device)
    _dev(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (T, ncols):
        raise ValueError(f"out must be [{T}, {ncols}]")
    _check("mot_routed_gemm", _lib().mot_routed_gemm(
        a.data_ptr(), w.data_ptr(), T, N, K, epilogue, ws.data_ptr(), ws.numel(), out.data_ptr(), _stream(a, stream)))
    return out


def mot_routed_gemm_noalloc(a, w, mod, epilogue: int = EPI_CAST, out=None, device_flags=None, stream=None):
    """mot_routed_gemm for callers that cannot allocate device memory: the routing plan is kept
    in the library's own fixed device array (T <= NOALLOC_MAX_TOKENS), so no workspace is
    passed. Calls whose work may overlap on the GPU share that array and must be ordered by
    the caller. `device_flags`, an optional int32 CUDA tensor of one element, receives the
    call's device error bits."""
    T, K = a.shape
    _dev(a, "a", torch.bfloat16, 2)
    _dev(w, "w", torch.bfloat16, 3)
    _dev(mod, "mod", torch.uint8, 1)
    if w.shape[0] != 2 or w.shape[2] != K or mod.numel() != T:
        raise ValueError("w must be [2, N, K] and mod [T]")
    N = w.shape[1]
    ncols = N // 2 if epilogue == EPI_SWIGLU else N
    if out is None:
        out = torch.empty((T, ncols), dtype=torch.bfloat16, device=a.device)
    _dev(out, "out", torch.bfloat16, 2)
    fp = _dev(device_flags, "device_flags", torch.int32, 1) if device_flags is not None else None
    _check("mot_routed_gemm_noalloc", _lib().mot_routed_gemm_noalloc(
        a.data_ptr(), w.data_ptr(), mod.data_ptr(), T, N, K, epilogue, out.data_ptr(), fp, _stream(a, stream)))
    return out


def mot_gather_rows(src, ws, out=None, stream=None):
    """Rows of src [T][K] in the plan's order (und rows ascending, then gen rows)."""
    T, K = src.shape
    _dev(src, "src", torch.bfloat16, 2)
    _dev(ws, "ws", torch.uint8, 1)
    if out is None:
        out = torch.empty_like(src)
    _dev(out, "out", torch.bfloat16, 2)
    _check("mot_gather_rows", _lib().mot_gather_rows(src.data_ptr(), T, K, ws.data_ptr(), ws.numel(), out.data_ptr(),
                                                     _stream(src, stream)))
    return out


def mot_swiglu_interleave(w_gate, w_up, out=None, stream=None):
    """[2][I][K] gate and up weights -> [2][2I][K] interleaved in 128-row blocks."""
    _dev(w_gate, "w_gate", torch.bfloat16, 3)
    _dev(w_up, "w_up", torch.bfloat16, 3)
    _, I, K = w_gate.shape
    if tuple(w_up.shape) != (2, I, K):
        raise ValueError("w_up must match w_gate")
    if out is None:
        out = torch.empty((2, 2 * I, K), dtype=torch.bfloat16, device=w_gate.device)
    _dev(out, "out", torch.bfloat16, 3)
    _check("mot_swiglu_interleave", _lib().mot_swiglu_interleave(
        w_gate.data_ptr(), w_up.data_ptr(), I, K, out.data_ptr(), _stream(w_gate, stream)))
    return out


def mot_routed_gemm_dx(dout, w, ws, flags: int = 0, out=None, stream=None):
    """Input gradient of the routed GEMM through both weight sets: dx[T][K] = bf16(dout W[mod]).
    `w` is the forward's [2][N][K] weight; `flags` may carry A_PLAN_ORDER / OUT_PLAN_ORDER."""
    T, N = dout.shape
    _dev(dout, "dout", torch.bfloat16, 2)
    _dev(w, "w", torch.bfloat16, 3)
    _dev(ws, "ws", torch.uint8, 1)
    if w.shape[0] != 2 or w.shape[1] != N:
        raise ValueError(f"w must be [2, {N}, K]")
    K = w.shape[2]
    if out is None:
        out = torch.empty((T, K), dtype=torch.bfloat16, device=dout.device)
    _dev(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (T, K):
        raise ValueError(f"out must be [{T}, {K}]")
    _check("mot_routed_gemm_dx", _lib().mot_routed_gemm_dx(
        dout.data_ptr(), w.data_ptr(), T, N, K, flags, ws.data_ptr(), ws.numel(), out.data_ptr(),
        _stream(dout, stream)))
    return out


def mot_routed_gemm_dw(dout, a, ws, expert: int = 1, flags: int = 0, out=None, stream=None):
    """Gradient [N][K] fp32 of weight set `expert` from dout [T][N] and a [T][K]: rows in token
    order, or in the plan's order with flags = A_PLAN_ORDER (the same bits either way)."""
    T, N = dout.shape
    _dev(dout, "dout", torch.bfloat16, 2)
    _dev(a, "a", torch.bfloat16, 2)
    _dev(ws, "ws", torch.uint8, 1)
    if a.shape[0] != T:
        raise ValueError("dout and a must have the same rows")
    K = a.shape[1]
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=dout.device)
    _dev(out, "out", torch.float32, 2)
    if tuple(out.shape) != (N, K):
        raise ValueError(f"out must be [{N}, {K}]")
    _check("mot_routed_gemm_dw", _lib().mot_routed_gemm_dw(
        dout.data_ptr(), a.data_ptr(), T, N, K, expert, flags, ws.data_ptr(), ws.numel(), out.data_ptr(),
        _stream(dout, stream)))
    return out


def mot_joint_attention(qkv, seqs, Hq: int, Hkv: int, D: int, ws, scale: float | None = None, out=None,
                        stream=None):
    """Attention of packed sequences over the fused QKV output [T][(Hq + 2 Hkv) D].
    `seqs` is a device int32 [n_seq][5] of (q_start, k_start, nq, nk, n_causal); `ws` (>= 64
    bytes) receives device errors. Returns out [T][Hq D] (rows that are no query untouched)."""
    T = qkv.shape[0]
    _dev(qkv, "qkv", torch.bfloat16, 2)
    _dev(seqs, "seqs", torch.int32, 2)
    _dev(ws, "ws", torch.uint8, 1)
    if qkv.shape[1] != (Hq + 2 * Hkv) * D:
        raise ValueError(f"qkv must be [T, {(Hq + 2 * Hkv) * D}]")
    if seqs.shape[1] != 5:
        raise ValueError("seqs must be [n_seq, 5]")
    if out is None:
        out = torch.zeros((T, Hq * D), dtype=torch.bfloat16, device=qkv.device)
    _dev(out, "out", torch.bfloat16, 2)
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check("mot_joint_attention", _lib().mot_joint_attention(
        qkv.data_ptr(), T, Hq, Hkv, D, seqs.data_ptr(), seqs.shape[0], sc, ws.data_ptr(), ws.numel(),
        out.data_ptr(), _stream(qkv, stream)))
    return out


def mot_add_rmsnorm_backward(dy, s, w, eps: float, ws, d_res_out=None, dx=None, rstd=None, dw_partials=None,
                             partial_sets: int = SET_BOTH, stream=None):
    """Input gradient of the fused add-RMSNorm: returns (dx [T][H] bf16, rstd [T] fp32).
    `s` is the forward's res_out and `ws` holds the routing plan of the forward's mod. If
    `dw_partials` (fp32 [H/64][T][64]) is given, the per-row weight-gradient partials of the
    rows of the weight sets in `partial_sets` are written there in the plan's row order."""
    T, H = dy.shape
    _dev(dy, "dy", torch.bfloat16, 2)
    _dev(s, "s", torch.bfloat16, 2)
    _dev(w, "w", torch.bfloat16, 2)
    _dev(ws, "ws", torch.uint8, 1)
    if tuple(s.shape) != (T, H) or tuple(w.shape) != (2, H):
        raise ValueError("s must be [T, H] and w [2, H]")
    rp = None
    if d_res_out is not None:
        _dev(d_res_out, "d_res_out", torch.bfloat16, 2)
        if tuple(d_res_out.shape) != (T, H):
            raise ValueError("d_res_out must be [T, H]")
        rp = d_res_out.data_ptr()
    pp = None
    if dw_partials is not None:
        _dev(dw_partials, "dw_partials", torch.float32, 3)
        if tuple(dw_partials.shape) != (H // 64, T, 64):
            raise ValueError(f"dw_partials must be [{H // 64}, {T}, 64]")
        pp = dw_partials.data_ptr()
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.bfloat16, device=dy.device)
    if rstd is None:
        rstd = torch.empty((T,), dtype=torch.float32, device=dy.device)
    _dev(dx, "dx", torch.bfloat16, 2)
    _dev(rstd, "rstd", torch.float32, 1)
    _check("mot_add_rmsnorm_backward", _lib().mot_add_rmsnorm_backward(
        dy.data_ptr(), rp, s.data_ptr(), w.data_ptr(), T, H, eps, ws.data_ptr(), ws.numel(), dx.data_ptr(),
        rstd.data_ptr(), pp, partial_sets, _stream(dy, stream)))
    return dx, rstd


def mot_rmsnorm_dweight(dw_partials, ws, dw=None, sets: int = SET_BOTH, stream=None):
    """Gradient of the norm weight sets in `sets`, rows of dw [2][H] fp32: the ascending-row fp32
    left fold of the partials of mot_add_rmsnorm_backward over each set's rows (the other set's
    row of dw is left as it is)."""
    nb, T, c64 = dw_partials.shape
    _dev(dw_partials, "dw_partials", torch.float32, 3)
    _dev(ws, "ws", torch.uint8, 1)
    if c64 != 64:
        raise ValueError("dw_partials must be [H/64, T, 64]")
    H = nb * 64
    if dw is None:
        dw = torch.empty((2, H), dtype=torch.float32, device=dw_partials.device)
    _dev(dw, "dw", torch.float32, 2)
    _check("mot_rmsnorm_dweight", _lib().mot_rmsnorm_dweight(
        dw_partials.data_ptr(), T, H, sets, ws.data_ptr(), ws.numel(), dw.data_ptr(), _stream(dw_partials, stream)))
    return dw


def mot_rope_table_fill_host(theta: float, D: int, P: int) -> torch.Tensor:
    """Host (cos, sin) table [P][D/2][2] as a CPU bf16 tensor (copy it to the device once)."""
    t = torch.empty((P, D // 2, 2), dtype=torch.bfloat16)
    _check("mot_rope_table_fill_host", _lib().mot_rope_table_fill_host(theta, D, P, t.data_ptr()))
    return t


def mot_rope_table_fill_host_fp32(theta: float, D: int, P: int) -> torch.Tensor:
    """Host fp32 (cos, sin) table [P][D/2][2] of the FP32 RoPE profile, as a CPU tensor."""
    t = torch.empty((P, D // 2, 2), dtype=torch.float32)
    _check("mot_rope_table_fill_host_fp32", _lib().mot_rope_table_fill_host_fp32(theta, D, P, t.data_ptr()))
    return t


def mot_flow_workspace_bytes(n_req: int, N: int) -> int:
    return int(_lib().mot_flow_workspace_bytes(n_req, N))


def mot_flow_schedule_host(n: int, shift: float) -> torch.Tensor:
    """The sampler's n step times from 1 down to 0 (built in double, stored fp32), a CPU tensor."""
    t = torch.empty((n,), dtype=torch.float32)
    _check("mot_flow_schedule_host", _lib().mot_flow_schedule_host(n, shift, t.data_ptr()))
    return t


def _flow_ws(ws, n_req: int, N: int, device) -> torch.Tensor:
    if ws is None:
        ws = torch.zeros(max(mot_flow_workspace_bytes(n_req, N), 64), dtype=torch.uint8, device=device)
    _dev(ws, "ws", torch.uint8, 1)
    return ws


def mot_cfg_combine_renorm(v_c, v_tu, v_iu, policy, ws=None, out=None, stream=None):
    """Three-branch renormalised CFG per request: v_c, v_tu, v_iu (or None) [n_req][N] bf16,
    policy a device fp32 [n_req][6] of (t, s_text, s_img, t_lo, t_hi, renorm_min). `ws` (>=
    mot_flow_workspace_bytes) is scratch after its 64-byte header. Returns out [n_req][N] fp32."""
    n_req, N = v_c.shape
    _dev(v_c, "v_c", torch.bfloat16, 2)
    _dev(v_tu, "v_tu", torch.bfloat16, 2)
    ip = None
    if v_iu is not None:
        _dev(v_iu, "v_iu", torch.bfloat16, 2)
        ip = v_iu.data_ptr()
    _dev(policy, "policy", torch.float32, 2)
    if tuple(v_tu.shape) != (n_req, N) or (v_iu is not None and tuple(v_iu.shape) != (n_req, N)):
        raise ValueError("the branches must all be [n_req, N]")
    if tuple(policy.shape) != (n_req, 6):
        raise ValueError("policy must be [n_req, 6]")
    ws = _flow_ws(ws, n_req, N, v_c.device)
    if out is None:
        out = torch.empty((n_req, N), dtype=torch.float32, device=v_c.device)
    _dev(out, "out", torch.float32, 2)
    _check("mot_cfg_combine_renorm", _lib().mot_cfg_combine_renorm(
        v_c.data_ptr(), v_tu.data_ptr(), ip, n_req, N, policy.data_ptr(), ws.data_ptr(), ws.numel(),
        out.data_ptr(), _stream(v_c, stream)))
    return out


def mot_flow_sde_step(x, v, z, times, ws=None, x_next=None, logp=None, stream=None):
    """One reverse-SDE step per request and its log-probability: x, v, z [n_req][N] fp32, times
    a device fp32 [n_req][2] of (t_i, t_next). With z None, x_next must be given and is scored
    instead of sampled. `ws`'s error word receives DEV_BAD_TIME. Returns (x_next, logp [n_req])."""
    n_req, N = x.shape
    _dev(x, "x", torch.float32, 2)
    _dev(v, "v", torch.float32, 2)
    _dev(times, "times", torch.float32, 2)
    if tuple(v.shape) != (n_req, N) or tuple(times.shape) != (n_req, 2):
        raise ValueError("v must be [n_req, N] and times [n_req, 2]")
    zp = None
    if z is not None:
        _dev(z, "z", torch.float32, 2)
        if tuple(z.shape) != (n_req, N):
            raise ValueError("z must be [n_req, N]")
        zp = z.data_ptr()
    elif x_next is None:
        raise ValueError("either z or x_next must be given")
    ws = _flow_ws(ws, n_req, N, x.device)
    if x_next is None:
        x_next = torch.empty((n_req, N), dtype=torch.float32, device=x.device)
    _dev(x_next, "x_next", torch.float32, 2)
    if tuple(x_next.shape) != (n_req, N):
        raise ValueError("x_next must be [n_req, N]")
    if logp is None:
        logp = torch.empty((n_req,), dtype=torch.float32, device=x.device)
    _dev(logp, "logp", torch.float32, 1)
    _check("mot_flow_sde_step", _lib().mot_flow_sde_step(
        x.data_ptr(), v.data_ptr(), zp, x_next.data_ptr(), n_req, N, times.data_ptr(), ws.data_ptr(), ws.numel(),
        logp.data_ptr(), _stream(x, stream)))
    return x_next, logp


def mot_flow_cfg_sde_step(v_c, v_tu, v_iu, policy, x, z, times, ws=None, x_next=None, v_out=None, logp=None,
                          stream=None):
    """CFG combine + renorm and the SDE step in one call, without writing the guided velocity:
    the branches and policy as for mot_cfg_combine_renorm, x, z, times as for mot_flow_sde_step
    (z None: x_next is given and scored). v_out, if given ([n_req][N] fp32), receives the guided
    velocity. Returns (x_next, logp), bit for bit those of the two calls in sequence."""
    n_req, N = v_c.shape
    _dev(v_c, "v_c", torch.bfloat16, 2)
    _dev(v_tu, "v_tu", torch.bfloat16, 2)
    ip = None
    if v_iu is not None:
        _dev(v_iu, "v_iu", torch.bfloat16, 2)
        ip = v_iu.data_ptr()
    _dev(policy, "policy", torch.float32, 2)
    _dev(x, "x", torch.float32, 2)
    _dev(times, "times", torch.float32, 2)
    if tuple(v_tu.shape) != (n_req, N) or (v_iu is not None and tuple(v_iu.shape) != (n_req, N)) \
            or tuple(x.shape) != (n_req, N):
        raise ValueError("the branches and x must all be [n_req, N]")
    if tuple(policy.shape) != (n_req, 6) or tuple(times.shape) != (n_req, 2):
        raise ValueError("policy must be [n_req, 6] and times [n_req, 2]")
    zp = None
    if z is not None:
        _dev(z, "z", torch.float32, 2)
        if tuple(z.shape) != (n_req, N):
            raise ValueError("z must be [n_req, N]")
        zp = z.data_ptr()
    elif x_next is None:
        raise ValueError("either z or x_next must be given")
    ws = _flow_ws(ws, n_req, N, x.device)
    if x_next is None:
        x_next = torch.empty((n_req, N), dtype=torch.float32, device=x.device)
    _dev(x_next, "x_next", torch.float32, 2)
    if tuple(x_next.shape) != (n_req, N):
        raise ValueError("x_next must be [n_req, N]")
    vp = None
    if v_out is not None:
        _dev(v_out, "v_out", torch.float32, 2)
        if tuple(v_out.shape) != (n_req, N):
            raise ValueError("v_out must be [n_req, N]")
        vp = v_out.data_ptr()
    if logp is None:
        logp = torch.empty((n_req,), dtype=torch.float32, device=x.device)
    _dev(logp, "logp", torch.float32, 1)
    _check("mot_flow_cfg_sde_step", _lib().mot_flow_cfg_sde_step(
        v_c.data_ptr(), v_tu.data_ptr(), ip, policy.data_ptr(), x.data_ptr(), zp, x_next.data_ptr(), n_req, N,
        times.data_ptr(), ws.data_ptr(), ws.numel(), vp, logp.data_ptr(), _stream(x, stream)))
    return x_next, logp


def mot_flow_noise(seeds, step: int, N: int, z=None, stream=None):
    """Per-sample standard normal noise [n_req][N] fp32 of sampler step `step`: `seeds` is a
    device int64 tensor [n_req] (reinterpreted as uint64), one seed per request."""
    _dev(seeds, "seeds", torch.int64, 1)
    n_req = seeds.shape[0]
    if z is None:
        z = torch.empty((n_req, N), dtype=torch.float32, device=seeds.device)
    _dev(z, "z", torch.float32, 2)
    if tuple(z.shape) != (n_req, N):
        raise ValueError(f"z must be [{n_req}, {N}]")
    _check("mot_flow_noise", _lib().mot_flow_noise(seeds.data_ptr(), int(step) & (2 ** 64 - 1), n_req, N,
                                                   z.data_ptr(), _stream(seeds, stream)))
    return z


def mot_selftest_wait_timeout(ws, stream=None) -> None:
    """Runs a bounded wait that nothing satisfies; afterwards ws's error word has DEV_TIMEOUT."""
    _dev(ws, "ws", torch.uint8, 1)
    _check("mot_selftest_wait_timeout", _lib().mot_selftest_wait_timeout(ws.data_ptr(), ws.numel(), _stream(ws, stream)))


def mot_device_status(ws, stream=None) -> int:
    """Synchronizes the stream and returns the workspace's device error bits (0 = clean)."""
    _dev(ws, "ws", torch.uint8, 1)
    flags = ctypes.c_uint32(0)
    _check("mot_device_status", _lib().mot_device_status(ws.data_ptr(), ctypes.byref(flags), _stream(ws, stream)))
    return int(flags.value)
