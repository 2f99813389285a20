"""Host-side tests of the C-ABI library (no GPU needed).

The library must load on a machine without a GPU, export every entry point that
include/mot.h declares, and reject invalid arguments before touching CUDA. The host-side
RoPE table builder is compared with the oracle's table bit for bit.
"""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import build as mot_build
from oracle import mot_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mot.h")

MOT_OK, MOT_ERR_NULL, MOT_ERR_ALIGN, MOT_ERR_GEOMETRY = 0, 1, 2, 3
MOT_ERR_DEVICE, MOT_ERR_WORKSPACE, MOT_ERR_ARCH, MOT_ERR_CUDA, MOT_ERR_ARG = 4, 5, 6, 7, 8


@pytest.fixture(scope="module")
def lib():
    mot_build.build()
    return mot.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mot_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("mot_fused_add_rmsnorm", "mot_routed_qkv_norm_rope", "mot_routed_gemm", "mot_route_plan",
                     "mot_workspace_bytes", "mot_abi_version", "mot_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version_and_status_strings(lib):
    assert lib.mot_abi_version() == mot.ABI_VERSION
    seen = set()
    for code in range(0, 10):
        s = lib.mot_status_string(code).decode()
        assert s and s not in seen
        seen.add(s)
    assert lib.mot_status_string(1234).decode() == "unknown status"


def test_workspace_bytes(lib):
    assert lib.mot_workspace_bytes(0) == 0
    assert lib.mot_workspace_bytes(-5) == 0
    assert lib.mot_workspace_bytes((1 << 24) + 1) == 0
    prev = 0
    for T in (1, 2, 127, 128, 129, 4096, 36864):
        b = lib.mot_workspace_bytes(T)
        # header + one int32 per row + one 16-byte tile record per 128 rows (+1)
        assert b >= 64 + 4 * T + 16 * ((T + 127) // 128 + 1)
        assert b % 16 == 0 and b >= prev
        prev = b


# fake, 16-byte aligned, non-NULL addresses: every check below fails before any CUDA call
A = 1 << 20
B = 2 << 20
C = 3 << 20
MIS = (4 << 20) + 8


def test_route_plan_rejects(lib):
    assert lib.mot_route_plan(None, 10, A, 1 << 20, None) == MOT_ERR_NULL
    assert lib.mot_route_plan(A, 0, B, 1 << 20, None) == MOT_ERR_GEOMETRY
    assert lib.mot_route_plan(A, (1 << 24) + 1, B, 1 << 30, None) == MOT_ERR_GEOMETRY
    assert lib.mot_route_plan(A, 10, MIS, 1 << 20, None) == MOT_ERR_ALIGN
    assert lib.mot_route_plan(A, 1000, B, 100, None) == MOT_ERR_WORKSPACE


def test_add_rmsnorm_rejects(lib):
    f = lib.mot_fused_add_rmsnorm
    assert f(None, A, A, A, 4, 256, 1e-6, B, C, None, 0, None) == MOT_ERR_NULL
    assert f(A, A, A, A, 4, 255, 1e-6, B, C, None, 0, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, A, 4, 128, 1e-6, B, C, None, 0, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, A, 4, 8448, 1e-6, B, C, None, 0, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, A, 0, 256, 1e-6, B, C, None, 0, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, A, 4, 256, 0.0, B, C, None, 0, None) == MOT_ERR_ARG
    assert f(A, A, A, A, 4, 256, float("nan"), B, C, None, 0, None) == MOT_ERR_ARG
    assert f(MIS, A, A, A, 4, 256, 1e-6, B, C, None, 0, None) == MOT_ERR_ALIGN
    assert f(A, A, A, A, 4, 256, 1e-6, B, MIS, None, 0, None) == MOT_ERR_ALIGN
    assert f(A, A, A, A, 4, 256, 1e-6, B, C, MIS, 1 << 20, None) == MOT_ERR_ALIGN
    assert f(A, A, A, A, 1000, 256, 1e-6, B, C, C, 100, None) == MOT_ERR_WORKSPACE


def test_qkv_rejects(lib):
    f = lib.mot_routed_qkv_norm_rope

    def call(**kw):
        a = dict(x=A, w=A, b=None, qn=A, kn=A, pos=A, cs=A, P=64, T=64, H=256, Hq=4, Hkv=2, D=64, eps=1e-6, ws=B,
                 wsb=1 << 20, out=C)
        a.update(kw)
        return f(a["x"], a["w"], a["b"], a["qn"], a["kn"], a["pos"], a["cs"], a["P"], a["T"], a["H"], a["Hq"],
                 a["Hkv"], a["D"], a["eps"], a["ws"], a["wsb"], a["out"], None)

    assert call(x=None) == MOT_ERR_NULL
    assert call(ws=None) == MOT_ERR_NULL
    assert call(D=96) == MOT_ERR_GEOMETRY
    assert call(Hq=3, Hkv=1, D=64) == MOT_ERR_GEOMETRY          # N = 320 is not a multiple of 256
    assert call(H=200) == MOT_ERR_GEOMETRY
    assert call(T=0) == MOT_ERR_GEOMETRY
    assert call(P=0) == MOT_ERR_ARG
    assert call(eps=-1.0) == MOT_ERR_ARG
    assert call(b=MIS) == MOT_ERR_ALIGN
    assert call(out=MIS) == MOT_ERR_ALIGN
    assert call(wsb=100) == MOT_ERR_WORKSPACE


def test_qkv_fp32_profile_rejects(lib):
    f = lib.mot_routed_qkv_norm_rope_fp32

    def call(**kw):
        a = dict(x=A, w=A, b=None, qn=A, kn=A, pos=A, cs=A, P=64, T=64, H=256, Hq=4, Hkv=2, D=64, eps=1e-6, ws=B,
                 wsb=1 << 20, out=C)
        a.update(kw)
        return f(a["x"], a["w"], a["b"], a["qn"], a["kn"], a["pos"], a["cs"], a["P"], a["T"], a["H"], a["Hq"],
                 a["Hkv"], a["D"], a["eps"], a["ws"], a["wsb"], a["out"], None)

    assert call(cs=None) == MOT_ERR_NULL
    assert call(cs=MIS) == MOT_ERR_ALIGN
    assert call(D=32) == MOT_ERR_GEOMETRY
    assert call(T=(1 << 24) + 1) == MOT_ERR_GEOMETRY
    assert call(P=0) == MOT_ERR_ARG
    assert call(eps=float("inf")) == MOT_ERR_ARG
    assert call(wsb=16) == MOT_ERR_WORKSPACE


def test_norm_backward_rejects(lib):
    f = lib.mot_add_rmsnorm_backward
    assert f(None, None, A, A, 8, 256, 1e-6, B, 1 << 20, C, C, None, 3, None) == MOT_ERR_NULL
    assert f(A, None, A, A, 8, 256, 1e-6, None, 1 << 20, C, C, None, 3, None) == MOT_ERR_NULL
    assert f(A, None, A, A, 8, 256, 1e-6, B, 1 << 20, C, None, None, 3, None) == MOT_ERR_NULL
    assert f(A, None, A, A, 8, 200, 1e-6, B, 1 << 20, C, C, None, 3, None) == MOT_ERR_GEOMETRY
    assert f(A, None, A, A, 8, 8448, 1e-6, B, 1 << 20, C, C, None, 3, None) == MOT_ERR_GEOMETRY
    assert f(A, None, A, A, 0, 256, 1e-6, B, 1 << 20, C, C, None, 3, None) == MOT_ERR_GEOMETRY
    assert f(A, None, A, A, 8, 256, 0.0, B, 1 << 20, C, C, None, 3, None) == MOT_ERR_ARG
    assert f(A, MIS, A, A, 8, 256, 1e-6, B, 1 << 20, C, C, None, 3, None) == MOT_ERR_ALIGN
    assert f(A, None, A, A, 8, 256, 1e-6, B, 1 << 20, C, MIS, None, 3, None) == MOT_ERR_ALIGN
    assert f(A, None, A, A, 8, 256, 1e-6, B, 1 << 20, C, C, MIS, 3, None) == MOT_ERR_ALIGN
    assert f(A, None, A, A, 1000, 256, 1e-6, B, 100, C, C, None, 3, None) == MOT_ERR_WORKSPACE
    # the partials' weight-set mask: MOT_SET_UND, MOT_SET_GEN or MOT_SET_BOTH; ignored without partials
    for bad in (0, 4, -1):
        assert f(A, None, A, A, 8, 256, 1e-6, B, 1 << 20, C, C, C, bad, None) == MOT_ERR_ARG
    assert f(A, None, A, A, 1000, 256, 1e-6, B, 100, C, C, None, 0, None) == MOT_ERR_WORKSPACE
    g = lib.mot_rmsnorm_dweight
    assert g(None, 8, 256, 3, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert g(A, 8, 255, 3, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert g(A, 8, 256, 3, MIS, 1 << 20, C, None) == MOT_ERR_ALIGN
    assert g(A, 1000, 256, 3, B, 100, C, None) == MOT_ERR_WORKSPACE
    for bad in (0, 4, -1):
        assert g(A, 8, 256, bad, B, 1 << 20, C, None) == MOT_ERR_ARG


def test_gemm_backward_rejects(lib):
    dx = lib.mot_routed_gemm_dx
    assert dx(None, A, 8, 64, 256, 0, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert dx(A, A, 8, 64, 256, 0x1, B, 1 << 20, C, None) == MOT_ERR_ARG          # no epilogue bits
    assert dx(A, A, 8, 64, 320, 0, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY       # output K % 256
    assert dx(A, A, 8, 96, 256, 0, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY       # reduction N % 64
    assert dx(A, MIS, 8, 64, 256, 0, B, 1 << 20, C, None) == MOT_ERR_ALIGN
    assert dx(A, A, 1000, 64, 256, 0, B, 100, C, None) == MOT_ERR_WORKSPACE
    dw = lib.mot_routed_gemm_dw
    assert dw(None, A, 8, 256, 256, 1, 0, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert dw(A, A, 8, 256, 256, 2, 0, B, 1 << 20, C, None) == MOT_ERR_ARG
    assert dw(A, A, 8, 256, 256, 1, 0x200, B, 1 << 20, C, None) == MOT_ERR_ARG     # only MOT_A_PLAN_ORDER
    assert dw(A, A, 8, 128, 256, 1, 0, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert dw(A, A, 8, 256, 320, 1, 0x100, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert dw(A, A, 8, 256, 256, 1, 0, B, 1 << 20, MIS, None) == MOT_ERR_ALIGN
    assert dw(A, A, 1000, 256, 256, 1, 0, B, 100, C, None) == MOT_ERR_WORKSPACE


def test_joint_attention_rejects(lib):
    f = lib.mot_joint_attention
    assert f(None, 64, 4, 2, 64, A, 1, 0.125, B, 64, C, None) == MOT_ERR_NULL
    assert f(A, 64, 4, 2, 64, None, 1, 0.125, B, 64, C, None) == MOT_ERR_NULL
    assert f(A, 64, 4, 2, 96, A, 1, 0.125, B, 64, C, None) == MOT_ERR_GEOMETRY      # D
    assert f(A, 64, 4, 3, 64, A, 1, 0.125, B, 64, C, None) == MOT_ERR_GEOMETRY      # Hq % Hkv
    assert f(A, 0, 4, 2, 64, A, 1, 0.125, B, 64, C, None) == MOT_ERR_GEOMETRY
    assert f(A, 64, 4, 2, 64, A, 0, 0.125, B, 64, C, None) == MOT_ERR_GEOMETRY      # no sequence
    assert f(A, 64, 4, 2, 64, A, 1, 0.0, B, 64, C, None) == MOT_ERR_ARG
    assert f(A, 64, 4, 2, 64, MIS, 1, 0.125, B, 64, C, None) == MOT_ERR_ALIGN
    assert f(A, 64, 4, 2, 64, A, 1, 0.125, B, 8, C, None) == MOT_ERR_WORKSPACE


def test_routed_gemm_rejects(lib):
    f = lib.mot_routed_gemm
    assert f(None, A, 8, 256, 64, 0, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, A, 8, 256, 64, 7, B, 1 << 20, C, None) == MOT_ERR_ARG
    assert f(A, A, 8, 320, 64, 0, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, 8, 256, 96, 0, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, 0, 256, 64, 0, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, MIS, 8, 256, 64, 0, B, 1 << 20, C, None) == MOT_ERR_ALIGN
    assert f(A, A, 8, 256, 64, 0, B, 10, C, None) == MOT_ERR_WORKSPACE


def test_noalloc_rejects_before_touching_cuda(lib):
    f = lib.mot_routed_gemm_noalloc
    assert f(None, A, A, 8, 256, 64, 0, C, None, None) == MOT_ERR_NULL
    assert f(A, A, A, 65537, 256, 64, 0, C, None, None) == 9          # above the scratch limit
    assert "MOT_NOALLOC_MAX_TOKENS" in lib.mot_status_string(9).decode()
    assert f(A, A, A, 0, 256, 64, 0, C, None, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, 8, 320, 64, 0, C, None, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, 8, 256, 64, 5, C, None, None) == MOT_ERR_ARG
    assert f(MIS, A, A, 8, 256, 64, 0, C, None, None) == MOT_ERR_ALIGN


def test_gather_rows_rejects(lib):
    f = lib.mot_gather_rows
    assert f(None, 10, 64, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, 10, 60, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, 0, 64, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, 10, 64, MIS, 1 << 20, C, None) == MOT_ERR_ALIGN
    assert f(A, 1000, 64, B, 100, C, None) == MOT_ERR_WORKSPACE
    assert f(A, 10, 64, B, 1 << 20, A, None) == MOT_ERR_ARG


def test_routed_gemm_order_flags_checked(lib):
    assert lib.mot_routed_gemm(A, A, 8, 256, 64, 0x400, B, 1 << 20, C, None) == MOT_ERR_ARG
    assert lib.mot_routed_gemm(A, A, 8, 256, 64, 0x2 | 0x100, B, 1 << 20, C, None) == MOT_ERR_ARG


def test_selftest_rejects(lib):
    assert lib.mot_selftest_wait_timeout(None, 64, None) == MOT_ERR_NULL
    assert lib.mot_selftest_wait_timeout(MIS, 64, None) == MOT_ERR_ALIGN
    assert lib.mot_selftest_wait_timeout(A, 8, None) == MOT_ERR_WORKSPACE


def test_interleave_and_status_reject(lib):
    assert lib.mot_swiglu_interleave(A, A, 100, 64, B, None) == MOT_ERR_GEOMETRY
    assert lib.mot_swiglu_interleave(None, A, 128, 64, B, None) == MOT_ERR_NULL
    flags = ctypes.c_uint32(0)
    assert lib.mot_device_status(None, ctypes.byref(flags), None) == MOT_ERR_NULL
    assert lib.mot_device_status(MIS, ctypes.byref(flags), None) == MOT_ERR_ALIGN


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_valid_arguments_without_gpu_fail_closed(lib):
    st = lib.mot_route_plan(A, 10, B, 1 << 20, None)
    assert st in (MOT_ERR_CUDA, MOT_ERR_DEVICE)


@pytest.mark.parametrize("D,P,theta", [(64, 64, 1e6), (128, 4096, 1e6), (128, 300, 1e4)])
def test_rope_table_matches_oracle(D, P, theta):
    t = mot.mot_rope_table_fill_host(theta, D, P)
    c, s = O.rope_cos_sin(theta, D, np.arange(P))
    got = t.float().numpy().astype(np.float64)
    np.testing.assert_array_equal(got[:, :, 0], c)
    np.testing.assert_array_equal(got[:, :, 1], s)


@pytest.mark.parametrize("D,P,theta", [(64, 64, 1e6), (128, 4096, 1e6), (128, 300, 1e4), (4, 8, 9.0)])
def test_rope_table_fp32_matches_oracle(D, P, theta):
    t = mot.mot_rope_table_fill_host_fp32(theta, D, P)
    c, s = O.rope_cos_sin_f32(theta, D, np.arange(P))
    got = t.numpy().astype(np.float64)
    np.testing.assert_array_equal(got[:, :, 0], c)
    np.testing.assert_array_equal(got[:, :, 1], s)
    # the bf16 table is this table rounded to bf16
    b = mot.mot_rope_table_fill_host(theta, D, P)
    assert torch.equal(b, t.to(torch.bfloat16))


def test_rope_table_rejects(lib):
    buf = (ctypes.c_uint16 * 16)()
    assert lib.mot_rope_table_fill_host(1e6, 3, 2, buf) == MOT_ERR_GEOMETRY
    assert lib.mot_rope_table_fill_host(0.5, 4, 2, buf) == MOT_ERR_ARG
    assert lib.mot_rope_table_fill_host(1e6, 4, 2, None) == MOT_ERR_NULL
    fbuf = (ctypes.c_float * 16)()
    assert lib.mot_rope_table_fill_host_fp32(1e6, 3, 2, fbuf) == MOT_ERR_GEOMETRY
    assert lib.mot_rope_table_fill_host_fp32(float("nan"), 4, 2, fbuf) == MOT_ERR_ARG
    assert lib.mot_rope_table_fill_host_fp32(1e6, 4, 2, None) == MOT_ERR_NULL


def test_flow_workspace_bytes(lib):
    f = lib.mot_flow_workspace_bytes
    assert f(0, 64) == 0 and f(1, 12) == 0 and f(1, 0) == 0 and f(65536, 64) == 0
    assert f(1, (1 << 24) + 8) == 0
    # header + 8 bytes per request and 8192-element segment, rounded to 16, + 4 bytes per
    # request and segment, rounded to 16
    assert f(1, 8) == 64 + 16 + 16
    assert f(3, 8192) == 64 + 32 + 16
    assert f(3, 8200) == 64 + 48 + 32
    assert f(16, 262144) == 64 + 16 * 32 * 8 + 16 * 32 * 4


def test_flow_schedule_matches_oracle():
    for n, shift in ((50, 1.0), (50, 3.0), (2, 0.5), (1000, 7.25)):
        got = mot.mot_flow_schedule_host(n, shift).numpy()
        np.testing.assert_array_equal(got, O.flow_schedule(n, shift))


def test_flow_schedule_rejects(lib):
    buf = (ctypes.c_float * 8)()
    assert lib.mot_flow_schedule_host(1, 3.0, buf) == MOT_ERR_GEOMETRY
    assert lib.mot_flow_schedule_host(4, 0.0, buf) == MOT_ERR_ARG
    assert lib.mot_flow_schedule_host(4, float("inf"), buf) == MOT_ERR_ARG
    assert lib.mot_flow_schedule_host(4, 3.0, None) == MOT_ERR_NULL


def test_cfg_combine_rejects(lib):
    f = lib.mot_cfg_combine_renorm
    assert f(None, A, A, 2, 64, A, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, None, A, 2, 64, A, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, A, A, 2, 64, None, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, A, A, 0, 64, A, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, 2, 60, A, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, 2, (1 << 24) + 8, A, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, MIS, 2, 64, A, B, 1 << 20, C, None) == MOT_ERR_ALIGN
    assert f(A, A, None, 2, 64, A, B, 64, C, None) == MOT_ERR_WORKSPACE


def test_flow_sde_step_rejects(lib):
    f = lib.mot_flow_sde_step
    assert f(None, A, A, C, 2, 64, A, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, A, A, None, 2, 64, A, B, 1 << 20, C, None) == MOT_ERR_NULL
    assert f(A, A, A, C, 2, 64, A, B, 1 << 20, None, None) == MOT_ERR_NULL
    assert f(A, A, A, C, 65536, 64, A, B, 1 << 30, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, A, C, 2, 4, A, B, 1 << 20, C, None) == MOT_ERR_GEOMETRY
    assert f(A, A, MIS, C, 2, 64, A, B, 1 << 20, C, None) == MOT_ERR_ALIGN
    assert f(A, A, None, C, 2, 64, A, B, 64, C, None) == MOT_ERR_WORKSPACE


def test_flow_cfg_sde_step_rejects(lib):
    f = lib.mot_flow_cfg_sde_step
    ok = (A, A, A, A, A, A, C, 2, 64, A, B, 1 << 20, C, C, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return f(*a)

    for i in (0, 1, 3, 4, 6, 9, 10, 13):       # v_c, v_tu, policy, x, x_next, times, ws, logp
        assert with_(i, None) == MOT_ERR_NULL, i
    assert with_(7, 0) == MOT_ERR_GEOMETRY
    assert with_(8, 60) == MOT_ERR_GEOMETRY
    assert with_(8, (1 << 24) + 8) == MOT_ERR_GEOMETRY
    assert with_(2, MIS) == MOT_ERR_ALIGN       # v_iu
    assert with_(5, MIS) == MOT_ERR_ALIGN       # z
    assert with_(12, MIS) == MOT_ERR_ALIGN      # v_out
    assert with_(11, 64) == MOT_ERR_WORKSPACE
    a = list(ok)
    a[2] = a[5] = a[12] = None                  # two branches, scoring, no v_out: still only a device error
    assert f(*a) not in (MOT_ERR_NULL, MOT_ERR_GEOMETRY, MOT_ERR_ALIGN, MOT_ERR_WORKSPACE, 0)


def test_flow_noise_rejects(lib):
    f = lib.mot_flow_noise
    assert f(None, 0, 2, 64, C, None) == MOT_ERR_NULL
    assert f(A, 0, 2, 64, None, None) == MOT_ERR_NULL
    assert f(A, 0, 0, 64, C, None) == MOT_ERR_GEOMETRY
    assert f(A, 0, 2, 12, C, None) == MOT_ERR_GEOMETRY
    assert f(A, 0, 2, (1 << 24) + 8, C, None) == MOT_ERR_GEOMETRY
    assert f(MIS, 0, 2, 64, C, None) == MOT_ERR_ALIGN

