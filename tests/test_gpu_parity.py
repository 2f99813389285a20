"""GPU parity: every entry point of libmot.so against the CPU oracle, through the C ABI.

  - integer and index work (the routing plan) is compared bit for bit with its definition;
  - the fused add-RMSNorm is compared bit for bit with the fp32 contract emulator E, and
    within the tolerance with the fp64 golden G;
  - the routed GEMMs are compared with G within the tolerance (bit for bit on integer-valued
    inputs, where every sum is exact), and their epilogues bit for bit with E fed the GPU's own
    bf16 GEMM output ("fused equals unfused").
Tolerance on bf16 outputs: max |diff| <= 2e-2 (or half a bf16 step where |value| >= 8, as no bf16
number lies closer) and relative L2 <= 4e-3 against G's value before its final cast. Sizes span several tiles and a ragged tail; the full-size cases check
sampled rows against G (rows are independent) and every row against E.
"""

import time

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W
from oracle import mot_oracle as O

from _util import (allowed_abs, assert_bitwise, assert_tolerance, bf16_step, check_end_to_end, decode_plan, f64,
                   need_gpu, np_bits)

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def cu(t):
    return t.cuda() if t is not None else None


# ---------------------------------------------------------------------------
# routing plan
# ---------------------------------------------------------------------------

def _mods():
    return {
        "bern1": W.modality_bernoulli(W.rng_for(1, 60), 1),
        "bern64": W.modality_bernoulli(W.rng_for(2, 60), 64),
        "bern1000": W.modality_bernoulli(W.rng_for(3, 60), 1000),
        "all_und300": torch.zeros(300, dtype=torch.uint8),
        "all_gen129": torch.ones(129, dtype=torch.uint8),
        "blocks4096": W.bagel_layer(1, T=4096)[1]["mod"],
        "scatter8192": W.modality_scattered(W.rng_for(4, 60), 8192, 2048),
        "cfg36864": W.cfg_pack_layout()[0],
        # above 65536 rows the plan is built by the many-CTA kernels (blocks of 8192 rows)
        "bern100003": W.modality_bernoulli(W.rng_for(5, 60), 100003),
        "scatter1M": W.modality_scattered(W.rng_for(6, 60), 1 << 20, 1 << 18),
        "blocks200k": W.modality_blocks([(0, 8191), (1, 3), (0, 70000), (1, 50000), (0, 1), (1, 71805)]),
        "all_gen65537": torch.ones(65537, dtype=torch.uint8),
    }


@pytest.mark.parametrize("name", list(_mods().keys()))
def test_route_plan_bitwise(name):
    mod = _mods()[name]
    T = mod.numel()
    ws = mot.mot_route_plan(mod.cuda())
    assert mot.mot_device_status(ws) == 0
    p = decode_plan(ws, T)
    m = mod.numpy()
    und, gen = np.nonzero(m == 0)[0], np.nonzero(m == 1)[0]
    assert p["T"] == T and p["count"] == (len(und), len(gen)) and p["error"] == 0
    np.testing.assert_array_equal(p["perm"], np.concatenate([und, gen]))
    want = []
    for e, rows, base in ((0, und, 0), (1, gen, len(und))):
        for i in range(0, len(rows), 128):
            chunk = rows[i:i + 128]
            row0 = int(chunk[0]) if chunk[-1] - chunk[0] == len(chunk) - 1 else -1
            want.append((base + i, len(chunk), e, row0))
    np.testing.assert_array_equal(p["tiles"], np.array(want, dtype=np.int32).reshape(-1, 4))


@pytest.mark.parametrize("name", ["bern1", "bern1000", "blocks4096", "scatter8192", "bern100003"])
def test_fused_norm_writes_the_same_plan(name):
    # the extra CTA of mot_fused_add_rmsnorm builds exactly the plan of mot_route_plan
    mod = _mods()[name].cuda()
    T = mod.numel()
    ref = mot.mot_route_plan(mod)
    x, res, w, _ = _norm_inputs(T, 256, 11)
    ws = torch.full_like(ref, 0xAB)
    mot.mot_fused_add_rmsnorm(x.cuda(), res.cuda(), w.cuda(), mod, EPS, ws=ws)
    assert mot.mot_device_status(ws) == 0
    a, b = decode_plan(ws, T), decode_plan(ref, T)
    assert (a["T"], a["count"], a["num_m_tiles"], a["magic"]) == (b["T"], b["count"], b["num_m_tiles"], b["magic"])
    np.testing.assert_array_equal(a["perm"], b["perm"])
    np.testing.assert_array_equal(a["tiles"], b["tiles"])


@pytest.mark.parametrize("T,bad_row", [(500, 321), (300000, 299999), (300000, 8192)])
def test_route_plan_rejects_bad_modality(T, bad_row):
    mod = torch.zeros(T, dtype=torch.uint8)
    mod[bad_row] = 2
    ws = mot.mot_route_plan(mod.cuda())
    assert mot.mot_device_status(ws) == mot.DEV_BAD_MODALITY
    assert decode_plan(ws, T)["num_m_tiles"] == 0


def test_fused_norm_with_a_many_cta_plan_flags_bad_modality():
    T = 70000
    x, res, w, mod = _norm_inputs(T, 256, 12)
    mod = mod.clone()
    mod[69999] = 3
    ws = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    mot.mot_fused_add_rmsnorm(x.cuda(), res.cuda(), w.cuda(), mod.cuda(), EPS, ws=ws)
    assert mot.mot_device_status(ws) & mot.DEV_BAD_MODALITY


# ---------------------------------------------------------------------------
# fused add-RMSNorm
# ---------------------------------------------------------------------------

def _norm_inputs(T, H, seed, mod=None):
    x = W.bf16_normal(W.rng_for(seed, 50), (T, H))
    res = W.bf16_normal(W.rng_for(seed, 51), (T, H))
    w = W.bf16_normal(W.rng_for(seed, 52), (2, H), mean=1.0, std=0.1)
    if mod is None:
        mod = W.modality_bernoulli(W.rng_for(seed, 53), T)
    return x, res, w, mod


@pytest.mark.parametrize("T,H,seed", [(64, 256, 1), (1, 256, 2), (333, 3584, 3), (1000, 768, 4), (4096, 3584, 5),
                                      (37, 8192, 6)])
def test_add_rmsnorm_bitwise_vs_emulator_and_tolerance_vs_golden(T, H, seed):
    x, res, w, mod = _norm_inputs(T, H, seed)
    y, ro = mot.mot_fused_add_rmsnorm(x.cuda(), res.cuda(), w.cuda(), mod.cuda(), EPS)
    e = O.e_fused_add_rmsnorm(f64(x), f64(res), f64(w), mod.numpy(), EPS)
    assert_bitwise(ro, np_bits(e["res_out"]), "res_out vs E")
    assert_bitwise(y, np_bits(e["y"]), "y vs E")
    g = O.g_fused_add_rmsnorm(f64(x), f64(res), f64(w), mod.numpy(), EPS)
    assert_tolerance(f64(y), g["y_pre"], "y vs G")


def test_add_rmsnorm_in_place_residual():
    x, res, w, mod = _norm_inputs(200, 512, 7)
    e = O.e_fused_add_rmsnorm(f64(x), f64(res), f64(w), mod.numpy(), EPS)
    r = res.cuda()
    y, ro = mot.mot_fused_add_rmsnorm(x.cuda(), r, w.cuda(), mod.cuda(), EPS, res_out=r)
    assert ro.data_ptr() == r.data_ptr()
    assert_bitwise(r, np_bits(e["res_out"]), "in-place res_out")
    assert_bitwise(y, np_bits(e["y"]), "y")


def test_add_rmsnorm_bad_modality_fails_closed():
    x, res, w, mod = _norm_inputs(64, 256, 8)
    mod[5] = 3
    ws = mot.mot_route_plan(torch.zeros(64, dtype=torch.uint8, device="cuda"))
    y = torch.full((64, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    mot.mot_fused_add_rmsnorm(x.cuda(), res.cuda(), w.cuda(), mod.cuda(), EPS, y=y, ws=ws)
    assert mot.mot_device_status(ws) & mot.DEV_BAD_MODALITY
    assert torch.all(y[5] == 7.0)                      # the bad row's y is not written


# ---------------------------------------------------------------------------
# routed GEMM (cast and SwiGLU epilogues)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,mode", [(300, "scatter"), (384, "blocks"), (1, "scatter"), (129, "gen")])
def test_routed_gemm_integer_inputs_exact(T, mode):
    # entries in {-1, 0, 1} and K = 128: every sum is an integer of magnitude <= 128, exact in
    # fp32 and bf16, so the GPU result is unique and must equal the oracle bit for bit
    K, N = 128, 512
    rng = W.rng_for(9, 61)
    a = W.bf16_integers(rng, (T, K), -1, 1)
    w = W.bf16_integers(W.rng_for(9, 62), (2, N, K), -1, 1)
    mod = {"scatter": W.modality_bernoulli(W.rng_for(9, 63), T),
           "blocks": W.modality_blocks([(0, T // 3), (1, T // 3), (0, T - 2 * (T // 3))]),
           "gen": torch.ones(T, dtype=torch.uint8)}[mode]
    ws = mot.mot_route_plan(mod.cuda())
    out = mot.mot_routed_gemm(a.cuda(), w.cuda(), ws, mot.EPI_CAST)
    assert mot.mot_device_status(ws) == 0
    g = O.g_routed_gemm_cast(f64(a), f64(w), mod.numpy())
    assert_bitwise(out, np_bits(g["out"]), "integer routed GEMM vs G")


@pytest.mark.parametrize("T,K,N,p_gen,seed", [(777, 1024, 768, 0.3, 1), (64, 256, 256, 0.5, 2), (1300, 512, 1024, 0.9, 3)])
def test_routed_gemm_cast_tolerance(T, K, N, p_gen, seed):
    a = W.bf16_normal(W.rng_for(seed, 64), (T, K))
    w = W.bf16_normal(W.rng_for(seed, 65), (2, N, K), std=0.02)
    mod = W.modality_bernoulli(W.rng_for(seed, 66), T, p_gen)
    ws = mot.mot_route_plan(mod.cuda())
    out = mot.mot_routed_gemm(a.cuda(), w.cuda(), ws, mot.EPI_CAST)
    assert mot.mot_device_status(ws) == 0
    g = O.g_routed_gemm_cast(f64(a), f64(w), mod.numpy())
    assert_tolerance(f64(out), g["out_pre"], "routed GEMM vs G")


def test_bounded_wait_times_out_and_context_stays_usable():
    # a wait that nothing satisfies gives up after about a second and reports a device error
    ws = torch.zeros(mot.mot_workspace_bytes(64), dtype=torch.uint8, device="cuda")
    t0 = time.time()
    mot.mot_selftest_wait_timeout(ws)
    flags = mot.mot_device_status(ws)
    dt = time.time() - t0
    assert flags & mot.DEV_TIMEOUT
    assert 0.5 < dt < 30.0
    # the context is still usable: a routed GEMM runs and is exact on integer inputs
    a = W.bf16_integers(W.rng_for(5, 90), (64, 128), -1, 1)
    w = W.bf16_integers(W.rng_for(5, 91), (2, 256, 128), -1, 1)
    mod = W.modality_bernoulli(W.rng_for(5, 92), 64)
    ws2 = mot.mot_route_plan(mod.cuda())
    out = mot.mot_routed_gemm(a.cuda(), w.cuda(), ws2, mot.EPI_CAST)
    assert mot.mot_device_status(ws2) == 0
    assert_bitwise(out, np_bits(O.g_routed_gemm_cast(f64(a), f64(w), mod.numpy())["out"]), "GEMM after a timeout")


def test_routed_gemm_plan_mismatch_fails_closed():
    a = W.bf16_normal(W.rng_for(1, 67), (100, 128)).cuda()
    w = W.bf16_normal(W.rng_for(1, 68), (2, 256, 128)).cuda()
    ws = mot.mot_route_plan(torch.zeros(90, dtype=torch.uint8, device="cuda"))   # plan of another T
    ws = torch.cat([ws, torch.zeros(4096, dtype=torch.uint8, device="cuda")])
    out = torch.full((100, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    mot.mot_routed_gemm(a, w, ws, mot.EPI_CAST, out=out)
    assert mot.mot_device_status(ws) & mot.DEV_PLAN_MISMATCH
    assert torch.all(out == 3.0)


def test_gather_rows_is_plan_order():
    T, K = 1000, 520
    src = W.bf16_normal(W.rng_for(3, 80), (T, K)).cuda()
    mod = W.modality_bernoulli(W.rng_for(3, 81), T, 0.3).cuda()
    ws = mot.mot_route_plan(mod)
    dst = mot.mot_gather_rows(src, ws)
    assert mot.mot_device_status(ws) == 0
    m = mod.cpu().numpy()
    perm = np.concatenate([np.nonzero(m == 0)[0], np.nonzero(m == 1)[0]])
    assert_bitwise(dst, src.cpu()[torch.from_numpy(perm)], "gathered rows")


@pytest.mark.parametrize("epi", ["cast", "swiglu"])
def test_plan_order_flags_give_the_same_bits(epi):
    # reading A in plan order and/or writing out in plan order moves rows, never changes them
    T, K = 777, 512
    a = W.bf16_normal(W.rng_for(4, 82), (T, K)).cuda()
    mod = W.modality_scattered(W.rng_for(4, 83), T, 200).cuda()
    ws = mot.mot_route_plan(mod)
    if epi == "cast":
        w = W.bf16_normal(W.rng_for(4, 84), (2, 512, K), std=0.02).cuda()
        e = mot.EPI_CAST
    else:
        w = mot.mot_swiglu_interleave(W.bf16_normal(W.rng_for(4, 85), (2, 256, K), std=0.02).cuda(),
                                      W.bf16_normal(W.rng_for(4, 86), (2, 256, K), std=0.02).cuda())
        e = mot.EPI_SWIGLU
    m = mod.cpu().numpy()
    perm = torch.from_numpy(np.concatenate([np.nonzero(m == 0)[0], np.nonzero(m == 1)[0]]))
    ref = mot.mot_routed_gemm(a, w, ws, e).cpu()                         # token order in and out
    a_plan = mot.mot_gather_rows(a, ws)
    in_plan = mot.mot_routed_gemm(a_plan, w, ws, e | mot.A_PLAN_ORDER).cpu()
    both = mot.mot_routed_gemm(a_plan, w, ws, e | mot.A_PLAN_ORDER | mot.OUT_PLAN_ORDER).cpu()
    out_plan = mot.mot_routed_gemm(a, w, ws, e | mot.OUT_PLAN_ORDER).cpu()
    assert mot.mot_device_status(ws) == 0
    assert_bitwise(in_plan, ref, "A in plan order")
    assert_bitwise(both, ref[perm], "A and out in plan order")
    assert_bitwise(out_plan, ref[perm], "out in plan order")


def test_swiglu_interleave_layout():
    I, K = 256, 64
    wg = W.bf16_normal(W.rng_for(2, 69), (2, I, K))
    wu = W.bf16_normal(W.rng_for(2, 70), (2, I, K))
    gu = mot.mot_swiglu_interleave(wg.cuda(), wu.cuda()).cpu()
    want = torch.cat([torch.cat([wg[:, b * 128:(b + 1) * 128], wu[:, b * 128:(b + 1) * 128]], dim=1)
                      for b in range(I // 128)], dim=1)
    assert_bitwise(gu, want, "interleaved gate/up layout")


@pytest.mark.parametrize("T,K,I,n_gen,seed", [(500, 512, 256, 125, 1), (1, 256, 256, 1, 2), (2048, 1024, 512, 512, 3)])
def test_routed_swiglu(T, K, I, n_gen, seed):
    a = W.bf16_normal(W.rng_for(seed, 71), (T, K))
    wg = W.bf16_normal(W.rng_for(seed, 72), (2, I, K), std=0.02)
    wu = W.bf16_normal(W.rng_for(seed, 73), (2, I, K), std=0.02)
    mod = W.modality_scattered(W.rng_for(seed, 74), T, n_gen)
    ws = mot.mot_route_plan(mod.cuda())
    gu = mot.mot_swiglu_interleave(wg.cuda(), wu.cuda())
    h = mot.mot_routed_gemm(a.cuda(), gu, ws, mot.EPI_SWIGLU)
    # teacher-forced epilogue check on the GPU's own bf16 gate/up outputs
    g = mot.mot_routed_gemm(a.cuda(), wg.cuda(), ws, mot.EPI_CAST)
    u = mot.mot_routed_gemm(a.cuda(), wu.cuda(), ws, mot.EPI_CAST)
    assert mot.mot_device_status(ws) == 0
    e = O.e_swiglu(f64(g), f64(u))
    hv = f64(h)
    _, ex = np.frexp(np.maximum(np.abs(e), 2.0 ** -120))
    # the only freedom is expf's last bit: within one bf16 step, and almost always equal
    assert np.all(np.abs(hv - e) <= np.ldexp(1.0, ex - 7))
    assert np.mean(hv == e) > 0.999
    ref = O.g_routed_swiglu(f64(a), f64(wg), f64(wu), mod.numpy())
    assert_tolerance(hv, ref["h_pre"], "SwiGLU vs G")


# ---------------------------------------------------------------------------
# routed QKV with QK RMSNorm and RoPE
# ---------------------------------------------------------------------------

PROFILES = ["bf16", "fp32"]


def _table(shape, P, profile):
    fill = mot.mot_rope_table_fill_host if profile == "bf16" else mot.mot_rope_table_fill_host_fp32
    return fill(shape.theta, shape.D, P).cuda()


def _qkv_run(shape, inp, with_bias=False, profile="bf16"):
    dev = {k: cu(v) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    P = int(inp["pos"].max()) + 1
    cs = _table(shape, P, profile)
    ws = mot.mot_route_plan(dev["mod"])
    out = mot.mot_routed_qkv_norm_rope(dev["x"], dev["w_qkv"], dev["q_norm"], dev["k_norm"], dev["pos"], cs, shape.Hq,
                                       shape.Hkv, shape.D, shape.eps, ws, b_qkv=dev.get("b_qkv") if with_bias else None)
    return out, ws, dev


def _check_qkv(shape, inp, out, ws, dev, rows=None, with_bias=False, profile="bf16"):
    assert mot.mot_device_status(ws) == 0
    mod = inp["mod"].numpy()
    pos = inp["pos"].numpy()
    r = np.arange(shape.T) if rows is None else rows
    g = O.g_qkv_norm_rope(f64(inp["x"])[r], f64(inp["w_qkv"]), f64(inp["b_qkv"]) if with_bias else None,
                          f64(inp["q_norm"]), f64(inp["k_norm"]), pos[r], mod[r], shape.Hq, shape.Hkv, shape.D,
                          shape.eps, shape.theta, rope_profile=profile)
    outv = f64(out)[r]
    if with_bias:
        # no unfused bias path to teacher-force from: bounded end-to-end check
        maxd = np.abs(outv - g["out_pre"])
        assert np.all(maxd <= 3 * bf16_step(np.maximum(np.abs(outv), np.abs(g["out_pre"]))))
        assert float(np.linalg.norm(outv - g["out_pre"]) / np.linalg.norm(g["out_pre"])) <= 4e-3
        return
    # stage 1: the routed GEMM's bf16 output against the exact accumulation
    q = mot.mot_routed_gemm(dev["x"], dev["w_qkv"], ws, mot.EPI_CAST)
    qv = f64(q)
    assert_tolerance(qv[r], g["acc"], "routed QKV GEMM (bf16 cast) vs G")
    # stage 2: the fused epilogue equals the fp32 contract emulator on the GPU's own q, bit for bit
    table = O.rope_cos_sin if profile == "bf16" else O.rope_cos_sin_f32
    c, s = table(shape.theta, shape.D, pos)
    e_out, _, u_e = O.e_qk_norm_rope(qv, f64(inp["q_norm"]), f64(inp["k_norm"]), c, s, mod, shape.Hq, shape.Hkv,
                                     shape.D, shape.eps, return_stats=True, rope_profile=profile)
    assert_bitwise(out, np_bits(e_out), f"fused QKV ({profile} RoPE) vs E on the cast GEMM output")
    # end to end against the golden chain
    acc_abs = O.g_routed_matmul(np.abs(f64(inp["x"])[r]), np.abs(f64(inp["w_qkv"])), mod[r])
    epi = {"q_norm": f64(inp["q_norm"]), "k_norm": f64(inp["k_norm"]), "pos": pos[r], "mod": mod[r]}
    check_end_to_end(outv, g, qv[r], u_e[r].astype(np.float64), acc_abs, shape, f"QKV ({profile} RoPE) vs G",
                     profile, epi)


@pytest.mark.parametrize("profile", PROFILES)
def test_qkv_tiny_layer(profile):
    shape, inp = W.tiny_layer(seed=1)
    out, ws, dev = _qkv_run(shape, inp, profile=profile)
    _check_qkv(shape, inp, out, ws, dev, profile=profile)


@pytest.mark.parametrize("profile", PROFILES)
@pytest.mark.parametrize("T,seed", [(640, 1), (161, 2)])
def test_qkv_bagel_shape_ragged(T, seed, profile):
    shape, inp = W.bagel_layer(seed=seed, T=T)
    out, ws, dev = _qkv_run(shape, inp, profile=profile)
    _check_qkv(shape, inp, out, ws, dev, profile=profile)


@pytest.mark.parametrize("profile", PROFILES)
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 4, 2), (64, 6, 1)])
def test_qkv_scattered_routing_and_positions(D, Hq, Hkv, profile):
    T, H = 300, 512
    shape = W.QKVShape(T=T, H=H, Hq=Hq, Hkv=Hkv, D=D)
    mod = W.modality_bernoulli(W.rng_for(3, 75), T, 0.4)
    pos = torch.from_numpy(W.rng_for(3, 76).integers(0, 50, T).astype(np.int32))   # repeated positions
    inp = W.qkv_layer_inputs(shape, mod, pos, seed=3)
    inp["x"] = W.bf16_normal(W.rng_for(3, 77), (T, H))
    out, ws, dev = _qkv_run(shape, inp, profile=profile)
    _check_qkv(shape, inp, out, ws, dev, profile=profile)


@pytest.mark.parametrize("profile", PROFILES)
def test_qkv_with_bias(profile):
    shape, inp = W.tiny_layer(seed=4)
    inp = W.qkv_layer_inputs(shape, inp["mod"], inp["pos"], seed=4, with_bias=True)
    out, ws, dev = _qkv_run(shape, inp, with_bias=True, profile=profile)
    _check_qkv(shape, inp, out, ws, dev, with_bias=True, profile=profile)


@pytest.mark.parametrize("profile", PROFILES)
@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 4, 2)])
def test_qkv_bias_epilogue_bitwise_on_integer_inputs(D, Hq, Hkv, profile):
    # Small-integer x and W make every partial sum of the routed GEMM an integer below 2^24, so
    # the tensor cores' fp32 accumulation is exact in any order and acc + b (b a bf16 number) is
    # exact too: q = bf16(acc + b) is known on the host. The fused epilogue must then equal the
    # fp32 emulator on that q bit for bit -- the stage check of the bias path.
    T, H = 200, 256
    shape = W.QKVShape(T=T, H=H, Hq=Hq, Hkv=Hkv, D=D)
    mod = W.modality_bernoulli(W.rng_for(8, 70), T, 0.5)
    pos = torch.from_numpy(W.rng_for(8, 71).integers(0, 64, T).astype(np.int32))
    inp = W.qkv_layer_inputs(shape, mod, pos, seed=8, with_bias=True)
    inp["x"] = W.bf16_integers(W.rng_for(8, 72), (T, H), -2, 2)
    inp["w_qkv"] = W.bf16_integers(W.rng_for(8, 73), (2, shape.n_qkv, H), -2, 2)
    out, ws, dev = _qkv_run(shape, inp, with_bias=True, profile=profile)
    assert mot.mot_device_status(ws) == 0
    m, p = mod.numpy(), pos.numpy()
    acc = O.g_routed_matmul(f64(inp["x"]), f64(inp["w_qkv"]), m) + f64(inp["b_qkv"])[m.astype(np.int64)]
    assert np.all(acc == acc.astype(np.float32)), "acc + b must be exact in fp32"
    q = O.bf16(acc)
    table = O.rope_cos_sin if profile == "bf16" else O.rope_cos_sin_f32
    c, s = table(shape.theta, D, p)
    e_out = O.e_qk_norm_rope(q, f64(inp["q_norm"]), f64(inp["k_norm"]), c, s, m, Hq, Hkv, D, shape.eps,
                             rope_profile=profile)
    assert_bitwise(out, np_bits(e_out), f"fused QKV with bias ({profile} RoPE) vs E on bf16(acc + b)")


@pytest.mark.parametrize("profile", PROFILES)
def test_qkv_single_row_and_single_modality(profile):
    for mod_val in (0, 1):
        shape = W.QKVShape(T=1, H=256, Hq=4, Hkv=2, D=64)
        inp = W.qkv_layer_inputs(shape, torch.full((1,), mod_val, dtype=torch.uint8),
                                 torch.tensor([17], dtype=torch.int32), seed=5)
        out, ws, dev = _qkv_run(shape, inp, profile=profile)
        _check_qkv(shape, inp, out, ws, dev, profile=profile)


@pytest.mark.parametrize("profile", PROFILES)
def test_qkv_position_out_of_table_flags(profile):
    shape, inp = W.tiny_layer(seed=6)
    dev = {k: cu(v) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    cs = _table(shape, 32, profile)    # positions 32..63 fall outside
    ws = mot.mot_route_plan(dev["mod"])
    mot.mot_routed_qkv_norm_rope(dev["x"], dev["w_qkv"], dev["q_norm"], dev["k_norm"], dev["pos"], cs, shape.Hq,
                                 shape.Hkv, shape.D, shape.eps, ws)
    assert mot.mot_device_status(ws) & mot.DEV_BAD_POSITION


@pytest.mark.parametrize("profile", PROFILES)
def test_qkv_bagel_layer_T4096_full_output(profile):
    # the timed layer (3072 und + 1024 gen rows, positions 0..4095), every element of the output
    shape, inp = W.bagel_layer(seed=1, T=4096)
    out, ws, dev = _qkv_run(shape, inp, profile=profile)
    _check_qkv(shape, inp, out, ws, dev, profile=profile)


def test_qkv_profiles_share_q_and_v():
    # the profiles differ only in the RoPE of Q/K heads: V columns are the same bits, and the
    # FP32 profile's entry point is selected by the table's dtype
    shape, inp = W.bagel_layer(seed=3, T=300)
    o16, ws, dev = _qkv_run(shape, inp, profile="bf16")
    o32 = mot.mot_routed_qkv_norm_rope_fp32(dev["x"], dev["w_qkv"], dev["q_norm"], dev["k_norm"], dev["pos"],
                                            _table(shape, shape.T, "fp32"), shape.Hq, shape.Hkv, shape.D,
                                            shape.eps, ws)
    assert mot.mot_device_status(ws) == 0
    v0 = (shape.Hq + shape.Hkv) * shape.D
    assert_bitwise(o16[:, v0:], o32[:, v0:], "V columns of the two profiles")
    a, b = f64(o16[:, :v0]), f64(o32[:, :v0])
    assert np.any(a != b)
    # both round the same rotation: they differ by a few bf16 steps of the rotated pair's
    # magnitude, which the rotation preserves (an element of a cancelling pair may be small)
    D = shape.D
    ah = a.reshape(shape.T, -1, D)
    pair = np.sqrt(ah ** 2 + np.roll(ah, D // 2, axis=2) ** 2).reshape(shape.T, -1)
    assert np.all(np.abs(a - b) <= 3 * bf16_step(pair) + bf16_step(np.maximum(np.abs(a), np.abs(b))))


@pytest.mark.parametrize("profile", PROFILES)
def test_layer_tiny_end_to_end(profile):
    # norm -> QKV through the library vs the golden layer
    shape, inp = W.tiny_layer(seed=7)
    dev = {k: cu(v) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    ws = mot.mot_route_plan(dev["mod"])
    y, ro = mot.mot_fused_add_rmsnorm(dev["x"], dev["res"], dev["w_norm"], dev["mod"], shape.eps, ws=ws)
    cs = _table(shape, shape.T, profile)
    out = mot.mot_routed_qkv_norm_rope(y, dev["w_qkv"], dev["q_norm"], dev["k_norm"], dev["pos"], cs, shape.Hq,
                                       shape.Hkv, shape.D, shape.eps, ws)
    assert mot.mot_device_status(ws) == 0
    g = O.g_layer(f64(inp["x"]), f64(inp["res"]), f64(inp["w_norm"]), f64(inp["w_qkv"]), None, f64(inp["q_norm"]),
                  f64(inp["k_norm"]), inp["pos"].numpy(), inp["mod"].numpy(), shape.Hq, shape.Hkv, shape.D,
                  shape.eps, shape.theta, rope_profile=profile)
    assert_tolerance(f64(y), g["y_pre"], "layer y vs G")
    assert_tolerance(f64(out), g["out_pre"], f"layer QKV ({profile} RoPE) vs G")
