"""Backward of the routed projection path on the GPU, through the C ABI, against the oracle.

add-RMSNorm backward ([RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap #435, §3 BAGEL
rules: the frozen und operators still need dX; [WS1][CUDA][Qwen3-Next] MoE route/combine
contract #503, gated-norm commit: a dx kernel and the weight gradient as an ascending-row fp32
left fold of per-row partials): dx, rstd and dw must equal the fp32 emulator E bit for bit,
and stay within the tolerance of the fp64 golden G.
"""

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W
from oracle import mot_oracle as O

from _util import assert_bitwise, assert_tolerance, f64, need_gpu, np_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _norm_bwd_inputs(T, H, seed, mod=None, with_dres=True):
    rng = W.rng_for(seed, 300)
    if mod is None:
        mod = W.modality_bernoulli(rng, T, 0.3)
    return {
        "dy": W.bf16_normal(W.rng_for(seed, 301), (T, H)),
        "s": W.bf16_normal(W.rng_for(seed, 302), (T, H)),
        "dro": W.bf16_normal(W.rng_for(seed, 303), (T, H)) if with_dres else None,
        "w": W.bf16_normal(W.rng_for(seed, 304), (2, H), mean=1.0, std=0.1),
        "mod": mod,
    }


def _run_norm_bwd(inp, eps=1e-6):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    T, H = d["dy"].shape
    ws = mot.mot_route_plan(d["mod"])
    part = torch.empty((H // 64, T, 64), dtype=torch.float32, device="cuda")
    dx, rstd = mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], eps, ws, d_res_out=d["dro"], dw_partials=part)
    dw = mot.mot_rmsnorm_dweight(part, ws)
    assert mot.mot_device_status(ws) == 0
    return dx, rstd, dw



@pytest.mark.parametrize("T,H,sets", [(333, 768, mot.SET_GEN), (333, 768, mot.SET_UND), (4096, 3584, mot.SET_GEN),
                                      (64, 256, mot.SET_GEN)])
def test_norm_backward_and_fold_of_one_weight_set(T, H, sets):
    # Phase A of the BAGEL training rules trains the gen set only: the partials of the other
    # set's rows and its row of dw stay as they were; dx, rstd, the selected partials and the
    # selected dw row equal the both-sets call bit for bit. (T = 64 at H = 256: Bernoulli rows
    # of both sets; T = 4096: the bench layer, 3072 und rows then 1024 gen rows.)
    mod = W.modality_blocks([(0, 3 * T // 4), (1, T - 3 * T // 4)]) if T == 4096 else None
    inp = _norm_bwd_inputs(T, H, 11, mod=mod)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ws = mot.mot_route_plan(d["mod"])
    part_all = torch.empty((H // 64, T, 64), dtype=torch.float32, device="cuda")
    dx_a, rstd_a = mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], 1e-6, ws, d_res_out=d["dro"],
                                                dw_partials=part_all)
    dw_all = mot.mot_rmsnorm_dweight(part_all, ws)
    part = torch.full((H // 64, T, 64), 7.0, dtype=torch.float32, device="cuda")
    dx, rstd = mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], 1e-6, ws, d_res_out=d["dro"], dw_partials=part,
                                            partial_sets=sets)
    dw = torch.full((2, H), 5.0, dtype=torch.float32, device="cuda")
    mot.mot_rmsnorm_dweight(part, ws, dw=dw, sets=sets)
    assert mot.mot_device_status(ws) == 0
    assert torch.equal(dx.view(torch.int16), dx_a.view(torch.int16)) and torch.equal(rstd, rstd_a)
    count0 = int((inp["mod"] == 0).sum())
    sel = slice(0, count0) if sets == mot.SET_UND else slice(count0, T)
    other = slice(count0, T) if sets == mot.SET_UND else slice(0, count0)
    assert torch.equal(part[:, sel].view(torch.int32), part_all[:, sel].view(torch.int32))
    assert bool((part[:, other] == 7.0).all())
    e = 0 if sets == mot.SET_UND else 1
    assert torch.equal(dw[e].view(torch.int32), dw_all[e].view(torch.int32))
    assert bool((dw[1 - e] == 5.0).all())



@pytest.mark.parametrize("row_set", [0, 1])
def test_one_set_masks_on_a_single_row(row_set):
    # one row: the set without rows folds to +0, and the mask leaves the other entries alone
    inp = _norm_bwd_inputs(1, 256, 12, mod=torch.tensor([row_set], dtype=torch.uint8))
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ws = mot.mot_route_plan(d["mod"])
    part = torch.full((4, 1, 64), 7.0, dtype=torch.float32, device="cuda")
    other = mot.SET_UND if row_set == 1 else mot.SET_GEN
    mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], 1e-6, ws, d_res_out=d["dro"], dw_partials=part,
                                 partial_sets=other)
    assert bool((part == 7.0).all())  # the row is not in the selected set
    dw = torch.full((2, 256), 5.0, dtype=torch.float32, device="cuda")
    mot.mot_rmsnorm_dweight(part, ws, dw=dw, sets=other)
    e_other = 0 if other == mot.SET_UND else 1
    assert torch.equal(dw[e_other].view(torch.int32), torch.zeros(256, dtype=torch.int32, device="cuda"))  # +0
    assert bool((dw[row_set] == 5.0).all())
    mine = mot.SET_GEN if row_set == 1 else mot.SET_UND
    mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], 1e-6, ws, d_res_out=d["dro"], dw_partials=part,
                                 partial_sets=mine)
    mot.mot_rmsnorm_dweight(part, ws, dw=dw, sets=mine)
    assert mot.mot_device_status(ws) == 0
    # a fold over one row is that row's partial
    assert torch.equal(dw[row_set].view(torch.int32), part[:, 0, :].reshape(256).view(torch.int32))


@pytest.mark.parametrize("T,H,seed,with_dres", [(64, 256, 1, True), (1, 256, 2, True), (333, 3584, 3, True),
                                                (1000, 768, 4, False), (300, 5120, 5, True),
                                                (4096, 3584, 6, True)])
def test_add_rmsnorm_backward_bitwise_vs_emulator(T, H, seed, with_dres):
    inp = _norm_bwd_inputs(T, H, seed, with_dres=with_dres)
    dx, rstd, dw = _run_norm_bwd(inp)
    dro = f64(inp["dro"]) if with_dres else None
    e = O.e_add_rmsnorm_backward(f64(inp["dy"]), f64(inp["s"]), f64(inp["w"]), inp["mod"].numpy(), 1e-6,
                                 d_res_out=dro)
    assert_bitwise(dx, np_bits(e["dx"]), "dx vs E")
    assert np.array_equal(rstd.cpu().numpy().view(np.uint32), e["rstd"].view(np.uint32)), "rstd vs E"
    assert np.array_equal(dw.cpu().numpy().view(np.uint32), e["dw"].view(np.uint32)), "dw vs E"
    g = O.g_add_rmsnorm_backward(f64(inp["dy"]), f64(inp["s"]), f64(inp["w"]), inp["mod"].numpy(), 1e-6,
                                 d_res_out=dro)
    assert_tolerance(f64(dx), g["dx_pre"], "dx vs G")
    # fp32 fold of T products against the exact sum: within T * 2^-23 of the sum of |partials|
    mod = inp["mod"].numpy()
    xh = f64(inp["s"]) * g["rstd"][:, None]
    for ex in (0, 1):
        r = mod == ex
        bound = (max(1, int(r.sum())) * 2.0 ** -23 + 1e-6) * np.sum(np.abs(f64(inp["dy"])[r] * xh[r]), axis=0)
        assert np.all(np.abs(dw.cpu().numpy()[ex].astype(np.float64) - g["dw"][ex]) <= bound + 1e-30)


def test_add_rmsnorm_backward_single_modality_and_empty_set():
    T, H = 200, 512
    inp = _norm_bwd_inputs(T, H, 7, mod=torch.zeros(T, dtype=torch.uint8))
    dx, rstd, dw = _run_norm_bwd(inp)
    e = O.e_add_rmsnorm_backward(f64(inp["dy"]), f64(inp["s"]), f64(inp["w"]), inp["mod"].numpy(), 1e-6,
                                 d_res_out=f64(inp["dro"]))
    assert_bitwise(dx, np_bits(e["dx"]), "dx vs E (all und)")
    dwn = dw.cpu().numpy()
    assert np.array_equal(dwn[0].view(np.uint32), e["dw"][0].view(np.uint32))
    assert np.all(dwn[1].view(np.uint32) == 0)      # +0.0 for the set without rows


def test_add_rmsnorm_backward_rows_are_batch_invariant():
    # a row's dx and rstd do not depend on the pack; dw of a sub-pack is the fold of its rows only
    T, H = 600, 1024
    inp = _norm_bwd_inputs(T, H, 8)
    dx, rstd, _ = _run_norm_bwd(inp)
    sel = np.sort(W.rng_for(8, 310).choice(T, 77, replace=False))
    sub = {k: (v[sel] if (v is not None and k != "w") else v) for k, v in inp.items()}
    dx2, rstd2, _ = _run_norm_bwd(sub)
    assert_bitwise(dx2, dx[torch.from_numpy(sel).cuda()], "dx of a sub-pack")
    assert torch.equal(rstd2, rstd[torch.from_numpy(sel).cuda()])


def test_add_rmsnorm_backward_flags_and_partials_layout():
    T, H = 64, 256
    inp = _norm_bwd_inputs(T, H, 9)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    # a plan for another T is refused on the device
    ws_other = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    mot.mot_route_plan(d["mod"][:50].contiguous(), ws=ws_other)
    mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], 1e-6, ws_other)
    assert mot.mot_device_status(ws_other) & mot.DEV_PLAN_MISMATCH
    part0 = torch.empty((H // 64, T, 64), dtype=torch.float32, device="cuda")
    ws_other2 = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    mot.mot_route_plan(d["mod"][:50].contiguous(), ws=ws_other2)
    mot.mot_rmsnorm_dweight(part0, ws_other2)
    assert mot.mot_device_status(ws_other2) & mot.DEV_PLAN_MISMATCH
    # the partials are p[r][j] = dy * (s * rstd) in blocks of 64 columns, rows in plan order
    ws = mot.mot_route_plan(d["mod"])
    part = torch.empty((H // 64, T, 64), dtype=torch.float32, device="cuda")
    _, rstd = mot.mot_add_rmsnorm_backward(d["dy"], d["s"], d["w"], 1e-6, ws, dw_partials=part)
    assert mot.mot_device_status(ws) == 0
    mod = inp["mod"].numpy()
    perm = np.concatenate([np.nonzero(mod == 0)[0], np.nonzero(mod == 1)[0]])
    dy32 = inp["dy"].float().numpy()
    xh = (inp["s"].float().numpy() * rstd.cpu().numpy()[:, None]).astype(np.float32)
    want = (dy32 * xh).astype(np.float32)[perm].reshape(T, H // 64, 64).transpose(1, 0, 2)
    assert np.array_equal(part.cpu().numpy().view(np.uint32), np.ascontiguousarray(want).view(np.uint32))


@pytest.mark.parametrize("T,H,case", [(4096, 3584, "bernoulli_0.25"), (4096, 3584, "contiguous_3_1"),
                                       (1, 256, "bernoulli_0.5"), (300, 8192, "bernoulli_0.3"),
                                       (5000, 256, "one_gen_row"), (5000, 768, "one_und_row"),
                                       (2500, 1024, "all_und"), (2500, 1024, "all_gen"),
                                       (20000, 512, "bernoulli_0.02")])
def test_rmsnorm_dweight_fold_bitwise_vs_emulator(T, H, case):
    # the fold alone, on random partials: the grid splits its CTAs between the sets by their row
    # counts, so one-row sets, empty sets and many units per CTA all take other assignments
    rng = W.rng_for(T * 7 + H, 320)
    if case.startswith("bernoulli"):
        mod = W.modality_bernoulli(rng, T, float(case.split("_")[1]))
    elif case == "contiguous_3_1":
        mod = torch.cat([torch.zeros(3 * T // 4, dtype=torch.uint8), torch.ones(T - 3 * T // 4, dtype=torch.uint8)])
    elif case in ("one_gen_row", "one_und_row"):
        mod = torch.full((T,), 0 if case == "one_gen_row" else 1, dtype=torch.uint8)
        mod[int(rng.integers(0, T))] = 1 if case == "one_gen_row" else 0
    else:
        mod = torch.full((T,), 0 if case == "all_und" else 1, dtype=torch.uint8)
    p = rng.standard_normal((T, H)).astype(np.float32) * np.float32(0.01)
    m = mod.numpy()
    perm = np.concatenate([np.nonzero(m == 0)[0], np.nonzero(m == 1)[0]])
    blocks = np.ascontiguousarray(p[perm].reshape(T, H // 64, 64).transpose(1, 0, 2))
    ws = mot.mot_route_plan(mod.cuda())
    dw = mot.mot_rmsnorm_dweight(torch.from_numpy(blocks).cuda(), ws)
    assert mot.mot_device_status(ws) == 0
    want = np.stack([O.e_left_fold_rows(p, m, 0), O.e_left_fold_rows(p, m, 1)]).astype(np.float32)
    assert np.array_equal(dw.cpu().numpy().view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------
# routed GEMM input gradient (both weight sets, MN-major weight operand)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,N,K,mode", [(300, 128, 256, "scatter"), (129, 512, 512, "gen"), (1, 64, 256, "scatter"),
                                        (640, 4608, 3584, "blocks")])
def test_routed_gemm_dx_integer_inputs_exact(T, N, K, mode):
    # small integers: every fp32 partial sum is exact, so the result is the exact gradient
    rng = W.rng_for(11, T + N)
    if mode == "scatter":
        mod = W.modality_bernoulli(rng, T, 0.4)
    elif mode == "gen":
        mod = torch.ones(T, dtype=torch.uint8)
    else:
        mod = W.modality_blocks([(0, T // 2), (1, T - T // 2)])
    dout = W.bf16_integers(W.rng_for(11, 1), (T, N), -2, 2)
    w = W.bf16_integers(W.rng_for(11, 2), (2, N, K), -2, 2)
    ws = mot.mot_route_plan(mod.cuda())
    dx = mot.mot_routed_gemm_dx(dout.cuda(), w.cuda(), ws)
    assert mot.mot_device_status(ws) == 0
    g = O.g_routed_gemm_dx(f64(dout), f64(w), mod.numpy())
    assert_bitwise(dx, np_bits(g["dx"]), "routed dX (integers)")


@pytest.mark.parametrize("T,N,K,p_gen,seed", [(777, 1024, 768, 0.3, 1), (4096, 4608, 3584, 0.25, 2),
                                              (500, 3584, 18944, 0.5, 3)])
def test_routed_gemm_dx_tolerance(T, N, K, p_gen, seed):
    mod = W.modality_bernoulli(W.rng_for(seed, 320), T, p_gen)
    dout = W.bf16_normal(W.rng_for(seed, 321), (T, N))
    w = W.bf16_normal(W.rng_for(seed, 322), (2, N, K), std=0.02)
    ws = mot.mot_route_plan(mod.cuda())
    dx = mot.mot_routed_gemm_dx(dout.cuda(), w.cuda(), ws)
    assert mot.mot_device_status(ws) == 0
    rows = np.arange(T) if T <= 1000 else np.unique(np.concatenate(
        [np.sort(W.rng_for(seed, 323).choice(T, 128, replace=False)), [0, T - 1]]))
    g = O.g_routed_gemm_dx(f64(dout)[rows], f64(w), mod.numpy()[rows])
    assert_tolerance(f64(dx)[rows], g["dx_pre"], "routed dX vs G")


def test_routed_gemm_dx_plan_order_flags_give_the_same_bits():
    T, N, K = 333, 512, 768
    mod = W.modality_bernoulli(W.rng_for(12, 330), T, 0.5)
    dout = W.bf16_normal(W.rng_for(12, 331), (T, N)).cuda()
    w = W.bf16_normal(W.rng_for(12, 332), (2, N, K), std=0.02).cuda()
    ws = mot.mot_route_plan(mod.cuda())
    ref = mot.mot_routed_gemm_dx(dout, w, ws)
    perm = torch.from_numpy(np.concatenate([np.nonzero(mod.numpy() == 0)[0], np.nonzero(mod.numpy() == 1)[0]])).cuda()
    dout_plan = mot.mot_gather_rows(dout, ws)
    a_plan = mot.mot_routed_gemm_dx(dout_plan, w, ws, flags=mot.A_PLAN_ORDER)
    both = mot.mot_routed_gemm_dx(dout_plan, w, ws, flags=mot.A_PLAN_ORDER | mot.OUT_PLAN_ORDER)
    out_plan = mot.mot_routed_gemm_dx(dout, w, ws, flags=mot.OUT_PLAN_ORDER)
    assert mot.mot_device_status(ws) == 0
    assert_bitwise(a_plan, ref, "dX, plan-order input")
    assert_bitwise(both, ref[perm], "dX, plan order in and out")
    assert_bitwise(out_plan, ref[perm], "dX, plan-order output")


# ---------------------------------------------------------------------------
# routed GEMM weight gradient (one weight set, rows ascending, fp32)
# ---------------------------------------------------------------------------

def _dw_run(dout, a, mod, expert):
    ws = mot.mot_route_plan(mod.cuda())
    dp = mot.mot_gather_rows(dout.cuda(), ws)
    ap = mot.mot_gather_rows(a.cuda(), ws)
    dw = mot.mot_routed_gemm_dw(dp, ap, ws, expert=expert, flags=mot.A_PLAN_ORDER)
    assert mot.mot_device_status(ws) == 0
    return dw


@pytest.mark.parametrize("T,N,K,mode,expert", [(300, 256, 512, "scatter", 1), (300, 256, 512, "scatter", 0),
                                               (129, 512, 256, "gen", 1), (250, 256, 256, "gen", 1),
                                               (64, 256, 256, "scatter", 0),
                                               (1000, 768, 1024, "blocks", 0), (300, 2560, 2816, "scatter", 1)])
def test_routed_gemm_dw_integer_inputs_exact(T, N, K, mode, expert):
    # small problems run every tile as two 128-column halves; 10 x 11 tiles on 76 clusters run
    # 76 whole tiles and the last 34 as halves; the sets' last 128-row blocks hold 1 (T = 129),
    # 122 (T = 250) and about 60 rows
    rng = W.rng_for(13, T + N + expert)
    if mode == "scatter":
        mod = W.modality_bernoulli(rng, T, 0.4)
    elif mode == "gen":
        mod = torch.ones(T, dtype=torch.uint8)
    else:
        mod = W.modality_blocks([(0, 700), (1, T - 700)])
    dout = W.bf16_integers(W.rng_for(13, 1), (T, N), -2, 2)
    a = W.bf16_integers(W.rng_for(13, 2), (T, K), -2, 2)
    dw = _dw_run(dout, a, mod, expert)
    g = O.g_routed_gemm_dw(f64(dout), f64(a), mod.numpy(), expert)
    np.testing.assert_array_equal(dw.cpu().numpy().astype(np.float64), g)


def test_routed_gemm_dw_set_without_rows_is_zero():
    T, N, K = 200, 256, 256
    mod = torch.zeros(T, dtype=torch.uint8)
    dw = _dw_run(W.bf16_normal(W.rng_for(14, 1), (T, N)), W.bf16_normal(W.rng_for(14, 2), (T, K)), mod, 1)
    assert torch.all(dw.view(torch.int32) == 0)


@pytest.mark.parametrize("T,N,K,p_gen,expert,seed", [(777, 1024, 768, 0.3, 1, 1), (777, 1024, 768, 0.3, 0, 1),
                                                     (4096, 4608, 3584, 0.25, 1, 2)])
def test_routed_gemm_dw_tolerance(T, N, K, p_gen, expert, seed):
    mod = W.modality_bernoulli(W.rng_for(seed, 340), T, p_gen)
    dout = W.bf16_normal(W.rng_for(seed, 341), (T, N))
    a = W.bf16_normal(W.rng_for(seed, 342), (T, K))
    dw = _dw_run(dout, a, mod, expert)
    rows = mod.numpy() == expert
    g = O.g_routed_gemm_dw(f64(dout), f64(a), mod.numpy(), expert)
    absum = np.abs(f64(dout)[rows]).T @ np.abs(f64(a)[rows])
    n = int(rows.sum())
    err = np.abs(dw.cpu().numpy().astype(np.float64) - g)
    # fp32 accumulation of n products (each exact in fp32) plus the final fp32 value
    assert np.all(err <= 2 * n * 2.0 ** -24 * absum + 2.0 ** -24 * np.abs(g)), float(np.max(err / (absum + 1e-30)))
    rel = float(np.linalg.norm(dw.cpu().numpy() - g) / np.linalg.norm(g))
    assert rel <= 1e-5, rel


def test_routed_gemm_dw_is_deterministic():
    T, N, K = 1500, 512, 512
    mod = W.modality_bernoulli(W.rng_for(15, 350), T, 0.6)
    dout = W.bf16_normal(W.rng_for(15, 351), (T, N))
    a = W.bf16_normal(W.rng_for(15, 352), (T, K))
    d1 = _dw_run(dout, a, mod, 1)
    d2 = _dw_run(dout, a, mod, 1)
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))


def test_routed_gemm_dw_into_16_byte_aligned_output_gives_the_same_bits():
    # the epilogue writes 32-byte sectors when dw is 32-byte aligned, 16-byte pieces otherwise
    T, N, K = 700, 512, 768
    mod = W.modality_bernoulli(W.rng_for(16, 360), T, 0.5)
    dout = W.bf16_normal(W.rng_for(16, 361), (T, N))
    a = W.bf16_normal(W.rng_for(16, 362), (T, K))
    ref = _dw_run(dout, a, mod, 1)
    ws = mot.mot_route_plan(mod.cuda())
    dp = mot.mot_gather_rows(dout.cuda(), ws)
    ap = mot.mot_gather_rows(a.cuda(), ws)
    buf = torch.empty(N * K + 4, dtype=torch.float32, device="cuda")
    out = buf[4:4 + N * K].view(N, K)
    assert out.data_ptr() % 32 == 16
    mot.mot_routed_gemm_dw(dp, ap, ws, expert=1, flags=mot.A_PLAN_ORDER, out=out)
    assert mot.mot_device_status(ws) == 0
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))


@pytest.mark.parametrize("T,N,K,layout,expert", [(300, 256, 512, "scatter", 1), (300, 256, 512, "scatter", 0),
                                                 (1000, 768, 1024, "blocks", 0), (1000, 768, 1024, "blocks", 1),
                                                 (4096, 4608, 3584, "bagel", 1), (777, 2560, 2816, "mixed", 1),
                                                 (129, 512, 256, "gen", 1), (64, 256, 256, "und", 1),
                                                 (36864, 256, 256, "cfg", 1), (36000, 256, 256, "cfg_ragged", 1),
                                                 (36000, 256, 256, "cfg_ragged", 0), (9000, 256, 512, "runs", 1)])
def test_routed_gemm_dw_token_order_gives_the_plan_order_bits(T, N, K, layout, expert):
    # token-order inputs: consecutive 128-row blocks by tiled loads, the others (and the ragged
    # last block) by four-row gathers through the plan; the same bytes as from gathered inputs.
    # cfg: 12 runs of 8 consecutive gen tiles at different offsets (96 tiles, three chunks of 32
    # tile records); cfg_ragged: runs of 1000 rows, so a gathered tile sits between runs; runs:
    # runs of 1500 gen rows, one crossing the 32-tile boundary of the records
    rng = W.rng_for(17, T + N)
    if layout == "cfg":
        mod = W.cfg_pack_layout(12, 2048, 1024)[0]
    elif layout == "cfg_ragged":
        mod = W.modality_blocks([b for _ in range(12) for b in ((0, 2000), (1, 1000))])
    elif layout == "runs":
        mod = W.modality_blocks([b for _ in range(4) for b in ((1, 1500), (0, 700))] + [(1, 200)])
    elif layout == "scatter":
        mod = W.modality_bernoulli(rng, T, 0.4)
    elif layout == "blocks":
        mod = W.modality_blocks([(0, 300), (1, 200), (0, 100), (1, T - 600)])
    elif layout == "bagel":
        mod = W.modality_blocks([(0, 3 * T // 4), (1, T - 3 * T // 4)])
    elif layout == "mixed":  # a long consecutive gen run, then scattered rows
        m = np.zeros(T, np.uint8)
        m[100:400] = 1
        m[400:] = (rng.random(T - 400) < 0.3).astype(np.uint8)
        mod = torch.from_numpy(m)
    else:
        mod = torch.full((T,), 1 if layout == "gen" else 0, dtype=torch.uint8)
    dout = W.bf16_normal(W.rng_for(17, 1), (T, N)).cuda()
    a = W.bf16_normal(W.rng_for(17, 2), (T, K)).cuda()
    ws = mot.mot_route_plan(mod.cuda())
    ref = mot.mot_routed_gemm_dw(mot.mot_gather_rows(dout, ws), mot.mot_gather_rows(a, ws), ws, expert=expert,
                                 flags=mot.A_PLAN_ORDER)
    got = mot.mot_routed_gemm_dw(dout, a, ws, expert=expert)
    assert mot.mot_device_status(ws) == 0
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
