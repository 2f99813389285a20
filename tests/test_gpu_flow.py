"""Flow sampler pieces on the GPU, through the C ABI, against the oracle.

[RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap #435: §1 Motivation items 2 and 3 (the
policy log-probability is the ODE-to-SDE transition density; three-branch renormalised CFG);
§2 (training and rollout produce exactly equal logp); §3 BAGEL-specific rules (FP32 SDE step
with sigma = t and dt > 0; the t = 1 first step and the t -> 0 last step as separate cases; the
CFG window on FP32 t; renorm per request, never coupled across the batch; cfg_text_scale <= 1
as its own case). The kernels follow the oracle's fp32 restatement bit for bit, except logp,
whose log of the step's std is the GPU's logf (at most an ulp or two from the host's log).
"""

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W
from oracle import mot_oracle as O

from _util import need_gpu

pytestmark = pytest.mark.gpu

F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bits(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=F32).view(np.uint32)


def assert_f32_bitwise(gpu, ref, what):
    g, r = _bits(gpu), _bits(ref)
    if not np.array_equal(g, r):
        bad = np.argwhere(g != r)
        raise AssertionError(f"{what}: {len(bad)} of {g.size} values differ, first {bad[:5].tolist()}")


def assert_close_f32(gpu, ref, what, rtol=2e-5):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    d = np.abs(gpu - ref)
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    assert d.max() <= rtol * scale and rel <= rtol, f"{what}: max|diff| {d.max():.3e} rel-L2 {rel:.3e}"


def logp_bound(N, std, lw, logp):
    """How far logp may move when the log of std is the GPU's logf instead of the host's: the
    log term N (log std + log sqrt(2 pi)) shifts by N times about two ulps of the bracket, then
    the product and the final difference round once more each."""
    br = abs(float(np.log(F32(std))) + float(F32(O.LOG_SQRT_2PI)))
    return (N * 2 * float(np.spacing(F32(br))) + 2 * float(np.spacing(F32(abs(lw))))
            + 2 * float(np.spacing(F32(abs(logp)))))


# ---------------------------------------------------------------------------
# CFG combine + renorm
# ---------------------------------------------------------------------------

# (t, s_text, s_img, t_lo, t_hi, renorm_min) per request
POLICIES = [
    (0.5, 4.0, 2.0, 0.4, 1.0, 0.0),      # guided, guided norm above ||c||: r < 1
    (0.3, 4.0, 2.0, 0.4, 1.0, 0.0),      # outside the window: out = c
    (0.4, 4.0, 2.0, 0.4, 1.0, 0.0),      # on the window's lower edge (fp32 0.4): guided
    (0.9, 4.0, 2.0, 0.4, 1.0, 0.9),      # the clamp from below: r = 0.9
    (0.7, 0.5, 1.0, 0.4, 1.0, 0.0),      # cfg_text_scale <= 1, zero unconditioned branches: r = 1
    (1.0, 4.0, 2.0, 0.4, 1.0, 0.0),      # t = 1 (the first step), all branches zero: r = 1, out = 0
]


def _cfg_case(n_req, N, seed):
    b = W.flow_branches(W.rng_for(seed, 700), n_req, N)
    if n_req == len(POLICIES):
        for k in ("c", "tu", "iu"):
            b[k][5].zero_()
        b["tu"][4].zero_()   # v2 = c / 2: the ratio 2 is clamped to 1
        b["iu"][4].zero_()
    pol = np.array([POLICIES[i % len(POLICIES)] for i in range(n_req)], dtype=F32)
    return b, pol


def _cfg_gpu(b, pol, three=True):
    d = {k: v.cuda() for k, v in b.items()}
    n_req, N = d["c"].shape
    ws = torch.zeros(mot.mot_flow_workspace_bytes(n_req, N), dtype=torch.uint8, device="cuda")
    out = mot.mot_cfg_combine_renorm(d["c"], d["tu"], d["iu"] if three else None, torch.from_numpy(pol).cuda(), ws=ws)
    assert mot.mot_device_status(ws) == 0
    return out.cpu().numpy()


def _cfg_oracle(b, pol, i, three=True, level="e"):
    f = O.e_cfg_combine_renorm if level == "e" else O.g_cfg_combine_renorm
    c, tu, iu = (b[k][i].float().numpy().astype(np.float64) for k in ("c", "tu", "iu"))
    t, s_text, s_img, t_lo, t_hi, rmin = (float(v) for v in pol[i])
    return f(c, tu, iu if three else None, t, s_text, s_img, t_lo, t_hi, rmin)


# 32 and 33 segments: the request's fold fetches its segment sums 32 at a time
@pytest.mark.parametrize("N", [8, 2056, 8192, 3 * 8192 + 40, 32 * 8192, 32 * 8192 + 8])
@pytest.mark.parametrize("three", [True, False])
def test_cfg_combine_bitwise_vs_oracle(N, three):
    b, pol = _cfg_case(len(POLICIES), N, seed=N + three)
    out = _cfg_gpu(b, pol, three)
    for i in range(len(POLICIES)):
        e = _cfg_oracle(b, pol, i, three)
        assert_f32_bitwise(out[i], e, f"cfg request {i} N={N} three={three}")
        g = _cfg_oracle(b, pol, i, three, level="g")
        if np.any(g):
            assert_close_f32(out[i], g, f"cfg request {i} vs fp64")
        else:
            assert not np.any(out[i])
    # the cases behave as labelled
    c0 = b["c"].float().numpy()
    np.testing.assert_array_equal(out[1], c0[1])                             # outside the window
    np.testing.assert_array_equal(out[4], c0[4] * F32(0.5))                 # r clamped to 1
    if three:
        n = np.linalg.norm
        assert abs(n(out[0]) - n(c0[0])) <= 1e-5 * n(c0[0])                  # rescaled to ||c||


def test_cfg_renorm_is_per_request():
    # A request's output does not depend on the other requests of the batch: alone, in a batch,
    # and in a batch whose other requests change, it is bit for bit the same.
    N = 8192 + 800
    b, pol = _cfg_case(6, N, seed=71)
    full = _cfg_gpu(b, pol)
    for i in (0, 3):
        alone = _cfg_gpu({k: v[i:i + 1].clone() for k, v in b.items()}, pol[i:i + 1].copy())
        assert_f32_bitwise(alone[0], full[i], f"request {i} alone vs in the batch")
    b2 = {k: v.clone() for k, v in b.items()}
    for k in b2:
        b2[k][1:3] *= 7
    changed = _cfg_gpu(b2, pol)
    assert_f32_bitwise(changed[0], full[0], "request 0 with its neighbours changed")


def test_cfg_window_edges_on_fp32_t():
    # t just below the window's lower edge is unguided, t on the upper edge guided
    N = 64
    b = W.flow_branches(W.rng_for(5, 701), 2, N)
    lo = F32(0.4)
    pol = np.array([(np.nextafter(lo, F32(0)), 4, 2, lo, 1, 0), (1.0, 4, 2, lo, 1, 0)], dtype=F32)
    out = _cfg_gpu(b, pol)
    np.testing.assert_array_equal(out[0], b["c"][0].float().numpy())
    assert_f32_bitwise(out[1], _cfg_oracle(b, pol, 1), "upper edge")
    assert not np.array_equal(out[1], b["c"][1].float().numpy())


def test_cfg_full_size_sampled():
    # 16 requests of a 1024 x 1024 latent (N = 262144), as timed; two requests checked in full
    n_req, N = W.FLOW_REQUESTS, W.FLOW_N_1024
    b = W.flow_branches(W.rng_for(6, 702), n_req, N)
    pol = np.array([(float(F32(0.4 + 0.6 * i / n_req)), 4.0, 2.0, 0.4, 1.0, 0.0) for i in range(n_req)], dtype=F32)
    out = _cfg_gpu(b, pol)
    for i in (0, n_req - 1):
        assert_f32_bitwise(out[i], _cfg_oracle(b, pol, i), f"full-size request {i}")


# ---------------------------------------------------------------------------
# SDE step + logp
# ---------------------------------------------------------------------------

SCHED = O.flow_schedule(W.FLOW_STEPS, W.FLOW_SHIFT)
# (t_i, t_next): the t = 1 first step, a middle step, the last step to t = 0, a tiny-t last step
STEPS = [(SCHED[0], SCHED[1]), (SCHED[25], SCHED[26]), (SCHED[-2], SCHED[-1]), (F32(1e-3), F32(0.0))]


def _sde_gpu(st, times, score_x_next=None):
    d = {k: v.cuda() for k, v in st.items()}
    n_req, N = d["x"].shape
    ws = torch.zeros(mot.mot_flow_workspace_bytes(n_req, N), dtype=torch.uint8, device="cuda")
    tt = torch.from_numpy(np.asarray(times, dtype=F32)).cuda()
    if score_x_next is None:
        xn, lp = mot.mot_flow_sde_step(d["x"], d["v"], d["z"], tt, ws=ws)
    else:
        xn, lp = mot.mot_flow_sde_step(d["x"], d["v"], None, tt, ws=ws, x_next=score_x_next.cuda().clone())
    return xn.cpu().numpy(), lp.cpu().numpy(), mot.mot_device_status(ws)


def _sde_check(st, times, xn, lp, i, what):
    x, v, z = (st[k][i].numpy().astype(np.float64) for k in ("x", "v", "z"))
    t, tn = (float(u) for u in times[i])
    e = O.e_flow_sde_step(x, v, z, t, tn)
    assert_f32_bitwise(xn[i], e["x_next"], f"{what}: x_next")
    N = x.size
    lw = float(F32(N) * (np.log(F32(e["std"])) + F32(O.LOG_SQRT_2PI)))
    assert abs(float(lp[i]) - float(e["logp"])) <= logp_bound(N, e["std"], lw, e["logp"]), \
        f"{what}: logp {lp[i]!r} vs {e['logp']!r}"
    g = O.g_flow_sde_step(x, v, z, t, tn)
    assert_close_f32(xn[i], g["x_next"], f"{what}: x_next vs fp64", rtol=1e-5)
    a_g = np.sum((g["x_next"] - g["mu"]) ** 2) / (2 * g["std"] ** 2)
    assert abs(float(lp[i]) - g["logp"]) <= 1e-4 * (a_g + abs(g["logp"] + a_g)), f"{what}: logp vs fp64"


@pytest.mark.parametrize("N", [8, 2056, 8192, 3 * 8192 + 40, 32 * 8192 + 8])
def test_sde_step_first_middle_last_steps(N):
    st = W.flow_state(W.rng_for(N, 710), len(STEPS), N)
    xn, lp, flags = _sde_gpu(st, STEPS)
    assert flags == 0
    for i, (t, tn) in enumerate(STEPS):
        _sde_check(st, STEPS, xn, lp, i, f"N={N} step {t}->{tn}")
    # the first step starts at t = 1 exactly and the last ends at 0 (the schedule's ends)
    assert STEPS[0][0] == F32(1.0) and STEPS[2][1] == F32(0.0)


def test_sde_scoring_reproduces_the_rollout_logp():
    # training evaluates the stored latent with the same x, v and times: logp bit for bit
    N = 2 * 8192 + 16
    st = W.flow_state(W.rng_for(3, 711), len(STEPS), N)
    xn, lp, _ = _sde_gpu(st, STEPS)
    xn2, lp2, flags = _sde_gpu(st, STEPS, score_x_next=torch.from_numpy(xn))
    assert flags == 0
    assert_f32_bitwise(lp2, lp, "scored logp vs rollout logp")
    assert_f32_bitwise(xn2, xn, "x_next untouched when scored")
    # a different latent is scored as a Gaussian around the same mean
    y = torch.from_numpy(W.flow_state(W.rng_for(4, 712), len(STEPS), N)["z"].numpy())
    _, lp3, _ = _sde_gpu(st, STEPS, score_x_next=y)
    for i, (t, tn) in enumerate(STEPS):
        x, v = (st[k][i].numpy().astype(np.float64) for k in ("x", "v"))
        e = O.e_flow_sde_step(x, v, None, float(t), float(tn), x_next=y[i].numpy())
        lw = float(F32(N) * (np.log(F32(e["std"])) + F32(O.LOG_SQRT_2PI)))
        assert abs(float(lp3[i]) - float(e["logp"])) <= logp_bound(N, e["std"], lw, e["logp"])


def test_sde_bad_times_fail_closed():
    # dt <= 0 (the sign), t_next < 0 and t_i > 1 set DEV_BAD_TIME; those requests' outputs are
    # left as they were, the valid request in the same call is computed
    N = 64
    times = [(0.5, 0.6), (0.5, 0.5), (0.2, -0.1), (1.5, 0.9), (0.6, 0.5)]
    st = W.flow_state(W.rng_for(8, 713), len(times), N)
    d = {k: v.cuda() for k, v in st.items()}
    ws = torch.zeros(mot.mot_flow_workspace_bytes(len(times), N), dtype=torch.uint8, device="cuda")
    xn = torch.full((len(times), N), 7.0, device="cuda")
    lp = torch.full((len(times),), 7.0, device="cuda")
    mot.mot_flow_sde_step(d["x"], d["v"], d["z"], torch.tensor(times, dtype=torch.float32, device="cuda"), ws=ws,
                          x_next=xn, logp=lp)
    assert mot.mot_device_status(ws) == mot.DEV_BAD_TIME
    xn, lp = xn.cpu().numpy(), lp.cpu().numpy()
    assert np.all(xn[:4] == 7.0) and np.all(lp[:4] == 7.0)
    _sde_check(st, np.array(times, dtype=F32), xn, lp, 4, "valid request beside bad ones")


def test_sde_batch_invariance_and_full_size_sampled():
    # 16 requests of a 1024 x 1024 latent at 16 different steps; two checked in full, one
    # recomputed alone bit for bit
    n_req, N = W.FLOW_REQUESTS, W.FLOW_N_1024
    st = W.flow_state(W.rng_for(9, 714), n_req, N)
    times = np.array([(SCHED[3 * i], SCHED[3 * i + 1]) for i in range(n_req)], dtype=F32)
    xn, lp, flags = _sde_gpu(st, times)
    assert flags == 0
    for i in (0, n_req - 1):
        _sde_check(st, times, xn, lp, i, f"full-size request {i}")
    xa, la, _ = _sde_gpu({k: v[5:6].clone() for k, v in st.items()}, times[5:6])
    assert_f32_bitwise(xa[0], xn[5], "x_next alone vs in the batch")
    assert_f32_bitwise(la, lp[5:6], "logp alone vs in the batch")


# ---------------------------------------------------------------------------
# Per-sample transition noise
# ---------------------------------------------------------------------------

SEEDS = [0, 1, 2 ** 63 + 5, 2 ** 64 - 1, 123456789]


def _seeds_dev(seeds):
    return torch.tensor(np.array(seeds, dtype=np.uint64).view(np.int64), device="cuda")


@pytest.mark.parametrize("N,step", [(8, 0), (2056, 3), (8192 + 40, 2 ** 40 + 7)])
def test_flow_noise_vs_oracle(N, step):
    # Philox4x64-10 counters and keys must match exactly (a slip gives unrelated deviates); the
    # fp32 Box-Muller (logf, sqrt, sincospif) is within a few ulps of the fp64 transform of the
    # same uniforms
    z = mot.mot_flow_noise(_seeds_dev(SEEDS), step, N).cpu().numpy().astype(np.float64)
    g = O.g_flow_noise(SEEDS, step, N)
    d = np.abs(z - g)
    assert np.all(d <= 1e-6 + 4e-6 * np.abs(g)), f"max |diff| {d.max():.3e}"


def test_flow_noise_per_sample_and_per_step():
    N = 4096
    full = mot.mot_flow_noise(_seeds_dev(SEEDS), 9, N)
    alone = mot.mot_flow_noise(_seeds_dev(SEEDS[2:3]), 9, N)
    assert torch.equal(alone[0], full[2])                        # independent of the batch
    other = mot.mot_flow_noise(_seeds_dev(SEEDS), 10, N)
    assert not torch.equal(other, full)                          # each step has its own stream
    again = mot.mot_flow_noise(_seeds_dev(SEEDS), 9, N)
    assert torch.equal(again, full)                              # deterministic
    zz = full.double()
    assert abs(float(zz.mean())) < 0.05 and abs(float(zz.var()) - 1.0) < 0.05


def _at_16_bytes(t):
    """A copy of the fp32 tensor t on the GPU whose data starts 16 bytes past a 32-byte boundary."""
    buf = torch.empty(t.numel() + 4, dtype=torch.float32, device="cuda")
    v = buf[4:4 + t.numel()].view(t.shape)
    assert v.data_ptr() % 32 == 16
    v.copy_(t.cuda())
    return v


def test_cfg_and_sde_with_16_byte_aligned_tensors_give_the_same_bits():
    # 32-byte loads and stores are used when every tensor allows them, 16-byte ones otherwise
    N = 3 * 8192 + 40
    b, pol = _cfg_case(len(POLICIES), N, seed=77)
    aligned = _cfg_gpu(b, pol)
    d = {k: v.cuda() for k, v in b.items()}
    ws = torch.zeros(mot.mot_flow_workspace_bytes(len(POLICIES), N), dtype=torch.uint8, device="cuda")
    out16 = _at_16_bytes(torch.zeros((len(POLICIES), N)))
    mot.mot_cfg_combine_renorm(d["c"], d["tu"], d["iu"], torch.from_numpy(pol).cuda(), ws=ws, out=out16)
    assert mot.mot_device_status(ws) == 0
    np.testing.assert_array_equal(out16.cpu().numpy().view(np.uint32), aligned.view(np.uint32))
    st = W.flow_state(W.rng_for(N, 711), len(STEPS), N)
    xn, lp, flags = _sde_gpu(st, STEPS)
    assert flags == 0
    ws2 = torch.zeros(mot.mot_flow_workspace_bytes(len(STEPS), N), dtype=torch.uint8, device="cuda")
    tt = torch.from_numpy(np.asarray(STEPS, dtype=F32)).cuda()
    xn16 = _at_16_bytes(torch.zeros((len(STEPS), N)))
    _, lp16 = mot.mot_flow_sde_step(_at_16_bytes(st["x"]), _at_16_bytes(st["v"]), _at_16_bytes(st["z"]), tt, ws=ws2,
                                    x_next=xn16)
    assert mot.mot_device_status(ws2) == 0
    np.testing.assert_array_equal(xn16.cpu().numpy().view(np.uint32), xn.view(np.uint32))
    np.testing.assert_array_equal(lp16.cpu().numpy().view(np.uint32), lp.view(np.uint32))


# ---------------------------------------------------------------------------
# CFG combine + renorm and the SDE step in one call
# ---------------------------------------------------------------------------

def _fused_inputs(N, seed, three=True):
    b, pol = _cfg_case(len(POLICIES), N, seed=seed)
    st = W.flow_state(W.rng_for(seed, 720), len(POLICIES), N)
    times = np.array([(p[0], p[0] - F32(0.05)) for p in pol], dtype=F32)   # t_i is the policy's t
    d = {k: v.cuda() for k, v in b.items()}
    d.update({k: v.cuda() for k, v in st.items() if k != "v"})
    return d, torch.from_numpy(pol).cuda(), torch.from_numpy(times).cuda()


def _chain(d, pol, times, three=True):
    n_req, N = d["c"].shape
    ws = torch.zeros(mot.mot_flow_workspace_bytes(n_req, N), dtype=torch.uint8, device="cuda")
    v = mot.mot_cfg_combine_renorm(d["c"], d["tu"], d["iu"] if three else None, pol, ws=ws)
    xn, lp = mot.mot_flow_sde_step(d["x"], v, d["z"], times, ws=ws)
    assert mot.mot_device_status(ws) == 0
    return v, xn, lp


@pytest.mark.parametrize("N", [8, 2056, 3 * 8192 + 40, 32 * 8192 + 8])
@pytest.mark.parametrize("three", [True, False])
def test_fused_cfg_sde_equals_the_two_calls(N, three):
    # the guided velocity, x_next and logp bit for bit those of mot_cfg_combine_renorm followed by
    # mot_flow_sde_step: guided and unguided requests, the window edge, the clamp, zero branches
    d, pol, times = _fused_inputs(N, N + 3 * three, three)
    v, xn, lp = _chain(d, pol, times, three)
    n_req = d["c"].shape[0]
    ws = torch.zeros(mot.mot_flow_workspace_bytes(n_req, N), dtype=torch.uint8, device="cuda")
    v2 = torch.empty_like(v)
    xn2, lp2 = mot.mot_flow_cfg_sde_step(d["c"], d["tu"], d["iu"] if three else None, pol, d["x"], d["z"], times,
                                         ws=ws, v_out=v2)
    assert mot.mot_device_status(ws) == 0
    assert_f32_bitwise(v2, v, "fused guided velocity vs the CFG call")
    assert_f32_bitwise(xn2, xn, "fused x_next vs the two calls")
    assert_f32_bitwise(lp2, lp, "fused logp vs the two calls")
    # without v_out, and scoring the sampled latent: the same logp
    xn3, lp3 = mot.mot_flow_cfg_sde_step(d["c"], d["tu"], d["iu"] if three else None, pol, d["x"], None, times,
                                         ws=ws, x_next=xn2.clone())
    assert mot.mot_device_status(ws) == 0
    assert_f32_bitwise(lp3, lp, "fused scoring of the sampled latent")
    # and against the oracle's fp32 restatement for one guided request
    e_v = _cfg_oracle({k: t.cpu() for k, t in d.items() if k in ("c", "tu", "iu")}, pol.cpu().numpy(), 0, three)
    assert_f32_bitwise(v2[0].cpu().numpy(), e_v, "fused guided velocity vs E")


def test_fused_cfg_sde_bad_times_fail_closed():
    N = 64
    d, pol, _ = _fused_inputs(N, 5)
    times = torch.tensor([(0.5, 0.6), (0.3, 0.3), (0.4, -0.1), (1.5, 0.9), (0.7, 0.6), (1.0, 0.95)],
                         dtype=torch.float32, device="cuda")
    ws = torch.zeros(mot.mot_flow_workspace_bytes(6, N), dtype=torch.uint8, device="cuda")
    xn = torch.full((6, N), 7.0, device="cuda")
    lp = torch.full((6,), 7.0, device="cuda")
    vo = torch.full((6, N), 7.0, device="cuda")
    mot.mot_flow_cfg_sde_step(d["c"], d["tu"], d["iu"], pol, d["x"], d["z"], times, ws=ws, x_next=xn, v_out=vo,
                              logp=lp)
    assert mot.mot_device_status(ws) == mot.DEV_BAD_TIME
    assert torch.all(xn[:4] == 7.0) and torch.all(lp[:4] == 7.0) and torch.all(vo[:4] == 7.0)
    v, xc, lc = _chain({k: t[4:] for k, t in d.items()}, pol[4:], times[4:])
    assert_f32_bitwise(xn[4:], xc, "valid requests beside bad ones: x_next")
    assert_f32_bitwise(lp[4:], lc, "valid requests beside bad ones: logp")
    assert_f32_bitwise(vo[4:], v, "valid requests beside bad ones: v")


def test_fused_cfg_sde_full_size_and_16_byte_alignment():
    # the bench leg: 16 requests of a 1024 x 1024 latent, each at its own step of the 50-step,
    # shift-3 schedule; the same bits as the two calls, and with 16-byte-aligned fp32 tensors
    n_req, N = W.FLOW_REQUESTS, W.FLOW_N_1024
    b = W.flow_branches(W.rng_for(30, 730), n_req, N)
    st = W.flow_state(W.rng_for(30, 731), n_req, N)
    p = W.FLOW_POLICY
    steps = [3 * i for i in range(n_req)]
    pol = torch.tensor([(float(SCHED[i]), p["s_text"], p["s_img"], p["t_lo"], p["t_hi"], p["renorm_min"])
                        for i in steps], dtype=torch.float32, device="cuda")
    times = torch.tensor(np.array([(SCHED[i], SCHED[i + 1]) for i in steps], dtype=F32), device="cuda")
    d = {k: v.cuda() for k, v in b.items()}
    d.update({k: v.cuda() for k, v in st.items() if k != "v"})
    v, xn, lp = _chain(d, pol, times)
    ws = torch.zeros(mot.mot_flow_workspace_bytes(n_req, N), dtype=torch.uint8, device="cuda")
    xn2, lp2 = mot.mot_flow_cfg_sde_step(d["c"], d["tu"], d["iu"], pol, d["x"], d["z"], times, ws=ws)
    assert mot.mot_device_status(ws) == 0
    assert_f32_bitwise(xn2, xn, "full-size fused x_next")
    assert_f32_bitwise(lp2, lp, "full-size fused logp")
    xn16 = _at_16_bytes(torch.zeros((n_req, N)))
    v16 = _at_16_bytes(torch.zeros((n_req, N)))
    _, lp16 = mot.mot_flow_cfg_sde_step(d["c"], d["tu"], d["iu"], pol, _at_16_bytes(d["x"]), _at_16_bytes(d["z"]),
                                        times, ws=ws, x_next=xn16, v_out=v16)
    assert mot.mot_device_status(ws) == 0
    assert_f32_bitwise(xn16, xn, "16-byte-aligned fused x_next")
    assert_f32_bitwise(lp16, lp, "16-byte-aligned fused logp")
    assert_f32_bitwise(v16, v, "16-byte-aligned fused v")
