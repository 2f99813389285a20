"""The end-to-end parity checker proves a cause for every element beyond the tolerance.

Runs on the CPU. A stand-in for the device path -- the routed QKV GEMM accumulated in fp32 by
numpy and cast to bf16 once, followed by the fp32 contract emulator's QK norm and RoPE -- is
checked against the fp64 golden on the BAGEL layer shape at T = 4096. The checker must accept
it, and must reject planted mistakes that the previous co-occurrence rule let through: an
output element moved by 0.03 in a head whose q has a one-step flip elsewhere, and a
GEMM output moved past its accumulation bound.
"""

import numpy as np
import pytest
import torch

from mixture_transformers_token_gb300 import workloads as W
from oracle import mot_oracle as O

from _util import bf16_step, check_end_to_end, f64


@pytest.fixture(scope="module")
def stand_in():
    shape, inp = W.bagel_layer(seed=2, T=4096)
    x, wq = f64(inp["x"]), f64(inp["w_qkv"])
    mod, pos = inp["mod"].numpy(), inp["pos"].numpy()
    qn, kn = f64(inp["q_norm"]), f64(inp["k_norm"])
    g = O.g_qkv_norm_rope(x, wq, None, qn, kn, pos, mod, shape.Hq, shape.Hkv, shape.D, shape.eps, shape.theta)
    acc32 = np.zeros((shape.T, shape.n_qkv), np.float32)
    for e in (0, 1):
        r = mod == e
        acc32[r] = x[r].astype(np.float32) @ wq[e].astype(np.float32).T
    q = O.bf16(acc32.astype(np.float64))
    c, s = O.rope_cos_sin(shape.theta, shape.D, pos)
    out, _, ue = O.e_qk_norm_rope(q, qn, kn, c, s, mod, shape.Hq, shape.Hkv, shape.D, shape.eps, return_stats=True)
    acc_abs = O.g_routed_matmul(np.abs(x), np.abs(wq), mod)
    epi = {"q_norm": qn, "k_norm": kn, "pos": pos, "mod": mod}
    return shape, g, q, out.astype(np.float64), ue.astype(np.float64), acc_abs, epi


def test_checker_accepts_the_fp32_stand_in(stand_in):
    shape, g, q, out, ue, acc_abs, epi = stand_in
    r = check_end_to_end(out, g, q, ue, acc_abs, shape, "fp32 stand-in", "bf16", epi)
    assert r["q_flips"] > 0
    assert r["beyond"] == r["gemm_cause"] + r["stats_cause"]


def test_checker_rejects_an_element_moved_in_a_head_with_a_q_flip(stand_in):
    shape, g, q, out, ue, acc_abs, epi = stand_in
    D = shape.D
    flips = q[:, : (shape.Hq + shape.Hkv) * D] != g["q"][:, : (shape.Hq + shape.Hkv) * D]
    r, c = map(int, np.argwhere(flips)[0])
    head = c // D
    # another element of the same head, the one of largest magnitude, moved by 0.03
    cols = np.array([k for k in range(head * D, head * D + D) if k != c])
    col = int(cols[np.argmax(np.abs(out[r, cols]))])
    bad = out.copy()
    step = bf16_step(bad[r, col])
    bad[r, col] += np.ceil(0.03 / step) * step
    assert abs(bad[r, col] - g["out_pre"][r, col]) > 2e-2
    with pytest.raises(AssertionError, match="no proven cause"):
        check_end_to_end(bad, g, q, ue, acc_abs, shape, "planted", "bf16", epi)


def test_checker_rejects_a_gemm_output_past_its_bound(stand_in):
    shape, g, q, out, ue, acc_abs, epi = stand_in
    bad = q.copy()
    bad[7, 100] = O.bf16(np.array(bad[7, 100] + 16 * bf16_step(bad[7, 100]) + 2 * shape.H * 2.0 ** -24 * acc_abs[7, 100]))
    with pytest.raises(AssertionError, match="accumulation bound"):
        check_end_to_end(out, g, bad, ue, acc_abs, shape, "planted", "bf16", epi)
