"""Batch invariance on the GPU: a row's output bytes do not depend on the pack it is in.

The requirement is stated in [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap #435, §1
Motivation item 1 (a row's bytes must not depend on the modality mix of the pack) and §2
Reference hazards (sequential, CFG-parallel, SP and step-batched paths pack rows differently);
the sweep follows the methodology of [WS1][CUDA][Qwen3-Next] MoE route/combine contract #503
(each item alone and inside sub-batches of 2, 7 and 64 at other offsets, and in a shuffled
order) and compares raw bits (signed zero distinct). Both RoPE profiles of the QKV projection
are swept.

2048 reference rows of the tiny layer shape (hidden 256, 4 Q / 2 KV heads of 64), each with
its own modality, position and data, are re-packed into packs of 8192 rows whose gen fraction
is 0, 1/8, 1/4, 1/2, 3/4 or 1 (at 0 and 1 only the reference rows of that modality take
part), with contiguous (und block then gen block) and interleaved routing and a shuffled
order. Every reference row's outputs -- y and res_out of the norm, the QKV projection in both
RoPE profiles, the cast and the SwiGLU GEMM -- must be bit-identical to its outputs in the
reference pack.
"""

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W

from _util import bits, need_gpu

pytestmark = pytest.mark.gpu

H, HQ, HKV, D, THETA, EPS = 256, 4, 2, 64, 1e6, 1e-6
N = (HQ + 2 * HKV) * D
N_REF, PACK, P = 2048, 8192, 4096


@pytest.fixture(scope="module")
def setup():
    need_gpu()
    dev = "cuda"
    ref = {
        "x": W.bf16_normal(W.rng_for(21, 1), (N_REF, H)),
        "res": W.bf16_normal(W.rng_for(21, 2), (N_REF, H)),
        "mod": W.modality_bernoulli(W.rng_for(21, 3), N_REF),
        "pos": torch.from_numpy(W.rng_for(21, 4).integers(0, P, N_REF).astype(np.int32)),
    }
    weights = {
        "w_norm": W.bf16_normal(W.rng_for(21, 5), (2, H), mean=1.0, std=0.1).to(dev),
        "w_qkv": W.bf16_normal(W.rng_for(21, 6), (2, N, H), std=0.02).to(dev),
        "q_norm": W.bf16_normal(W.rng_for(21, 7), (2, D), mean=1.0, std=0.1).to(dev),
        "k_norm": W.bf16_normal(W.rng_for(21, 8), (2, D), mean=1.0, std=0.1).to(dev),
        "w_o": W.bf16_normal(W.rng_for(21, 9), (2, 512, H), std=0.02).to(dev),
        "cs": mot.mot_rope_table_fill_host(THETA, D, P).to(dev),
        "cs32": mot.mot_rope_table_fill_host_fp32(THETA, D, P).to(dev),
    }
    weights["w_gu"] = mot.mot_swiglu_interleave(W.bf16_normal(W.rng_for(21, 10), (2, 256, H), std=0.02).to(dev),
                                                W.bf16_normal(W.rng_for(21, 11), (2, 256, H), std=0.02).to(dev))
    base = run_pack(ref, weights)
    return ref, weights, base


def run_pack(pack, wt):
    dev = "cuda"
    x, res, mod, pos = (pack[k].to(dev) for k in ("x", "res", "mod", "pos"))
    ws = mot.mot_route_plan(mod)
    y, ro = mot.mot_fused_add_rmsnorm(x, res, wt["w_norm"], mod, EPS, ws=ws)
    qkv = mot.mot_routed_qkv_norm_rope(y, wt["w_qkv"], wt["q_norm"], wt["k_norm"], pos, wt["cs"], HQ, HKV, D, EPS, ws)
    qkv32 = mot.mot_routed_qkv_norm_rope_fp32(y, wt["w_qkv"], wt["q_norm"], wt["k_norm"], pos, wt["cs32"], HQ, HKV, D,
                                              EPS, ws)
    o = mot.mot_routed_gemm(y, wt["w_o"], ws, mot.EPI_CAST)
    h = mot.mot_routed_gemm(y, wt["w_gu"], ws, mot.EPI_SWIGLU)
    assert mot.mot_device_status(ws) == 0
    return {k: bits(v) for k, v in (("y", y), ("res_out", ro), ("qkv", qkv), ("qkv_fp32_rope", qkv32), ("o", o),
                                    ("h", h))}


def build_pack(ref, sel, slots, T, filler_mod, seed):
    """A pack of T rows: reference rows `sel` at positions `slots`, random filler elsewhere."""
    rng = W.rng_for(seed, 30)
    pack = {
        "x": W.bf16_normal(W.rng_for(seed, 31), (T, H)),
        "res": W.bf16_normal(W.rng_for(seed, 32), (T, H)),
        "mod": filler_mod.clone(),
        "pos": torch.from_numpy(rng.integers(0, P, T).astype(np.int32)),
    }
    for k in pack:
        pack[k][slots] = ref[k][sel]
    return pack


def check_rows(out, base, sel, slots, what):
    for k in base:
        a = out[k][slots]
        b = base[k][sel]
        if not np.array_equal(a, b):
            bad = np.argwhere(np.any(a != b, axis=1))[:, 0]
            raise AssertionError(f"{what}: {k} differs for {len(bad)} reference rows, e.g. {sel[bad[:5]].tolist()}")


@pytest.mark.parametrize("frac", [0.0, 0.125, 0.25, 0.5, 0.75, 1.0])
@pytest.mark.parametrize("layout", ["contiguous", "interleaved", "shuffled"])
def test_pack_mix_and_order(setup, frac, layout):
    ref, wt, base = setup
    rmod = ref["mod"].numpy()
    if frac == 0.0:
        sel = np.nonzero(rmod == 0)[0]
    elif frac == 1.0:
        sel = np.nonzero(rmod == 1)[0]
    else:
        sel = np.arange(N_REF)
    seed = 100 + int(frac * 8) * 3 + ["contiguous", "interleaved", "shuffled"].index(layout)
    rng = W.rng_for(seed, 40)
    n_fill = PACK - len(sel)
    gen_total = int(round(frac * PACK))
    fill_gen = int(np.clip(gen_total - int(rmod[sel].sum()), 0, n_fill))
    fill_mod = np.zeros(n_fill, np.uint8)
    fill_mod[rng.choice(n_fill, fill_gen, replace=False)] = 1
    # row order of the pack: reference rows (tagged >= 0) and filler rows (tagged -1)
    tags = np.concatenate([sel, -np.ones(n_fill, np.int64)])
    mods = np.concatenate([rmod[sel], fill_mod])
    if layout == "contiguous":
        order = np.argsort(mods, kind="stable")                 # all und rows, then all gen rows
    else:
        order = rng.permutation(PACK)
    tags, mods = tags[order], mods[order]
    slots = np.nonzero(tags >= 0)[0]
    sel_in_pack = tags[slots]
    pack = build_pack(ref, torch.from_numpy(sel_in_pack), torch.from_numpy(slots), PACK, torch.from_numpy(mods), seed)
    out = run_pack(pack, wt)
    check_rows(out, base, sel_in_pack, slots, f"frac={frac} {layout}")


@pytest.mark.parametrize("size", [1, 2, 7, 64])
def test_sub_batches_at_other_offsets(setup, size):
    ref, wt, base = setup
    rng = W.rng_for(200 + size, 41)
    groups = 16 if size == 1 else 8
    for gi in range(groups):
        sel = np.sort(rng.choice(N_REF, size, replace=False))
        T = size + int(rng.integers(0, 300))
        slots = np.sort(rng.choice(T, size, replace=False))
        fill_mod = torch.from_numpy((rng.random(T) < 0.5).astype(np.uint8))
        pack = build_pack(ref, torch.from_numpy(sel), torch.from_numpy(slots), T, fill_mod, 300 + size * 50 + gi)
        out = run_pack(pack, wt)
        check_rows(out, base, sel, slots, f"sub-batch size {size} group {gi}")


def test_repeat_is_deterministic(setup):
    ref, wt, base = setup
    again = run_pack(ref, wt)
    for k in base:
        assert np.array_equal(again[k], base[k]), k


def _out_at_16_bytes(T, n):
    """A [T][n] bf16 output whose data starts 16 bytes past a 32-byte boundary."""
    buf = torch.empty(T * n + 16, dtype=torch.bfloat16, device="cuda")
    v = buf[8:8 + T * n].view(T, n)
    assert v.data_ptr() % 32 == 16
    return v


def test_outputs_only_16_byte_aligned_give_the_same_bits(setup):
    # the epilogues write whole 32-byte sectors when the output allows it, 16-byte pieces
    # otherwise; both must produce the same bytes
    ref, wt, base = setup
    dev = "cuda"
    x, res, mod, pos = (ref[k].to(dev) for k in ("x", "res", "mod", "pos"))
    ws = mot.mot_route_plan(mod)
    y, _ = mot.mot_fused_add_rmsnorm(x, res, wt["w_norm"], mod, EPS, ws=ws)
    qkv = mot.mot_routed_qkv_norm_rope(y, wt["w_qkv"], wt["q_norm"], wt["k_norm"], pos, wt["cs"], HQ, HKV, D, EPS, ws,
                                       out=_out_at_16_bytes(N_REF, N))
    qkv32 = mot.mot_routed_qkv_norm_rope_fp32(y, wt["w_qkv"], wt["q_norm"], wt["k_norm"], pos, wt["cs32"], HQ, HKV, D,
                                              EPS, ws, out=_out_at_16_bytes(N_REF, N))
    o = mot.mot_routed_gemm(y, wt["w_o"], ws, mot.EPI_CAST, out=_out_at_16_bytes(N_REF, 512))
    h = mot.mot_routed_gemm(y, wt["w_gu"], ws, mot.EPI_SWIGLU, out=_out_at_16_bytes(N_REF, 256))
    assert mot.mot_device_status(ws) == 0
    for k, v in (("qkv", qkv), ("qkv_fp32_rope", qkv32), ("o", o), ("h", h)):
        assert np.array_equal(bits(v), base[k]), k
