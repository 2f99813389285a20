"""Batch invariance at the timed BAGEL layer shape: a row's output bytes do not depend on the pack.

The requirement is stated in [RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap #435, §1
Motivation item 1 (a row's bytes must not depend on the modality mix of the pack) and §2
Reference hazards (sequential, CFG-parallel, SP and step-batched paths pack rows differently);
the sweep follows [WS1][CUDA][Qwen3-Next] MoE route/combine contract #503 (items alone and in
sub-batches of 7 and 64 at other offsets, shuffled order) and compares raw bits.

This is the shape bench.py times: hidden 3584, 28 Q / 4 KV heads of 128 (QKV out 4608, 56
K-blocks of 64), the fused add-RMSNorm at H = 3584, the QKV epilogue in both RoPE profiles,
the cast and SwiGLU GEMMs at K = 3584 and the cast GEMM at K = 18944 (the down projection's
reduction length), the MLP chain also through the plan-order flags bench.py uses. 256
reference rows, each with its own modality, position and data, are re-packed into packs of
1024 rows with gen fraction 0, 1/4 or 1 (at 0 and 1 only the reference rows of that modality
take part), in contiguous, interleaved and shuffled layouts.
"""

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W

from _util import bits, need_gpu

pytestmark = pytest.mark.gpu

H, HQ, HKV, D, I, THETA, EPS = 3584, 28, 4, 128, 18944, 1e6, 1e-6
N = (HQ + 2 * HKV) * D
N_REF, PACK, P = 256, 1024, 4096
KEYS = ("x", "res", "mod", "pos", "hid")


@pytest.fixture(scope="module")
def setup():
    need_gpu()
    dev = "cuda"
    ref = {
        "x": W.bf16_normal(W.rng_for(61, 1), (N_REF, H)),
        "res": W.bf16_normal(W.rng_for(61, 2), (N_REF, H)),
        "mod": W.modality_bernoulli(W.rng_for(61, 3), N_REF),
        "pos": torch.from_numpy(W.rng_for(61, 4).integers(0, P, N_REF).astype(np.int32)),
        "hid": W.bf16_normal(W.rng_for(61, 5), (N_REF, I)),
    }
    weights = {
        "w_norm": W.bf16_normal_device(61, 10, (2, H), dev, mean=1.0, std=0.1),
        "w_qkv": W.bf16_normal_device(61, 11, (2, N, H), dev, std=0.02),
        "q_norm": W.bf16_normal_device(61, 12, (2, D), dev, mean=1.0, std=0.1),
        "k_norm": W.bf16_normal_device(61, 13, (2, D), dev, mean=1.0, std=0.1),
        "w_o": W.bf16_normal_device(61, 14, (2, 512, H), dev, std=0.02),
        "w_gu": mot.mot_swiglu_interleave(W.bf16_normal_device(61, 15, (2, 256, H), dev, std=0.02),
                                          W.bf16_normal_device(61, 16, (2, 256, H), dev, std=0.02)),
        "w_down": W.bf16_normal_device(61, 17, (2, 256, I), dev, std=0.02),
        "cs": mot.mot_rope_table_fill_host(THETA, D, P).to(dev),
        "cs32": mot.mot_rope_table_fill_host_fp32(THETA, D, P).to(dev),
    }
    base = run_pack(ref, weights)
    return ref, weights, base


def run_pack(pack, wt):
    dev = "cuda"
    x, res, mod, pos, hid = (pack[k].to(dev) for k in KEYS)
    T = x.shape[0]
    ws = mot.mot_route_plan(mod)
    y, ro = mot.mot_fused_add_rmsnorm(x, res, wt["w_norm"], mod, EPS, ws=ws)
    qkv = mot.mot_routed_qkv_norm_rope(y, wt["w_qkv"], wt["q_norm"], wt["k_norm"], pos, wt["cs"], HQ, HKV, D, EPS, ws)
    qkv32 = mot.mot_routed_qkv_norm_rope_fp32(y, wt["w_qkv"], wt["q_norm"], wt["k_norm"], pos, wt["cs32"], HQ, HKV, D,
                                              EPS, ws)
    o = mot.mot_routed_gemm(y, wt["w_o"], ws, mot.EPI_CAST)
    h = mot.mot_routed_gemm(y, wt["w_gu"], ws, mot.EPI_SWIGLU)
    dn = mot.mot_routed_gemm(hid, wt["w_down"], ws, mot.EPI_CAST)
    # the MLP chain as bench.py runs it: rows into plan order, gate/up in and out of plan order,
    # down from plan order back to token order
    y_plan = mot.mot_gather_rows(y, ws)
    h_plan = mot.mot_routed_gemm(y_plan, wt["w_gu"], ws, mot.EPI_SWIGLU | mot.A_PLAN_ORDER | mot.OUT_PLAN_ORDER)
    hid_plan = mot.mot_gather_rows(hid, ws)
    dn_plan = mot.mot_routed_gemm(hid_plan, wt["w_down"], ws, mot.EPI_CAST | mot.A_PLAN_ORDER)
    assert mot.mot_device_status(ws) == 0
    m = pack["mod"].numpy()
    perm = np.concatenate([np.nonzero(m == 0)[0], np.nonzero(m == 1)[0]])
    inv = np.empty(T, np.int64)
    inv[perm] = np.arange(T)
    h_tok = bits(h_plan)[inv]
    return {k: bits(v) for k, v in (("y", y), ("res_out", ro), ("qkv", qkv), ("qkv_fp32_rope", qkv32), ("o", o),
                                    ("h", h), ("down_K18944", dn), ("down_plan_order_in", dn_plan))} | \
        {"h_plan_order": h_tok}


def build_pack(ref, sel, slots, T, filler_mod, seed):
    """A pack of T rows: reference rows `sel` at positions `slots`, random filler elsewhere."""
    rng = W.rng_for(seed, 30)
    pack = {
        "x": W.bf16_normal(W.rng_for(seed, 31), (T, H)),
        "res": W.bf16_normal(W.rng_for(seed, 32), (T, H)),
        "mod": filler_mod.clone(),
        "pos": torch.from_numpy(rng.integers(0, P, T).astype(np.int32)),
        "hid": W.bf16_normal(W.rng_for(seed, 33), (T, I)),
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


def test_plan_order_chain_matches_token_order(setup):
    # the plan-order flags only move rows: the same bits as the token-order GEMMs
    _, _, base = setup
    assert np.array_equal(base["h_plan_order"], base["h"])
    assert np.array_equal(base["down_plan_order_in"], base["down_K18944"])


@pytest.mark.parametrize("frac", [0.0, 0.25, 1.0])
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
    seed = 700 + int(frac * 8) * 3 + ["contiguous", "interleaved", "shuffled"].index(layout)
    rng = W.rng_for(seed, 40)
    n_fill = PACK - len(sel)
    gen_total = int(round(frac * PACK))
    fill_gen = int(np.clip(gen_total - int(rmod[sel].sum()), 0, n_fill))
    fill_mod = np.zeros(n_fill, np.uint8)
    fill_mod[rng.choice(n_fill, fill_gen, replace=False)] = 1
    tags = np.concatenate([sel, -np.ones(n_fill, np.int64)])
    mods = np.concatenate([rmod[sel], fill_mod])
    if layout == "contiguous":
        order = np.argsort(mods, kind="stable")                 # all und rows, then all gen rows
    elif layout == "interleaved":
        # und and gen rows alternate as far as the counts allow, reference rows spread through
        und, gen = np.nonzero(mods == 0)[0], np.nonzero(mods == 1)[0]
        und, gen = rng.permutation(und), rng.permutation(gen)
        k = min(len(und), len(gen))
        order = np.concatenate([np.stack([und[:k], gen[:k]], axis=1).reshape(-1), und[k:], gen[k:]])
    else:
        order = rng.permutation(PACK)
    tags, mods = tags[order], mods[order]
    slots = np.nonzero(tags >= 0)[0]
    sel_in_pack = tags[slots]
    pack = build_pack(ref, torch.from_numpy(sel_in_pack), torch.from_numpy(slots), PACK, torch.from_numpy(mods), seed)
    out = run_pack(pack, wt)
    check_rows(out, base, sel_in_pack, slots, f"frac={frac} {layout}")


@pytest.mark.parametrize("size", [1, 7, 64])
def test_sub_batches_at_other_offsets(setup, size):
    ref, wt, base = setup
    rng = W.rng_for(800 + size, 41)
    groups = 8 if size == 1 else 4
    for gi in range(groups):
        sel = np.sort(rng.choice(N_REF, size, replace=False))
        T = size + int(rng.integers(0, 300))
        slots = np.sort(rng.choice(T, size, replace=False))
        fill_mod = torch.from_numpy((rng.random(T) < 0.5).astype(np.uint8))
        pack = build_pack(ref, torch.from_numpy(sel), torch.from_numpy(slots), T, fill_mod, 900 + size * 50 + gi)
        out = run_pack(pack, wt)
        check_rows(out, base, sel, slots, f"sub-batch size {size} group {gi}")
