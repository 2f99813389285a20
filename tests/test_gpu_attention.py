"""Joint attention of packed sequences on the GPU, through the C ABI, against the oracle.

[RFC][BAGEL-7B-MoT][CUDA/ROCm] WS1/WS2 kernel roadmap #435: §1 Motivation item 2 (latent tokens
query the prompt KV non-causally at every step), §2 Reference hazards (cached prefill needs a
bottom-right causal mask), §3 Numerical contract (no split-KV; a row's bits do not depend on
the pack). The fp64 golden is the reference within the tolerance; the kernel is also checked
against itself bit for bit across packs.
"""

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W
from oracle import mot_oracle as O

from _util import assert_bitwise, assert_tolerance, f64, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _qkv(T, Hq, Hkv, D, seed):
    """Post-RoPE q/k/v stand-ins: bf16 N(0, 1) rows of the fused layout."""
    return W.bf16_normal(W.rng_for(seed, 500), (T, (Hq + 2 * Hkv) * D))


def _run(qkv, seqs, Hq, Hkv, D, out=None):
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    s = torch.tensor(seqs, dtype=torch.int32, device="cuda")
    out = mot.mot_joint_attention(qkv.cuda(), s, Hq, Hkv, D, ws, out=out)
    flags = mot.mot_device_status(ws)
    return out, flags


def _query_rows(seqs):
    return np.concatenate([np.arange(q0, q0 + nq) for q0, k0, nq, nk, nc in seqs])


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 8, 1), (128, 28, 4)])
def test_attention_packed_causal_and_latent_vs_golden(D, Hq, Hkv):
    # two sequences of prompt rows then latent rows, ragged lengths over several tiles
    seqs = [(0, 0, 300, 300, 200), (300, 300, 213, 213, 77)]
    T = 513
    qkv = _qkv(T, Hq, Hkv, D, seed=D + Hq)
    out, flags = _run(qkv, seqs, Hq, Hkv, D)
    assert flags == 0
    g = O.g_joint_attention(f64(qkv), seqs, Hq, Hkv, D)
    rows = _query_rows(seqs)
    assert_tolerance(f64(out)[rows], g["out_pre"][rows], f"attention D={D} Hq={Hq} Hkv={Hkv}")


def test_attention_cached_prefix_bottom_right_and_latents_only():
    # sequence 1: 70 new prompt rows after a 250-row cached prefix (keys = prefix + new rows);
    # sequence 2: 64 latent rows querying 200 prompt rows plus themselves (no causal rows);
    # sequence 3: a single causal query at the bottom right of 129 keys
    D, Hq, Hkv = 128, 4, 2
    T = 1000
    seqs = [(250, 0, 70, 320, 70), (520, 320, 64, 264, 0), (900, 771, 1, 129, 1)]
    qkv = _qkv(T, Hq, Hkv, D, seed=7)
    # rows that are no sequence's query keep what the caller left there
    sentinel = torch.full((T, Hq * D), -7.0, dtype=torch.bfloat16, device="cuda")
    out, flags = _run(qkv, seqs, Hq, Hkv, D, out=sentinel.clone())
    assert flags == 0
    g = O.g_joint_attention(f64(qkv), seqs, Hq, Hkv, D)
    rows = _query_rows(seqs)
    assert_tolerance(f64(out)[rows], g["out_pre"][rows], "cached prefix / latents only")
    others = np.setdiff1d(np.arange(T), rows)
    assert torch.equal(out[torch.from_numpy(others).cuda()], sentinel[: len(others)])


def test_attention_full_tiles_leave_neighbouring_rows_untouched():
    # sequences of whole 128-row tiles (written by tensor stores) between untouched rows
    D, Hq, Hkv = 128, 4, 2
    T = 1280
    seqs = [(128, 0, 256, 384, 128), (640, 512, 512, 640, 0)]
    qkv = _qkv(T, Hq, Hkv, D, seed=8)
    sentinel = torch.full((T, Hq * D), 3.0, dtype=torch.bfloat16, device="cuda")
    out, flags = _run(qkv, seqs, Hq, Hkv, D, out=sentinel.clone())
    assert flags == 0
    g = O.g_joint_attention(f64(qkv), seqs, Hq, Hkv, D)
    rows = _query_rows(seqs)
    assert_tolerance(f64(out)[rows], g["out_pre"][rows], "whole tiles")
    others = np.setdiff1d(np.arange(T), rows)
    assert torch.equal(out[torch.from_numpy(others).cuda()], sentinel[: len(others)])


def test_attention_rows_do_not_depend_on_the_pack():
    D, Hq, Hkv = 128, 8, 2
    base = _qkv(400, Hq, Hkv, D, seed=11)
    alone, _ = _run(base, [(0, 0, 400, 400, 250)], Hq, Hkv, D)
    # the same sequence at another offset, after another sequence, in a longer pack
    other = _qkv(333, Hq, Hkv, D, seed=12)
    packed = torch.cat([other, base, _qkv(50, Hq, Hkv, D, seed=13)])
    out, flags = _run(packed, [(0, 0, 333, 333, 100), (333, 333, 400, 400, 250)], Hq, Hkv, D)
    assert flags == 0
    assert_bitwise(out[333:733], alone[:400], "a sequence alone vs packed")
    again, _ = _run(packed, [(0, 0, 333, 333, 100), (333, 333, 400, 400, 250)], Hq, Hkv, D)
    assert_bitwise(again, out, "repeat")


def test_attention_more_than_64_sequences():
    # past 64 sequences the grid takes the items sequence by sequence instead of heaviest first
    D, Hq, Hkv = 64, 2, 1
    rng = W.rng_for(9, 501)
    lens = rng.integers(1, 40, 70)
    seqs, q0 = [], 0
    for i, n in enumerate(lens):
        n = int(n)
        seqs.append((q0, q0, n, n, n if i % 3 else n // 2))   # causal, half causal, ...
        q0 += n
    T = q0 + 5
    qkv = _qkv(T, Hq, Hkv, D, seed=16)
    out, flags = _run(qkv, seqs, Hq, Hkv, D)
    assert flags == 0
    g = O.g_joint_attention(f64(qkv), seqs, Hq, Hkv, D)
    rows = _query_rows(seqs)
    assert_tolerance(f64(out)[rows], g["out_pre"][rows], "70 sequences")


def test_attention_bad_descriptor_flags():
    D, Hq, Hkv = 64, 2, 1
    qkv = _qkv(100, Hq, Hkv, D, seed=14)
    for seqs in ([(0, 0, 50, 40, 10)], [(90, 0, 20, 20, 0)], [(0, 0, 60, 60, 0), (30, 0, 60, 60, 0)]):
        _, flags = _run(qkv, seqs, Hq, Hkv, D)
        assert flags & mot.DEV_BAD_SEQUENCE, seqs


def test_attention_bagel_layer_full_size_sampled():
    # the BAGEL layer's pack: one sequence of 3072 prompt rows (causal) and 1024 latent rows
    shape, inp = W.bagel_layer(seed=1, T=4096)
    T, Hq, Hkv, D = 4096, shape.Hq, shape.Hkv, shape.D
    qkv = _qkv(T, Hq, Hkv, D, seed=15)
    out, flags = _run(qkv, [(0, 0, T, T, 3072)], Hq, Hkv, D)
    assert flags == 0
    rows = np.unique(np.concatenate([W.rng_for(15, 501).choice(T, 48, replace=False), [0, 127, 128, 3071, 3072, 4095]]))
    q = f64(qkv)
    got, want = [], []
    for r in rows:
        # one query at the bottom right of keys 0..r (prompt row) or of all keys (latent row)
        seq = (int(r), 0, 1, int(r) + 1, 1) if r < 3072 else (int(r), 0, 1, T, 0)
        g = O.g_joint_attention(q, [seq], Hq, Hkv, D)
        want.append(g["out_pre"][r])
        got.append(f64(out)[r])
    assert_tolerance(np.array(got), np.array(want), "BAGEL layer attention, sampled rows")


def test_attention_cfg_pack_whole_sequences():
    # The CFG pack bench.py times: 12 sequences of 2048 causal prompt rows and 1024 latent rows
    # (T = 36864), 28 query / 4 KV heads of 128, the same device-drawn Q/K/V; every output
    # element of the first and the last sequence against the fp64 golden.
    T, Hq, Hkv, D = 36864, 28, 4, 128
    seqs = [(3072 * i, 3072 * i, 3072, 3072, 2048) for i in range(12)]
    qkv = W.bf16_normal_device(9, 600, (T, (Hq + 2 * Hkv) * D), "cuda")
    out, flags = _run(qkv, seqs, Hq, Hkv, D)
    assert flags == 0
    for i in (0, 11):
        rows = slice(3072 * i, 3072 * (i + 1))
        g = O.g_joint_attention(f64(qkv[rows]), [(0, 0, 3072, 3072, 2048)], Hq, Hkv, D)
        assert_tolerance(f64(out[rows]), g["out_pre"], f"CFG pack attention, sequence {i} (all rows and heads)")
