"""Seeded synthetic inputs for the MoT token-routed dense projection.

This module only draws random numbers and builds index patterns (modality masks,
positions). It holds none of the method's arithmetic, so both the CUDA path and
the CPU oracle can be fed from it without sharing any computation.

Shapes follow the BAGEL-7B-MoT decoder layer described in RFC #435 "[RFC][BAGEL-7B-MoT]
[CUDA/ROCm] WS1/WS2 kernel roadmap", §1 Motivation (a Qwen2.5-7B-shaped decoder with
two weight sets; 28 query heads per §3 "Required invariances"). Value distributions
stand in for trained weights: activations ~ N(0, 1), projection weights ~ N(0, 0.02),
norm weights ~ 1 + N(0, 0.1).

Random draws are made in float32 with numpy's PCG64 generator and rounded to bf16 by
torch's round-to-nearest-even conversion.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

UND = 0  # understanding expert: text and ViT tokens
GEN = 1  # generation expert: VAE-latent tokens


def rng_for(seed: int, stream: int = 0) -> np.random.Generator:
    """A PCG64 generator for (seed, stream); streams keep tensors independent."""
    return np.random.Generator(np.random.PCG64([seed, stream]))


def bf16_normal(rng: np.random.Generator, shape, mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    """A CPU bf16 tensor of N(mean, std^2) draws."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return torch.from_numpy(a).to(torch.bfloat16)


def bf16_normal_device(seed: int, stream: int, shape, device, mean: float = 0.0, std: float = 1.0) -> torch.Tensor:
    """A device bf16 tensor of N(mean, std^2) draws from torch's seeded generator on `device`.

    Used for the large weights of throughput-only workloads, where drawing on the host would
    dominate the run; inputs that the oracle also sees come from the host generators above.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def bf16_integers(rng: np.random.Generator, shape, lo: int, hi: int) -> torch.Tensor:
    """A CPU bf16 tensor of small integers in [lo, hi] (exact in bf16 when |v| <= 256)."""
    a = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return torch.from_numpy(a).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# modality patterns
# ---------------------------------------------------------------------------

def modality_bernoulli(rng: np.random.Generator, T: int, p_gen: float = 0.5) -> torch.Tensor:
    return torch.from_numpy((rng.random(T) < p_gen).astype(np.uint8))


def modality_blocks(blocks) -> torch.Tensor:
    """Concatenate runs given as [(modality, length), ...]."""
    parts = [np.full(n, m, dtype=np.uint8) for m, n in blocks]
    return torch.from_numpy(np.concatenate(parts) if parts else np.zeros(0, np.uint8))


def modality_scattered(rng: np.random.Generator, T: int, n_gen: int) -> torch.Tensor:
    """Exactly n_gen generation rows chosen uniformly without replacement."""
    m = np.zeros(T, dtype=np.uint8)
    m[rng.choice(T, size=n_gen, replace=False)] = GEN
    return torch.from_numpy(m)


def positions_restarting(lengths) -> torch.Tensor:
    """Positions 0..len-1 for each sequence of a pack, concatenated."""
    return torch.from_numpy(np.concatenate([np.arange(n, dtype=np.int32) for n in lengths]))


# ---------------------------------------------------------------------------
# layer shapes
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class QKVShape:
    T: int
    H: int
    Hq: int
    Hkv: int
    D: int
    theta: float = 1.0e6
    eps: float = 1.0e-6

    @property
    def n_qkv(self) -> int:
        return (self.Hq + 2 * self.Hkv) * self.D


TINY = QKVShape(T=64, H=256, Hq=4, Hkv=2, D=64)
BAGEL_LAYER = QKVShape(T=4096, H=3584, Hq=28, Hkv=4, D=128)
CFG_PACK = QKVShape(T=36864, H=3584, Hq=28, Hkv=4, D=128)
MLP_T, MLP_H, MLP_I = 8192, 3584, 18944


def qkv_layer_inputs(shape: QKVShape, mod: torch.Tensor, pos: torch.Tensor, seed: int,
                     with_bias: bool = False) -> dict:
    """All inputs of one routed QKV layer with a fused add-RMSNorm in front."""
    T, H, D, N = shape.T, shape.H, shape.D, shape.n_qkv
    out = {
        "x": bf16_normal(rng_for(seed, 1), (T, H)),
        "res": bf16_normal(rng_for(seed, 2), (T, H)),
        "w_norm": bf16_normal(rng_for(seed, 3), (2, H), mean=1.0, std=0.1),
        "w_qkv": bf16_normal(rng_for(seed, 4), (2, N, H), std=0.02),
        "q_norm": bf16_normal(rng_for(seed, 5), (2, D), mean=1.0, std=0.1),
        "k_norm": bf16_normal(rng_for(seed, 6), (2, D), mean=1.0, std=0.1),
        "b_qkv": bf16_normal(rng_for(seed, 7), (2, N), std=0.5) if with_bias else None,
        "mod": mod,
        "pos": pos,
    }
    return out


def tiny_layer(seed: int = 1) -> tuple[QKVShape, dict]:
    """64 packed tokens, hidden 256, 4 Q / 2 KV heads of 64, Bernoulli(0.5) modality, positions 0..63."""
    s = TINY
    mod = modality_bernoulli(rng_for(seed, 0), s.T)
    pos = torch.arange(s.T, dtype=torch.int32)
    return s, qkv_layer_inputs(s, mod, pos, seed)


def bagel_layer(seed: int = 1, T: int = 4096) -> tuple[QKVShape, dict]:
    """BAGEL-shaped layer: 3/4 text (und) rows, then a contiguous gen block (32x32 latents at T=4096)."""
    s = QKVShape(T=T, H=3584, Hq=28, Hkv=4, D=128)
    n_und = (3 * T) // 4
    mod = modality_blocks([(UND, n_und), (GEN, T - n_und)])
    pos = torch.arange(T, dtype=torch.int32)
    return s, qkv_layer_inputs(s, mod, pos, seed)


def cfg_pack_layout(n_seq: int = 12, n_und: int = 2048, n_gen: int = 1024):
    """Modality and positions of a CFG pack: n_seq sequences of (n_und text, n_gen latent) rows."""
    mod = modality_blocks([b for _ in range(n_seq) for b in ((UND, n_und), (GEN, n_gen))])
    pos = positions_restarting([n_und + n_gen] * n_seq)
    return mod, pos


def mlp_inputs(T: int, H: int, I: int, n_gen: int, seed: int) -> dict:
    """Routed SwiGLU MLP inputs: separate gate and up weights [2][I][H], down weights [2][H][I]."""
    return {
        "x": bf16_normal(rng_for(seed, 11), (T, H)),
        "res": bf16_normal(rng_for(seed, 12), (T, H)),
        "w_norm": bf16_normal(rng_for(seed, 13), (2, H), mean=1.0, std=0.1),
        "w_gate": bf16_normal(rng_for(seed, 14), (2, I, H), std=0.02),
        "w_up": bf16_normal(rng_for(seed, 15), (2, I, H), std=0.02),
        "w_down": bf16_normal(rng_for(seed, 16), (2, H, I), std=0.02),
        "mod": modality_scattered(rng_for(seed, 10), T, n_gen),
    }


def mlp_device_inputs(device, seed: int = 3) -> dict:
    """Routed SwiGLU MLP at T = 8192, hidden 3584, intermediate 18944, exactly 2048 gen rows
    scattered uniformly: x, res, norm weights and separate gate / up / down weights drawn on the
    device (the modality index on the host)."""
    t, h, i = MLP_T, MLP_H, MLP_I
    return {
        "x": bf16_normal_device(seed, 1, (t, h), device),
        "res": bf16_normal_device(seed, 2, (t, h), device),
        "w_norm": bf16_normal_device(seed, 3, (2, h), device, mean=1.0, std=0.1),
        "w_gate": bf16_normal_device(seed, 4, (2, i, h), device, std=0.02),
        "w_up": bf16_normal_device(seed, 5, (2, i, h), device, std=0.02),
        "w_down": bf16_normal_device(seed, 6, (2, h, i), device, std=0.02),
        "mod": modality_scattered(rng_for(seed, 7), t, 2048).to(device),
    }


def cfg_pack_device_inputs(device, seed: int = 5) -> dict:
    """CFG pack: 12 sequences of 2048 und + 1024 gen rows (T = 36864), positions restarting per
    sequence; `attn` stands in for the attention output that feeds the routed O projection."""
    s = CFG_PACK
    t, h = s.T, s.H
    mod, pos = cfg_pack_layout()
    return {
        "mod": mod.to(device), "pos": pos.to(device),
        "x": bf16_normal_device(seed, 1, (t, h), device),
        "res": bf16_normal_device(seed, 2, (t, h), device),
        "attn": bf16_normal_device(seed, 3, (t, h), device),
        "w_norm": bf16_normal_device(seed, 4, (2, h), device, mean=1.0, std=0.1),
        "w_qkv": bf16_normal_device(seed, 5, (2, s.n_qkv, h), device, std=0.02),
        "q_norm": bf16_normal_device(seed, 6, (2, s.D), device, mean=1.0, std=0.1),
        "k_norm": bf16_normal_device(seed, 7, (2, s.D), device, mean=1.0, std=0.1),
        "w_o": bf16_normal_device(seed, 8, (2, h, h), device, std=0.02),
    }


# Flow sampler. BAGEL's latents are VAE latents (8x downsampling, 16 channels) patchified 2 x 2,
# so a 1024 x 1024 image is 64 x 64 latent tokens of 64 values: N = 262144 per request; a
# 512 x 512 image has N = 65536. 50 steps with shift 3 and the window [0.4, 1] are the settings
# under which the schedule gives the 41 guided steps of RFC #435 §2; the scales (text 4, image 2)
# and renorm min 0 are stand-ins, since the pages fix no values for them.
FLOW_N_1024 = 64 * 64 * 64
FLOW_N_512 = 32 * 32 * 64
FLOW_REQUESTS = 16
FLOW_POLICY = {"s_text": 4.0, "s_img": 2.0, "t_lo": 0.4, "t_hi": 1.0, "renorm_min": 0.0}
FLOW_STEPS, FLOW_SHIFT = 50, 3.0


def flow_branches(rng: np.random.Generator, n_req: int, N: int, spread: float = 0.5) -> dict:
    """Three CFG branches [n_req][N] bf16: the conditioned velocity c ~ N(0, 1) and the text- and
    image-unconditioned ones, c plus N(0, spread^2) draws (the branches of one request are the
    same model's outputs on the same latent, so they are correlated)."""
    c = rng.standard_normal(size=(n_req, N), dtype=np.float32)
    tu = c + np.float32(spread) * rng.standard_normal(size=(n_req, N), dtype=np.float32)
    iu = c + np.float32(spread) * rng.standard_normal(size=(n_req, N), dtype=np.float32)
    return {k: torch.from_numpy(v).to(torch.bfloat16) for k, v in (("c", c), ("tu", tu), ("iu", iu))}


def flow_state(rng: np.random.Generator, n_req: int, N: int) -> dict:
    """SDE step inputs [n_req][N] fp32: the latent x ~ N(0, 1), a velocity v ~ N(0, 1) and the
    step's standard normal noise z."""
    return {k: torch.from_numpy(rng.standard_normal(size=(n_req, N), dtype=np.float32)) for k in ("x", "v", "z")}
