"""The allocation-free routed GEMM gives the same results as the workspace entry point.

Some callers cannot allocate device memory: inference engines that reserve all of it at
start-up and refuse later allocations, and plug-ins whose host framework owns the device
memory without lending them an allocator. They cannot pass the routing-plan workspace that
mot_routed_gemm needs, so mot_routed_gemm_noalloc keeps the plan in a fixed array inside the
library. This test calls it through the C ABI twice in a row (different row counts, modality
mixes and epilogues, so a stale plan left in the shared array by the first call would show in
the second) and compares each result with mot_routed_gemm on a caller-owned workspace bit for
bit: both build the same routing plan with the same kernel and run the same GEMM, so the only
difference is where the plan lives. One more call fills the array to its limit of
MOT_NOALLOC_MAX_TOKENS rows.

The file name makes pytest collect it last, so a run that stops at the first failure has
already run every other test; it needs nothing from them and also passes on its own.
"""

import numpy as np
import pytest
import torch

import mixture_transformers_token_gb300 as mot
from mixture_transformers_token_gb300 import workloads as W

from _util import assert_bitwise, f64, need_gpu

pytestmark = pytest.mark.gpu


def _noalloc_through_c_abi(lib, a, w, mod, epilogue, ncols):
    T, K = a.shape
    N = w.shape[1]
    out = torch.full((T, ncols), float("nan"), dtype=torch.bfloat16, device=a.device)
    flags = torch.full((1,), -1, dtype=torch.int32, device=a.device)
    status = lib.mot_routed_gemm_noalloc(a.data_ptr(), w.data_ptr(), mod.data_ptr(), T, N, K, epilogue,
                                         out.data_ptr(), flags.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert status == 0, lib.mot_status_string(status).decode()
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    return out


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    need_gpu()
    lib = mot.load_library()
    dev = torch.device("cuda")
    # call 1: cast epilogue, 1000 rows, 30 % gen rows scattered
    a1 = W.bf16_normal(W.rng_for(31, 1), (1000, 512)).to(dev)
    w1 = W.bf16_normal(W.rng_for(31, 2), (2, 768, 512), std=0.02).to(dev)
    m1 = W.modality_bernoulli(W.rng_for(31, 3), 1000, 0.3).to(dev)
    # call 2: SwiGLU epilogue, 300 rows in und/gen blocks, fewer rows than call 1
    a2 = W.bf16_normal(W.rng_for(32, 1), (300, 256)).to(dev)
    wg = W.bf16_normal(W.rng_for(32, 2), (2, 256, 256), std=0.02).to(dev)
    wu = W.bf16_normal(W.rng_for(32, 3), (2, 256, 256), std=0.02).to(dev)
    w2 = mot.mot_swiglu_interleave(wg, wu)
    m2 = W.modality_blocks([(1, 100), (0, 150), (1, 50)]).to(dev)

    got1 = _noalloc_through_c_abi(lib, a1, w1, m1, mot.EPI_CAST, 768)
    got2 = _noalloc_through_c_abi(lib, a2, w2, m2, mot.EPI_SWIGLU, 256)

    ref1 = mot.mot_routed_gemm(a1, w1, mot.mot_route_plan(m1), mot.EPI_CAST)
    ref2 = mot.mot_routed_gemm(a2, w2, mot.mot_route_plan(m2), mot.EPI_SWIGLU)
    torch.cuda.synchronize()
    assert_bitwise(got1, ref1, "allocation-free call 1 vs mot_routed_gemm")
    assert_bitwise(got2, ref2, "allocation-free call 2 vs mot_routed_gemm")
    assert np.isfinite(f64(got1)).all() and np.isfinite(f64(got2)).all()


def test_noalloc_at_its_row_limit():
    # the largest plan the array holds: MOT_NOALLOC_MAX_TOKENS rows, gen rows scattered so every
    # tile record and the whole row list are written
    need_gpu()
    lib = mot.load_library()
    dev = torch.device("cuda")
    T = mot.NOALLOC_MAX_TOKENS
    a = W.bf16_normal_device(33, 1, (T, 128), dev)
    w = W.bf16_normal_device(33, 2, (2, 256, 128), dev, std=0.02)
    m = W.modality_bernoulli(W.rng_for(33, 3), T, 0.25).to(dev)
    got = _noalloc_through_c_abi(lib, a, w, m, mot.EPI_CAST, 256)
    ref = mot.mot_routed_gemm(a, w, mot.mot_route_plan(m), mot.EPI_CAST)
    torch.cuda.synchronize()
    assert_bitwise(got, ref, "allocation-free call at MOT_NOALLOC_MAX_TOKENS rows vs mot_routed_gemm")


def test_noalloc_rejects_rows_beyond_its_limit():
    need_gpu()
    lib = mot.load_library()
    T = mot.NOALLOC_MAX_TOKENS + 1
    a = torch.empty((T, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((2, 256, 64), dtype=torch.bfloat16, device="cuda")
    m = torch.zeros(T, dtype=torch.uint8, device="cuda")
    out = torch.empty((T, 256), dtype=torch.bfloat16, device="cuda")
    status = lib.mot_routed_gemm_noalloc(a.data_ptr(), w.data_ptr(), m.data_ptr(), T, 256, 64, mot.EPI_CAST,
                                         out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert status == 9 and "MOT_NOALLOC_MAX_TOKENS" in lib.mot_status_string(status).decode()
