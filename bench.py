#!/usr/bin/env python
"""Benchmark of the MoT token-routed projection step on GB300.

One step is one pass of the projection path over a packed batch: the routing pre-pass,
the fused residual-add RMSNorm and the routed QKV GEMM with its per-head QK RMSNorm and BF16
RoPE epilogue. The workload is the BAGEL-shaped layer: T = 4096 packed bf16 tokens, hidden
3584, Q 28 x 128, KV 4 x 128 (QKV out 4608), und/gen weight sets W ~ N(0, 0.02), the first 3072
tokens und then a contiguous 1024-token gen block, positions 0..4095, eps 1e-6, theta 1e6.
Inputs are synthetic and seeded (one pack per rank); L2 is flushed (a write and a read of twice its
size) before every timed step, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is whole-job TFLOP/s of the routed QKV projection
(2 T H N flops per rank) over the whole step time, max over ranks. `--impl reference` times
the CPU oracle on the host cores instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed QKV+QKnorm+RoPE TFLOP/s at T=4096 (% BF16 peak); add-RMSNorm GB/s"
WORKLOAD = "bagel_layer_T4096_H3584_q28x128_kv4x128_und3072_gen1024"
T, H, HQ, HKV, D = 4096, 3584, 28, 4, 128
N_QKV = (HQ + 2 * HKV) * D
QKV_FLOPS = 2 * T * H * N_QKV                     # 135.29 GFLOP per step
NORM_BYTES = 8 * T * H + 4 * H + T                # read x, res; write y, res_out; weights; modality

# DRAM traffic of one QKV kernel launch from an ncu capture of this workload, keyed by the
# hash of the kernel source it was taken on (null once the kernel has changed).
NCU_TRAFFIC = {"b2d0b5f87d477e24": 119274496}   # profiles/routed_gemm_qkv128_bagel_layer_T4096.md


def src_hash(name: str) -> str:
    p = os.path.join(ROOT, "mixture_transformers_token_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "of measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "of fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5:
            time.sleep(0.05)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        inside = [r for t, r in self.rows if self.t_start - 0.05 <= t <= self.t_end + 0.15]
        if not inside:
            inside = [r for _, r in self.rows]
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((float(r[4]) for r in inside if r[4].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def make_inputs(seed: int, dev):
    import torch

    from mixture_transformers_token_gb300 import workloads as W

    shape, inp = W.bagel_layer(seed=seed, T=T)
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    return shape, inp, d


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import build as mot_build

    if rank == 0 or world == 1:
        mot_build.build()
    if world > 1:
        dist.barrier()
    mot.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shape, inp, d = make_inputs(1 + rank, dev)
    stream = torch.cuda.current_stream(dev)
    cs = mot.mot_rope_table_fill_host(shape.theta, D, T).to(dev)
    ws = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ro = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, N_QKV), dtype=torch.bfloat16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20) // 4, dtype=torch.int32, device=dev)

    def flush_l2(i):
        # write twice L2 (evicts everything, our outputs' dirty lines are written back here),
        # then read it back so the timed step starts with only clean lines in L2
        flush.fill_(i)
        flush.sum()

    def step(x, res):
        # the norm launch also writes the routing plan of mod into ws (one extra CTA)
        mot.mot_fused_add_rmsnorm(x, res, d["w_norm"], d["mod"], shape.eps, y=y, res_out=ro, ws=ws)
        mot.mot_routed_qkv_norm_rope(y, d["w_qkv"], d["q_norm"], d["k_norm"], d["pos"], cs, HQ, HKV, D, shape.eps,
                                     ws, out=out)

    for i in range(args.warmup):
        flush_l2(i)
        step(d["x"], d["res"])
    torch.cuda.synchronize()
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("start")
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush_l2(i)
        e = ev[i]
        e[0].record(stream)
        mot.mot_fused_add_rmsnorm(d["x"], d["res"], d["w_norm"], d["mod"], shape.eps, y=y, res_out=ro, ws=ws)
        e[1].record(stream)
        mot.mot_routed_qkv_norm_rope(y, d["w_qkv"], d["q_norm"], d["k_norm"], d["pos"], cs, HQ, HKV, D, shape.eps,
                                     ws, out=out)
        e[2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if sampler:
        sampler.mark("end")
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    flags = mot.mot_device_status(ws)
    if flags != 0:
        raise RuntimeError(f"device error flags {flags:#x} in the timed region")

    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    norm_ms = [e[0].elapsed_time(e[1]) for e in ev]
    qkv_ms = [e[1].elapsed_time(e[2]) for e in ev]
    mean = statistics.fmean
    local = torch.tensor([mean(step_ms), mean(qkv_ms), mean(norm_ms)], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(local, op=dist.ReduceOp.MAX)
    step_s, qkv_s, norm_s = (v / 1e3 for v in local.tolist())

    # end to end through the public API: host (pinned) inputs in, results back to the host
    e2e = run_e2e(args, shape, d, cs, ws, stream, dev, world)

    if rank != 0:
        return None
    pk = peaks()
    qkv_tflops = QKV_FLOPS / qkv_s / 1e12
    norm_gbs = NORM_BYTES / norm_s / 1e9
    h = src_hash("mot_gemm.cu")
    traffic = NCU_TRAFFIC.get(h)
    res = {
        "metric": METRIC,
        "value": round(world * QKV_FLOPS / step_s / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the BAGEL layer shape)",
        "config": {"workload": WORKLOAD, "T": T, "hidden": H, "q_heads": HQ, "kv_heads": HKV, "head_dim": D,
                   "und_rows": 3072, "gen_rows": 1024,
                   "step": "fused add-RMSNorm (its launch also builds the routing plan) + routed QKV/QK-norm/RoPE",
                   "l2": "flushed before every timed step (write then read of 2x L2, outside the timed events)",
                   "parallelism": f"replicas x{world} (one pack per GPU, no collective)"},
        "roofline": {"kernel": "routed_gemm_kernel<QKV128>", "bound": "tensor", "achieved": round(qkv_tflops, 2),
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(qkv_tflops / pk["bf16_tflops"], 4),
                     "peak_source": pk["source"] + " (bf16 dense, burst)", "traffic": traffic,
                     "algorithmic": "2*T*H*N flops per launch = 1.3529e11"},
        "roofline_norm": {"kernel": "add_rmsnorm_kernel (+ routing-plan CTA)", "bound": "hbm",
                          "achieved": round(norm_gbs, 1),
                          "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(norm_gbs / pk["hbm_gbs"], 4),
                          "peak_source": pk["source"], "algorithmic": "8*T*H + 4*H + T bytes per launch"},
        "kernels_us": {"add_rmsnorm_and_route_plan": round(norm_s * 1e6, 2), "qkv_norm_rope": round(qkv_s * 1e6, 2)},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "wall_s_timed_loop": round(wall, 3),
        "kernel_src": h,
    }
    if args.cpu_baseline and world == 1:
        res["cpu_baseline"] = cpu_baseline(rows=args.cpu_rows)
    return res


def run_e2e(args, shape, d, cs, ws, stream, dev, world):
    import torch
    import torch.distributed as dist

    import mixture_transformers_token_gb300 as mot

    x_h = d["x"].cpu().pin_memory()
    r_h = d["res"].cpu().pin_memory()
    out_h = torch.empty((T, N_QKV), dtype=torch.bfloat16).pin_memory()
    ro_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(d["x"])
    r_d = torch.empty_like(d["res"])
    y = torch.empty_like(d["x"])
    ro = torch.empty_like(d["x"])
    out = torch.empty((T, N_QKV), dtype=torch.bfloat16, device=dev)
    steps = max(3, min(args.steps, 200))

    def one():
        x_d.copy_(x_h, non_blocking=True)
        r_d.copy_(r_h, non_blocking=True)
        mot.mot_fused_add_rmsnorm(x_d, r_d, d["w_norm"], d["mod"], shape.eps, y=y, res_out=ro, ws=ws)
        mot.mot_routed_qkv_norm_rope(y, d["w_qkv"], d["q_norm"], d["k_norm"], d["pos"], cs, HQ, HKV, D, shape.eps,
                                     ws, out=out)
        out_h.copy_(out, non_blocking=True)
        ro_h.copy_(ro, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    s = a.elapsed_time(b) / 1e3 / steps
    t = torch.tensor([s], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    s = float(t.item())
    return {"value": round(world * QKV_FLOPS / s / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(s * 1e3, 4),
            "steps": steps, "h2d_bytes_per_step": 2 * T * H * 2, "d2h_bytes_per_step": T * N_QKV * 2 + T * H * 2}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_layer_rows(rows, seed=1):
    """Inputs of the bench workload restricted to `rows`, as the oracle's float64 arrays."""
    import numpy as np

    from mixture_transformers_token_gb300 import workloads as W

    shape, inp = W.bagel_layer(seed=seed, T=T)

    def f(t):
        return t.float().numpy().astype(np.float64)

    return shape, {"x": f(inp["x"])[rows], "res": f(inp["res"])[rows], "w_norm": f(inp["w_norm"]),
                   "w_qkv": f(inp["w_qkv"]), "q_norm": f(inp["q_norm"]), "k_norm": f(inp["k_norm"]),
                   "pos": inp["pos"].numpy()[rows], "mod": inp["mod"].numpy()[rows]}


def oracle_step(shape, a):
    from oracle import mot_oracle as O

    return O.g_layer(a["x"], a["res"], a["w_norm"], a["w_qkv"], None, a["q_norm"], a["k_norm"], a["pos"], a["mod"],
                     HQ, HKV, D, shape.eps, shape.theta)


def cpu_baseline_child(rows_n: int) -> None:
    import numpy as np

    rows = np.sort(np.random.default_rng(5).choice(T, rows_n, replace=False))
    shape, a = oracle_layer_rows(rows)
    t0 = time.perf_counter()
    oracle_step(shape, a)
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "rows": rows_n}))


def cpu_baseline(rows: int) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", str(rows)], env=env,
                       capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"value": None, "error": r.stderr[-400:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    flops = QKV_FLOPS * d["rows"] / T
    return {"value": round(flops / d["seconds"] / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{d['rows']} of {T} rows of the same pack (fp64 golden: add-RMSNorm + routed QKV + QK-norm "
                      f"+ RoPE), {d['seconds']:.1f} s single-threaded; rows are independent, so the rate scales"}


def run_reference(args, rank, world) -> dict | None:
    if rank != 0:
        return None
    import numpy as np

    rows_per_step = int(max(1, min(64, 4096 // max(1, args.steps + args.warmup))))
    rng = np.random.default_rng(7)
    shape, full = oracle_layer_rows(np.arange(T))
    times = []
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(T, rows_per_step, replace=False))
        a = dict(full, x=full["x"][rows], res=full["res"][rows], pos=full["pos"][rows], mod=full["mod"][rows])
        t0 = time.perf_counter()
        oracle_step(shape, a)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec_per_row = sum(times) / (len(times) * rows_per_step)
    value = QKV_FLOPS / (sec_per_row * T) / 1e12
    threads = os.environ.get("OMP_NUM_THREADS") or os.environ.get("OPENBLAS_NUM_THREADS") or str(os.cpu_count())
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec_per_row * T * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "step": "oracle fp64 golden on a row sample, scaled to the full pack"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": int(threads) if threads.isdigit()
                             else threads, "kind": "oracle",
                             "sample": f"{rows_per_step} random rows of {T} per step, scaled to the pack"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-baseline", dest="cpu_baseline", action="store_true", default=True)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-rows", type=int, default=512)
    ap.add_argument("--cpu-baseline-child", type=int, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_baseline_child is not None:
        cpu_baseline_child(args.cpu_baseline_child)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist

            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        res = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
