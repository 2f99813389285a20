#!/usr/bin/env python
"""Benchmark of the MoT token-routed projection step on GB300.

One step is one pass of the projection path over a packed batch: the fused residual-add
RMSNorm (whose launch also builds the routing plan) and the routed QKV GEMM with its per-head
QK RMSNorm and BF16 RoPE epilogue. The workload is the BAGEL-shaped layer: T = 4096 packed bf16
tokens, hidden 3584, Q 28 x 128, KV 4 x 128 (QKV out 4608), und/gen weight sets W ~ N(0, 0.02),
the first 3072 tokens und then a contiguous 1024-token gen block, positions 0..4095, eps 1e-6,
theta 1e6. Inputs are synthetic and seeded (one pack per rank); L2 is flushed (a write and a
read of twice its size) before every timed step, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). `value` is whole-job TFLOP/s of the routed QKV projection
(2 T H N flops per rank) over the whole step time, max over ranks. The line also carries
secondary measurements of the other rows of the path on their own workloads (the routed
SwiGLU MLP at T = 8192 with scattered gen rows, and the CFG pack at T = 36864 with the routed
O projection), each against its roofline. `--impl reference` times the CPU oracle on the host
cores instead (rank 0 only).
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


def norm_bytes(t: int, h: int) -> int:
    """Algorithmic bytes of the fused add-RMSNorm: read x, res; write y, res_out; weights; modality."""
    return 8 * t * h + 4 * h + t


# DRAM traffic of one QKV kernel launch from an ncu capture of this workload, keyed by the
# hash of the kernel source it was taken on (null once the kernel has changed).
NCU_TRAFFIC = {"9ab96611dfcd50e6": 127521792}


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


def bench_config(world: int) -> dict:
    """The workload both arms measure (the same dict on the reference arm's line)."""
    return {"workload": WORKLOAD, "T": T, "hidden": H, "q_heads": HQ, "kv_heads": HKV, "head_dim": D,
            "und_rows": 3072, "gen_rows": 1024,
            "step": "fused add-RMSNorm (its launch also builds the routing plan) + routed QKV/QK-norm/RoPE",
            "l2": "flushed before every timed step (write then read of 2x L2, outside the timed events)",
            "parallelism": f"replicas x{world} (one pack per GPU, no collective)"}


# ---------------------------------------------------------------------------
# ranks: one pack per GPU, no collective on the data path
# ---------------------------------------------------------------------------

def reduce_max(values, world: int, device=None) -> list:
    """Element-wise maximum over ranks (identity on one rank)."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, work_per_rank: float, seconds: float) -> float:
    """Work of all ranks over the slowest rank's time (weak scaling: per-rank work is fixed)."""
    return world * work_per_rank / seconds


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
# device timing
# ---------------------------------------------------------------------------

class L2Flush:
    """Writes and then reads a buffer of twice the L2 size, so a timed region starts with a cold
    L2 holding only clean lines (a write-only flush would leave dirty lines whose write-back
    lands inside the timed kernels)."""

    def __init__(self, dev):
        import torch

        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.empty(2 * max(l2, 64 << 20) // 4, dtype=torch.int32, device=dev)
        self.i = 0

    def __call__(self):
        self.i += 1
        self.buf.fill_(self.i)
        self.buf.sum()


def time_stages(stages, steps: int, warmup: int, flush, stream) -> dict:
    """Runs the list of (name, fn) as one step `warmup + steps` times with an L2 flush before
    every step; returns the mean device time of each stage and of the step, in seconds, and
    under "dist" their median, 10th and 90th percentiles in microseconds."""
    import torch

    for _ in range(warmup):
        flush()
        for _, fn in stages:
            fn()
    torch.cuda.synchronize()
    if steps == 0:
        return {}
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    samples = {name: [e[j].elapsed_time(e[j + 1]) / 1e3 for e in ev] for j, (name, _) in enumerate(stages)}
    samples["step"] = [e[0].elapsed_time(e[-1]) / 1e3 for e in ev]
    out = {name: statistics.fmean(v) for name, v in samples.items()}
    out["dist"] = {name: percentiles_us(v) for name, v in samples.items()}
    return out


def time_compared(candidates: dict, steps: int, warmup: int, flush, stream) -> dict:
    """Times several candidate stage lists against each other: every iteration runs each
    candidate once, after its own L2 flush, in an order that is reversed on every other
    iteration, so drift and order effects fall on all candidates alike. Returns, per candidate,
    what time_stages returns."""
    import torch

    names = list(candidates)
    for _ in range(warmup):
        for name in names:
            flush()
            for _, fn in candidates[name]:
                fn()
    torch.cuda.synchronize()
    ev = {name: [[torch.cuda.Event(enable_timing=True) for _ in range(len(candidates[name]) + 1)]
                 for _ in range(steps)] for name in names}
    for i in range(steps):
        for name in (names if i % 2 == 0 else names[::-1]):
            flush()
            e = ev[name][i]
            e[0].record(stream)
            for j, (_, fn) in enumerate(candidates[name]):
                fn()
                e[j + 1].record(stream)
    torch.cuda.synchronize()
    out = {}
    for name in names:
        stages = candidates[name]
        samples = {sn: [e[j].elapsed_time(e[j + 1]) / 1e3 for e in ev[name]] for j, (sn, _) in enumerate(stages)}
        samples["step"] = [e[0].elapsed_time(e[-1]) / 1e3 for e in ev[name]]
        r = {sn: statistics.fmean(v) for sn, v in samples.items()}
        r["dist"] = {sn: percentiles_us(v) for sn, v in samples.items()}
        out[name] = r
    return out


def percentiles_us(seconds: list) -> dict:
    v = sorted(seconds)

    def q(f):  # nearest-rank percentile
        return round(v[min(len(v) - 1, max(0, int(round(f * (len(v) - 1)))))] * 1e6, 2)

    return {"median": q(0.5), "p10": q(0.1), "p90": q(0.9)}


def time_warm(fn, iters: int, stream) -> float:
    """Mean device time of `fn` run back to back with no flush (inputs left in L2 by the
    previous call), in seconds."""
    import torch

    for _ in range(3):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / iters


def _cmd(argv: list) -> str | None:
    try:
        r = subprocess.run(argv, capture_output=True, text=True, timeout=20)
        return r.stdout.strip() if r.returncode == 0 else None
    except (OSError, subprocess.SubprocessError):
        return None


def provenance(dev) -> dict:
    """Where the numbers came from: source revision, toolchain, device and the peak figures."""
    import torch

    commit = _cmd(["git", "-C", ROOT, "rev-parse", "HEAD"])
    dirty = None
    if commit is not None:
        st = _cmd(["git", "-C", ROOT, "status", "--porcelain", "--untracked-files=no"])
        dirty = None if st is None else bool(st)
    nvcc = _cmd(["nvcc", "--version"])
    props = torch.cuda.get_device_properties(dev)
    return {
        "git_commit": commit, "git_dirty": dirty,
        "kernel_src": {n: src_hash(n) for n in ("mot_gemm.cu", "mot_route_norm.cu", "mot_misc.cu")},
        "nvcc": nvcc.splitlines()[-1] if nvcc else None,
        "driver": _cmd(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader", "-i",
                        str(dev.index or 0)]),
        "torch": torch.__version__, "torch_cuda": torch.version.cuda,
        "gpu": props.name, "sm_count": props.multi_processor_count, "cc": f"{props.major}.{props.minor}",
        "l2_bytes": props.L2_cache_size, "peaks": peaks(),
    }


def host_cpu() -> dict:
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if model is None:
        out = _cmd(["lscpu"])
        for line in (out or "").splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    return {"model": model, "affinity_cores": len(os.sched_getaffinity(0))}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import build as mot_build
    from mixture_transformers_token_gb300 import workloads as W

    if rank == 0 or world == 1:
        mot_build.build()
    if world > 1:
        dist.barrier()
    mot.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shape, inp = W.bagel_layer(seed=1 + rank, T=T)
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    stream = torch.cuda.current_stream(dev)
    cs = mot.mot_rope_table_fill_host(shape.theta, D, T).to(dev)
    ws = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ro = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, N_QKV), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)

    def norm():  # its launch also writes the routing plan of mod into ws (one extra CTA)
        mot.mot_fused_add_rmsnorm(d["x"], d["res"], d["w_norm"], d["mod"], shape.eps, y=y, res_out=ro, ws=ws)

    def qkv():
        mot.mot_routed_qkv_norm_rope(y, d["w_qkv"], d["q_norm"], d["k_norm"], d["pos"], cs, HQ, HKV, D, shape.eps,
                                     ws, out=out)

    def step():
        norm()
        qkv()

    stages = [("add_rmsnorm_and_route_plan", norm), ("qkv_norm_rope", qkv)]
    time_stages(stages, 0, args.warmup, flush, stream)
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set during warm-up")
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("start")
    # The step is timed with events only around each step: an event recorded between the norm
    # and the QKV kernel ends the QKV's programmatic overlap of the norm's tail (about 3.4 us per
    # step). A second pass of the same K steps, with an event after each kernel, gives the kernel
    # durations that the rooflines use.
    t_wall = time.perf_counter()
    times_step = time_stages([("step", step)], args.steps, 0, flush, stream)
    wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    times = time_stages(stages, args.steps, 0, flush, stream)
    if sampler:
        sampler.mark("end")
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    flags = mot.mot_device_status(ws)
    if flags != 0:
        raise RuntimeError(f"device error flags {flags:#x} in the timed region")
    step_s, qkv_s, norm_s, step_ev_s = reduce_max([times_step["step"], times["qkv_norm_rope"],
                                                   times["add_rmsnorm_and_route_plan"], times["step"]], world, dev)

    warm_qkv = time_warm(qkv, 50, stream)
    e2e = run_e2e(args, shape, d, cs, ws, dev, world)
    secondary = None
    if rank == 0 and args.secondary:
        secondary = {"swiglu_mlp_T8192": run_mlp(dev, flush), "cfg_pack_T36864": run_cfg_pack(dev, flush),
                     "fp32_rope_profile_T4096": run_qkv_fp32_rope(dev, flush),
                     "backward_T4096": run_backward(dev, flush),
                     "joint_attention": run_attention(dev, flush),
                     "flow_step": run_flow(dev, flush)}
    if rank == 0 and secondary is not None and args.cpu_baseline and world == 1:
        secondary["swiglu_mlp_T8192"]["cpu_baseline"] = cpu_baseline_secondary("mlp")
        secondary["cfg_pack_T36864"]["cpu_baseline"] = cpu_baseline_secondary("cfg")
    if world > 1:
        dist.barrier()
    if rank != 0:
        return None

    pk = peaks()
    qkv_tflops = QKV_FLOPS / qkv_s / 1e12
    norm_gbs = norm_bytes(T, H) / norm_s / 1e9
    h = src_hash("mot_gemm.cu")
    res = {
        "metric": METRIC,
        "value": round(whole_job_rate(world, QKV_FLOPS, step_s) / 1e12, 2),
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
        "config": bench_config(world),
        "roofline": {"kernel": "routed_gemm_kernel<QKV128>", "bound": "tensor", "achieved": round(qkv_tflops, 2),
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(qkv_tflops / pk["bf16_tflops"], 4),
                     "peak_source": pk["source"] + " (bf16 dense, burst)", "traffic": NCU_TRAFFIC.get(h),
                     "algorithmic": "2*T*H*N flops per launch = 1.3529e11"},
        "roofline_norm": {"kernel": "add_rmsnorm_kernel (+ routing-plan CTA)", "bound": "hbm",
                          "achieved": round(norm_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                          "frac": round(norm_gbs / pk["hbm_gbs"], 4), "peak_source": pk["source"],
                          "algorithmic": "8*T*H + 4*H + T bytes per launch"},
        "kernels_us": {"add_rmsnorm_and_route_plan": round(norm_s * 1e6, 2), "qkv_norm_rope": round(qkv_s * 1e6, 2)},
        "distribution_us": {"step": times_step["dist"]["step"], **{k: times["dist"][k] for k in (
            "add_rmsnorm_and_route_plan", "qkv_norm_rope")}, "step_with_kernel_events": times["dist"]["step"]},
        "timing": {"step": "events only around each of the K timed steps (value, ms_per_step)",
                   "kernels": "a second pass of the same K steps with an event after each kernel (kernels_us, "
                              "roofline, roofline_norm); those events end the QKV kernel's programmatic overlap "
                              "of the norm", "step_with_kernel_events_ms": round(step_ev_s * 1e3, 4)},
        "l2_warm": {"qkv_norm_rope_us": round(warm_qkv * 1e6, 2),
                    "qkv_tflops": round(QKV_FLOPS / warm_qkv / 1e12, 2),
                    "note": "QKV launches back to back with no flush (L2-warm), rank 0; not the headline"},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "wall_s_timed_loop": round(wall, 3),
        "kernel_src": h,
        "provenance": provenance(dev),
    }
    if secondary is not None:
        res["secondary"] = secondary
    if args.cpu_baseline and world == 1:
        res["cpu_baseline"] = cpu_baseline(rows=args.cpu_rows)
    return res


def run_e2e(args, shape, d, cs, ws, dev, world):
    """The same step through the public API from pinned host buffers: every step copies its
    inputs (x, res) to the device and reads its results (qkv, res_out) back. Copies run on their
    own streams with two device buffer sets, so the copies of neighbouring steps overlap the
    compute; the rate is the steps' total device time over the timed steps."""
    import torch
    import torch.distributed as dist

    import mixture_transformers_token_gb300 as mot

    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    x_h = d["x"].cpu().pin_memory()
    r_h = d["res"].cpu().pin_memory()
    out_h = [torch.empty((T, N_QKV), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ro_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(d["x"]) for _ in range(2)]
    r_d = [torch.empty_like(d["res"]) for _ in range(2)]
    ro_d = [torch.empty_like(d["x"]) for _ in range(2)]
    out_d = [torch.empty((T, N_QKV), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    y = torch.empty_like(d["x"])
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    steps = max(3, min(args.steps, 200))

    def one(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(comp_done[b])            # the slot's inputs are consumed
            x_d[b].copy_(x_h, non_blocking=True)
            r_d[b].copy_(r_h, non_blocking=True)
            in_done[b].record(s_in)
        comp.wait_event(in_done[b])
        if i >= 2:
            comp.wait_event(out_done[b])                 # the slot's outputs are read back
        mot.mot_fused_add_rmsnorm(x_d[b], r_d[b], d["w_norm"], d["mod"], shape.eps, y=y, res_out=ro_d[b], ws=ws,
                                  stream=comp)
        mot.mot_routed_qkv_norm_rope(y, d["w_qkv"], d["q_norm"], d["k_norm"], d["pos"], cs, HQ, HKV, D, shape.eps,
                                     ws, out=out_d[b], stream=comp)
        comp_done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            out_h[b].copy_(out_d[b], non_blocking=True)
            ro_h[b].copy_(ro_d[b], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        one(i)
    s_out.wait_stream(comp)
    b.record(s_out)
    torch.cuda.synchronize()
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set in the end-to-end loop")
    s = reduce_max([a.elapsed_time(b) / 1e3 / steps], world, dev)[0]
    return {"value": round(whole_job_rate(world, QKV_FLOPS, s) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(s * 1e3, 4), "steps": steps, "h2d_bytes_per_step": 2 * T * H * 2,
            "d2h_bytes_per_step": T * N_QKV * 2 + T * H * 2,
            "note": "pinned host inputs copied in and results read back every step; copies overlap neighbouring steps"}


def _tflops(flops, s):
    return round(flops / s / 1e12, 2)


def run_mlp(dev, flush) -> dict:
    """Routed SwiGLU MLP, T = 8192, hidden 3584, intermediate 18944, 2048 gen rows scattered:
    add-RMSNorm (+ plan) -> rows into plan order -> gate/up + SwiGLU (plan order in and out) ->
    down (plan order in, token order out)."""
    import torch

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import workloads as W

    t, h, i = W.MLP_T, W.MLP_H, W.MLP_I
    stream = torch.cuda.current_stream(dev)
    m = W.mlp_device_inputs(dev)
    x, res, w_norm, mod, w_down = m["x"], m["res"], m["w_norm"], m["mod"], m["w_down"]
    w_gu = mot.mot_swiglu_interleave(m.pop("w_gate"), m.pop("w_up"))
    ws = torch.empty(mot.mot_workspace_bytes(t), dtype=torch.uint8, device=dev)
    y, ro, y_plan = (torch.empty((t, h), dtype=torch.bfloat16, device=dev) for _ in range(3))
    hid = torch.empty((t, i), dtype=torch.bfloat16, device=dev)
    out = torch.empty((t, h), dtype=torch.bfloat16, device=dev)
    stages = [
        ("add_rmsnorm_and_route_plan", lambda: mot.mot_fused_add_rmsnorm(x, res, w_norm, mod, 1e-6, y=y, res_out=ro,
                                                                         ws=ws)),
        ("gather_rows", lambda: mot.mot_gather_rows(y, ws, out=y_plan)),
        ("gate_up_swiglu", lambda: mot.mot_routed_gemm(y_plan, w_gu, ws, mot.EPI_SWIGLU | mot.A_PLAN_ORDER
                                                       | mot.OUT_PLAN_ORDER, out=hid)),
        ("down", lambda: mot.mot_routed_gemm(hid, w_down, ws, mot.EPI_CAST | mot.A_PLAN_ORDER, out=out)),
    ]
    r = time_stages(stages, 50, 5, flush, stream)
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set in the MLP workload")
    pk = peaks()
    f_gu, f_dn = 2 * t * h * 2 * i, 2 * t * i * h
    nb = norm_bytes(t, h)
    result = {
        "workload": "T8192_H3584_I18944_gen2048_scattered",
        "add_rmsnorm_us": round(r["add_rmsnorm_and_route_plan"] * 1e6, 2),
        "add_rmsnorm_gbs": round(nb / r["add_rmsnorm_and_route_plan"] / 1e9, 1),
        "add_rmsnorm_frac_hbm": round(nb / r["add_rmsnorm_and_route_plan"] / 1e9 / pk["hbm_gbs"], 4),
        "gather_rows_us": round(r["gather_rows"] * 1e6, 2),
        "gather_rows_gbs": round(2 * t * h * 2 / r["gather_rows"] / 1e9, 1),
        "gate_up_swiglu_us": round(r["gate_up_swiglu"] * 1e6, 2),
        "gate_up_swiglu_tflops": _tflops(f_gu, r["gate_up_swiglu"]),
        "gate_up_swiglu_frac": round(f_gu / r["gate_up_swiglu"] / 1e12 / pk["bf16_tflops"], 4),
        "down_us": round(r["down"] * 1e6, 2),
        "down_tflops": _tflops(f_dn, r["down"]),
        "down_frac": round(f_dn / r["down"] / 1e12 / pk["bf16_tflops"], 4),
        "step_us": round(r["step"] * 1e6, 2),
        "peaks": f"{pk['source']}: bf16 {pk['bf16_tflops']} TFLOP/s (burst), HBM {pk['hbm_gbs']} GB/s",
    }
    del w_gu, w_down, hid
    return result


def run_qkv_fp32_rope(dev, flush) -> dict:
    """The FP32 RoPE profile of the QKV projection on the bench workload (T = 4096): add-RMSNorm
    (+ plan) once, then the routed QKV with QK-norm and RoPE in fp32 (fp32 table, one cast)."""
    import torch

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import workloads as W

    stream = torch.cuda.current_stream(dev)
    shape, inp = W.bagel_layer(seed=1, T=T)
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    cs32 = mot.mot_rope_table_fill_host_fp32(shape.theta, D, T).to(dev)
    ws = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device=dev)
    y, ro = mot.mot_fused_add_rmsnorm(d["x"], d["res"], d["w_norm"], d["mod"], shape.eps, ws=ws)
    out = torch.empty((T, N_QKV), dtype=torch.bfloat16, device=dev)
    stages = [("qkv_fp32_rope", lambda: mot.mot_routed_qkv_norm_rope_fp32(
        y, d["w_qkv"], d["q_norm"], d["k_norm"], d["pos"], cs32, HQ, HKV, D, shape.eps, ws, out=out))]
    r = time_stages(stages, 200, 5, flush, stream)
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set in the FP32 RoPE workload")
    pk = peaks()
    return {"workload": WORKLOAD, "qkv_fp32_rope_us": round(r["qkv_fp32_rope"] * 1e6, 2),
            "qkv_fp32_rope_tflops": _tflops(QKV_FLOPS, r["qkv_fp32_rope"]),
            "qkv_fp32_rope_frac": round(QKV_FLOPS / r["qkv_fp32_rope"] / 1e12 / pk["bf16_tflops"], 4),
            "distribution_us": r["dist"]["qkv_fp32_rope"]}


def run_backward(dev, flush) -> dict:
    """Backward of the bench layer's projection step (T = 4096, hidden 3584, QKV out 4608): the
    QKV GEMM's input gradient through both weight sets, add-RMSNorm backward (dx, rstd and the
    per-row weight partials), the norm-weight fold, and the gen set's weight gradient (1024 rows)
    from token-order dqkv and y; and the same chain in phase A (the gen set trained: the norm's
    weight partials and fold of the gen rows only)."""
    import torch

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import workloads as W

    stream = torch.cuda.current_stream(dev)
    shape, inp = W.bagel_layer(seed=1, T=T)
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    ws = torch.empty(mot.mot_workspace_bytes(T), dtype=torch.uint8, device=dev)
    y, s_res = mot.mot_fused_add_rmsnorm(d["x"], d["res"], d["w_norm"], d["mod"], shape.eps, ws=ws)
    dqkv = W.bf16_normal_device(1, 400, (T, N_QKV), dev)
    dres = W.bf16_normal_device(1, 401, (T, H), dev)
    dy = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    dxn = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    rstd = torch.empty((T,), dtype=torch.float32, device=dev)
    dwn = torch.empty((2, H), dtype=torch.float32, device=dev)
    part = torch.empty((H // 64, T, 64), dtype=torch.float32, device=dev)
    dw_gen = torch.empty((N_QKV, H), dtype=torch.float32, device=dev)
    stages = [
        ("qkv_dx", lambda: mot.mot_routed_gemm_dx(dqkv, d["w_qkv"], ws, out=dy)),
        ("add_rmsnorm_dx", lambda: mot.mot_add_rmsnorm_backward(dy, s_res, d["w_norm"], shape.eps, ws,
                                                                d_res_out=dres, dx=dxn, rstd=rstd,
                                                                dw_partials=part)),
        ("rmsnorm_dweight", lambda: mot.mot_rmsnorm_dweight(part, ws, dw=dwn)),
        ("qkv_dw_gen", lambda: mot.mot_routed_gemm_dw(dqkv, y, ws, expert=1, out=dw_gen)),
    ]
    r = time_stages(stages, 50, 5, flush, stream)
    # phase A of the BAGEL training rules trains the gen set only: the norm backward writes the
    # gen rows' weight partials alone (every row's dx still) and the fold runs over the gen set
    stages_a = [
        stages[0],
        ("add_rmsnorm_dx", lambda: mot.mot_add_rmsnorm_backward(dy, s_res, d["w_norm"], shape.eps, ws,
                                                                d_res_out=dres, dx=dxn, rstd=rstd,
                                                                dw_partials=part, partial_sets=mot.SET_GEN)),
        ("rmsnorm_dweight", lambda: mot.mot_rmsnorm_dweight(part, ws, dw=dwn, sets=mot.SET_GEN)),
        stages[3],
    ]
    ra = time_stages(stages_a, 50, 5, flush, stream)

    def whole():
        for _, fn in stages:
            fn()

    def whole_a():
        for _, fn in stages_a:
            fn()

    # the same chains with events only around them: every kernel after the first is a programmatic
    # dependent of the one before, which the events between stages above rule out
    rw = time_stages([("step", whole)], 50, 5, flush, stream)
    rwa = time_stages([("step", whole_a)], 50, 5, flush, stream)
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set in the backward workload")
    pk = peaks()
    n_gen = int(inp["mod"].sum())
    f_dx, f_dw = 2 * T * N_QKV * H, 2 * n_gen * N_QKV * H
    b_dx = 12 * T * H + 8 * T + 4 * H         # dy, s, d_res_out read; dx, fp32 partials, rstd written; plan; w
    b_dw = 4 * T * H + 8 * H                  # fp32 partials read; dw written
    b_dx_a = 8 * T * H + 4 * n_gen * H + 8 * T + 4 * H   # phase A: the gen rows' partials only
    b_dw_a = 4 * n_gen * H + 4 * H

    def gbs(b, name):
        return round(b / r[name] / 1e9, 1)

    return {
        "workload": WORKLOAD + "_backward",
        "qkv_dx_us": round(r["qkv_dx"] * 1e6, 2), "qkv_dx_tflops": _tflops(f_dx, r["qkv_dx"]),
        "qkv_dx_frac": round(f_dx / r["qkv_dx"] / 1e12 / pk["bf16_tflops"], 4),
        "add_rmsnorm_dx_us": round(r["add_rmsnorm_dx"] * 1e6, 2),
        "add_rmsnorm_dx_gbs": gbs(b_dx, "add_rmsnorm_dx"),
        "add_rmsnorm_dx_frac_hbm": round(b_dx / r["add_rmsnorm_dx"] / 1e9 / pk["hbm_gbs"], 4),
        "rmsnorm_dweight_us": round(r["rmsnorm_dweight"] * 1e6, 2),
        "rmsnorm_dweight_gbs": gbs(b_dw, "rmsnorm_dweight"),
        "rmsnorm_dweight_frac_hbm": round(b_dw / r["rmsnorm_dweight"] / 1e9 / pk["hbm_gbs"], 4),
        "qkv_dw_gen_us": round(r["qkv_dw_gen"] * 1e6, 2), "qkv_dw_gen_tflops": _tflops(f_dw, r["qkv_dw_gen"]),
        "qkv_dw_gen_frac": round(f_dw / r["qkv_dw_gen"] / 1e12 / pk["bf16_tflops"], 4),
        "gen_rows": n_gen, "step_us": round(rw["step"] * 1e6, 2),
        "step_us_with_stage_events": round(r["step"] * 1e6, 2),
        "phase_a": {
            "what": "the gen set trained: norm-weight partials and fold of the gen rows only (dX, dx of every row)",
            "add_rmsnorm_dx_us": round(ra["add_rmsnorm_dx"] * 1e6, 2),
            "add_rmsnorm_dx_frac_hbm": round(b_dx_a / ra["add_rmsnorm_dx"] / 1e9 / pk["hbm_gbs"], 4),
            "rmsnorm_dweight_us": round(ra["rmsnorm_dweight"] * 1e6, 2),
            "rmsnorm_dweight_frac_hbm": round(b_dw_a / ra["rmsnorm_dweight"] / 1e9 / pk["hbm_gbs"], 4),
            "step_us": round(rwa["step"] * 1e6, 2),
            "step_us_with_stage_events": round(ra["step"] * 1e6, 2),
        },
    }


def attention_flops(seqs, Hq: int, D: int) -> int:
    """4 D flops per visible (query, key) pair and query head: Q K^T and P V."""
    pairs = 0
    for q0, k0, nq, nk, nc in seqs:
        c = min(nc, nq)
        # causal rows i < c see nk - nq + i + 1 keys; the others see nk
        pairs += c * (nk - nq) + c * (c + 1) // 2 + (nq - c) * nk
    return 4 * D * Hq * pairs


def run_attention(dev, flush) -> dict:
    """Joint attention on the BAGEL layer's pack (one sequence: 3072 causal prompt rows, then
    1024 latent rows seeing all 4096 keys) and on the CFG pack (12 x (2048 prompt + 1024 latent)
    rows, T = 36864), Q/K/V from the fused QKV layout (28 q heads, 4 kv heads of 128)."""
    import torch

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import workloads as W

    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    res = {}
    for name, t, seqs in (
            ("bagel_layer_T4096", T, [(0, 0, T, T, 3072)]),
            ("cfg_pack_T36864", 36864, [(3072 * i, 3072 * i, 3072, 3072, 2048) for i in range(12)])):
        qkv = W.bf16_normal_device(9, 600, (t, N_QKV), dev)
        s = torch.tensor(seqs, dtype=torch.int32, device=dev)
        ws = torch.zeros(64, dtype=torch.uint8, device=dev)
        out = torch.empty((t, HQ * D), dtype=torch.bfloat16, device=dev)
        r = time_stages([("attention", lambda: mot.mot_joint_attention(qkv, s, HQ, HKV, D, ws, out=out))], 20, 3,
                        flush, stream)
        if mot.mot_device_status(ws) != 0:
            raise RuntimeError("device error flags set in the attention workload")
        f = attention_flops(seqs, HQ, D)
        res[name] = {"attention_us": round(r["attention"] * 1e6, 2), "tflops": _tflops(f, r["attention"]),
                     "frac": round(f / r["attention"] / 1e12 / pk["bf16_tflops"], 4), "flops": f,
                     "distribution_us": r["dist"]["attention"]}
        del qkv, out
    return res


def run_flow(dev, flush) -> dict:
    """One flow-sampler step of 16 requests of a 1024 x 1024 latent (64 x 64 tokens of 64
    values, N = 262144 each): the per-sample transition noise, then three-branch renormalised
    CFG of bf16 velocities and the SDE step (x and the noise in; x_next and logp out) in one
    call, every request at a different step of the 50-step schedule with shift 3. The same
    step as two calls (CFG into an fp32 velocity, then the SDE step) is timed in the same loop,
    the two orders alternating."""
    import numpy as np
    import torch

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import workloads as W

    stream = torch.cuda.current_stream(dev)
    n_req, n = W.FLOW_REQUESTS, W.FLOW_N_1024
    br = {k: W.bf16_normal_device(11, 800 + i, (n_req, n), dev) for i, k in enumerate(("c", "tu", "iu"))}
    x = W.bf16_normal_device(11, 810, (n_req, n), dev).float()
    z = torch.empty((n_req, n), dtype=torch.float32, device=dev)
    seeds = torch.arange(1000, 1000 + n_req, dtype=torch.int64, device=dev)
    sched = mot.mot_flow_schedule_host(W.FLOW_STEPS, W.FLOW_SHIFT).numpy()
    p = W.FLOW_POLICY
    steps = [3 * i for i in range(n_req)]
    policy = torch.tensor([(float(sched[i]), p["s_text"], p["s_img"], p["t_lo"], p["t_hi"], p["renorm_min"])
                           for i in steps], dtype=torch.float32, device=dev)
    times = torch.tensor(np.array([(sched[i], sched[i + 1]) for i in steps], dtype=np.float32), device=dev)
    ws = torch.zeros(mot.mot_flow_workspace_bytes(n_req, n), dtype=torch.uint8, device=dev)
    v = torch.empty((n_req, n), dtype=torch.float32, device=dev)
    x_next = torch.empty_like(v)
    logp = torch.empty((n_req,), dtype=torch.float32, device=dev)
    stages = [
        ("flow_noise", lambda: mot.mot_flow_noise(seeds, 7, n, z=z)),
        ("cfg_sde_step", lambda: mot.mot_flow_cfg_sde_step(br["c"], br["tu"], br["iu"], policy, x, z, times, ws=ws,
                                                           x_next=x_next, logp=logp)),
    ]
    chain = [
        ("cfg_combine_renorm", lambda: mot.mot_cfg_combine_renorm(br["c"], br["tu"], br["iu"], policy, ws=ws, out=v)),
        ("flow_sde_step", lambda: mot.mot_flow_sde_step(x, v, z, times, ws=ws, x_next=x_next, logp=logp)),
    ]
    # the one-call step and the two calls, in the same loop with the order reversed every step
    both = time_compared({"one_call": stages, "two_calls": chain}, 100, 5, flush, stream)
    r, rc = both["one_call"], both["two_calls"]
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set in the flow workload")
    pk = peaks()
    e = n_req * n
    b_fused = 18 * e + 36 * n_req         # three bf16 branches, x and z read, x_next written; policy, times, logp
    b_cfg = 10 * e + 24 * n_req           # three bf16 branches read, fp32 out written, policy
    b_sde = 16 * e + 12 * n_req           # x, v, z read, x_next written, times, logp
    return {
        "workload": f"flow_step_{n_req}x{n}",
        "flow_noise_us": round(r["flow_noise"] * 1e6, 2),
        "flow_noise_gdev_per_s": round(e / r["flow_noise"] / 1e9, 1),
        "cfg_sde_step_us": round(r["cfg_sde_step"] * 1e6, 2),
        "cfg_sde_step_gbs": round(b_fused / r["cfg_sde_step"] / 1e9, 1),
        "cfg_sde_step_frac_hbm": round(b_fused / r["cfg_sde_step"] / 1e9 / pk["hbm_gbs"], 4),
        "two_calls": {
            "cfg_combine_renorm_us": round(rc["cfg_combine_renorm"] * 1e6, 2),
            "cfg_combine_renorm_frac_hbm": round(b_cfg / rc["cfg_combine_renorm"] / 1e9 / pk["hbm_gbs"], 4),
            "flow_sde_step_us": round(rc["flow_sde_step"] * 1e6, 2),
            "flow_sde_step_frac_hbm": round(b_sde / rc["flow_sde_step"] / 1e9 / pk["hbm_gbs"], 4),
            "sum_us": round((rc["cfg_combine_renorm"] + rc["flow_sde_step"]) * 1e6, 2)},
        "step_us": round(r["step"] * 1e6, 2), "elements": e,
        "bytes": {"cfg_sde_step": b_fused, "cfg": b_cfg, "sde": b_sde},
        "distribution_us": {k: r["dist"][k] for k in ("flow_noise", "cfg_sde_step")},
    }


def run_cfg_pack(dev, flush) -> dict:
    """CFG pack: 12 sequences of 2048 und + 1024 gen rows (T = 36864), positions restarting per
    sequence: add-RMSNorm (+ plan), routed QKV + QK-norm + RoPE, routed O projection 3584 -> 3584
    (its input stands in for the attention output)."""
    import torch

    import mixture_transformers_token_gb300 as mot
    from mixture_transformers_token_gb300 import workloads as W

    s = W.CFG_PACK
    t, h = s.T, s.H
    stream = torch.cuda.current_stream(dev)
    c = W.cfg_pack_device_inputs(dev)
    mod, pos, x, res, attn = c["mod"], c["pos"], c["x"], c["res"], c["attn"]
    w_norm, w_qkv, qn, kn, w_o = c["w_norm"], c["w_qkv"], c["q_norm"], c["k_norm"], c["w_o"]
    cs = mot.mot_rope_table_fill_host(s.theta, s.D, 3072).to(dev)
    ws = torch.empty(mot.mot_workspace_bytes(t), dtype=torch.uint8, device=dev)
    y, ro, o = (torch.empty((t, h), dtype=torch.bfloat16, device=dev) for _ in range(3))
    qkv = torch.empty((t, s.n_qkv), dtype=torch.bfloat16, device=dev)
    stages = [
        ("add_rmsnorm_and_route_plan", lambda: mot.mot_fused_add_rmsnorm(x, res, w_norm, mod, s.eps, y=y, res_out=ro,
                                                                         ws=ws)),
        ("qkv_norm_rope", lambda: mot.mot_routed_qkv_norm_rope(y, w_qkv, qn, kn, pos, cs, s.Hq, s.Hkv, s.D, s.eps, ws,
                                                               out=qkv)),
        ("o_proj", lambda: mot.mot_routed_gemm(attn, w_o, ws, mot.EPI_CAST, out=o)),
    ]
    r = time_stages(stages, 50, 5, flush, stream)
    if mot.mot_device_status(ws) != 0:
        raise RuntimeError("device error flags set in the CFG-pack workload")
    pk = peaks()
    f_qkv, f_o = 2 * t * h * s.n_qkv, 2 * t * h * h
    nb = norm_bytes(t, h)
    return {
        "workload": "T36864_12x(2048und+1024gen)_H3584_q28x128_kv4x128",
        "add_rmsnorm_us": round(r["add_rmsnorm_and_route_plan"] * 1e6, 2),
        "add_rmsnorm_gbs": round(nb / r["add_rmsnorm_and_route_plan"] / 1e9, 1),
        "add_rmsnorm_frac_hbm": round(nb / r["add_rmsnorm_and_route_plan"] / 1e9 / pk["hbm_gbs"], 4),
        "qkv_us": round(r["qkv_norm_rope"] * 1e6, 2),
        "qkv_tflops": _tflops(f_qkv, r["qkv_norm_rope"]),
        "qkv_frac": round(f_qkv / r["qkv_norm_rope"] / 1e12 / pk["bf16_tflops"], 4),
        "o_proj_us": round(r["o_proj"] * 1e6, 2),
        "o_proj_tflops": _tflops(f_o, r["o_proj"]),
        "o_proj_frac": round(f_o / r["o_proj"] / 1e12 / pk["bf16_tflops"], 4),
        "step_us": round(r["step"] * 1e6, 2),
    }


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

SINGLE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                     "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1"}


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


def _host_sample_inputs(kind: str, rows_n: int):
    """Host-drawn inputs of a secondary workload restricted to a uniform sample of rows (the
    same shapes and distributions as the device-drawn ones; the rows are independent, so a
    sample's cost scales to the whole pack). Returns (arrays, flops of the sample)."""
    import numpy as np
    import torch

    from mixture_transformers_token_gb300 import workloads as W

    def f(t):
        return t.float().numpy().astype(np.float64)

    if kind == "mlp":
        t, h, i = W.MLP_T, W.MLP_H, W.MLP_I
        rows = np.sort(np.random.default_rng(5).choice(t, rows_n, replace=False))
        m = W.mlp_inputs(t, h, i, 2048, seed=3)
        a = {"x": f(m["x"])[rows], "res": f(m["res"])[rows], "w_norm": f(m["w_norm"]), "w_gate": f(m["w_gate"]),
             "w_up": f(m["w_up"]), "w_down": f(m["w_down"]), "mod": m["mod"].numpy()[rows]}
        return a, rows_n * (2 * h * 2 * i + 2 * i * h)
    s = W.CFG_PACK
    mod, pos = W.cfg_pack_layout()
    rows = np.sort(np.random.default_rng(5).choice(s.T, rows_n, replace=False))
    inp = W.qkv_layer_inputs(W.QKVShape(T=rows_n, H=s.H, Hq=s.Hq, Hkv=s.Hkv, D=s.D), mod[rows], pos[rows], seed=5)
    a = {k: f(v) for k, v in inp.items() if isinstance(v, torch.Tensor) and k not in ("mod", "pos")}
    a["mod"], a["pos"] = mod.numpy()[rows], pos.numpy()[rows]
    a["attn"] = f(W.bf16_normal(W.rng_for(5, 99), (rows_n, s.H)))
    a["w_o"] = f(W.bf16_normal(W.rng_for(5, 98), (2, s.H, s.H), std=0.02))
    return a, rows_n * (2 * s.H * s.n_qkv + 2 * s.H * s.H)


def _oracle_secondary(kind: str, a) -> None:
    from oracle import mot_oracle as O

    from mixture_transformers_token_gb300 import workloads as W

    if kind == "mlp":
        n = O.g_fused_add_rmsnorm(a["x"], a["res"], a["w_norm"], a["mod"], 1e-6)
        g = O.g_routed_swiglu(n["y"], a["w_gate"], a["w_up"], a["mod"])
        O.g_routed_gemm_cast(g["h"], a["w_down"], a["mod"])
        return
    s = W.CFG_PACK
    O.g_layer(a["x"], a["res"], a["w_norm"], a["w_qkv"], None, a["q_norm"], a["k_norm"], a["pos"], a["mod"], s.Hq,
              s.Hkv, s.D, s.eps, s.theta)
    O.g_routed_gemm_cast(a["attn"], a["w_o"], a["mod"])


def cpu_baseline_child(kind: str, rows_n: int) -> None:
    import numpy as np

    if kind == "layer":
        rows = np.sort(np.random.default_rng(5).choice(T, rows_n, replace=False))
        shape, a = oracle_layer_rows(rows)
        t0 = time.perf_counter()
        oracle_step(shape, a)
        dt = time.perf_counter() - t0
        flops = QKV_FLOPS * rows_n / T
    else:
        a, flops = _host_sample_inputs(kind, rows_n)
        t0 = time.perf_counter()
        _oracle_secondary(kind, a)
        dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "rows": rows_n, "flops": flops}))


def _run_child(argv: list, timeout: int = 900) -> dict:
    env = dict(os.environ, **SINGLE_THREAD_ENV)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), *argv], env=env, capture_output=True, text=True,
                       timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-400:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(rows: int) -> dict:
    try:
        d = _run_child(["--cpu-baseline-child", "layer", str(rows)])
    except (RuntimeError, subprocess.SubprocessError) as e:
        return {"value": None, "error": str(e)[-400:]}
    return {"value": round(d["flops"] / d["seconds"] / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"{d['rows']} of {T} rows of the same pack (fp64 golden: add-RMSNorm + routed QKV + QK-norm "
                      f"+ RoPE), {d['seconds']:.1f} s single-threaded; rows are independent, so the rate scales"}


def cpu_baseline_secondary(kind: str, rows: int = 256) -> dict:
    """The fp64 golden of a secondary workload, single-threaded, on a uniform sample of `rows`
    rows, as a rate (TFLOP/s of the workload's GEMMs): the rate of the whole pack extrapolated
    from the sample."""
    try:
        d = _run_child(["--cpu-baseline-child", kind, str(rows)])
    except (RuntimeError, subprocess.SubprocessError) as e:
        return {"value": None, "error": str(e)[-400:]}
    what = {"mlp": "add-RMSNorm + routed gate/up + SwiGLU + routed down, T=8192",
            "cfg": "add-RMSNorm + routed QKV + QK-norm + RoPE + routed O, T=36864"}[kind]
    return {"value": round(d["flops"] / d["seconds"] / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "extrapolated": True,
            "sample": f"{d['rows']} uniformly sampled rows of the pack (fp64 golden: {what}; host-drawn inputs of the "
                      f"same shapes), {d['seconds']:.1f} s single-threaded; scaled to the pack by rows"}


def reference_child(steps: int, warmup: int, rows_per_step: int) -> None:
    """The reference arm's timed loop, run in a child process with the thread count fixed by
    its environment: every step evaluates the fp64 golden on its own random sample of rows."""
    import numpy as np

    rng = np.random.default_rng(7)
    shape, full = oracle_layer_rows(np.arange(T))
    times = []
    for i in range(warmup + steps):
        rows = np.sort(rng.choice(T, rows_per_step, replace=False))
        a = dict(full, x=full["x"][rows], res=full["res"][rows], pos=full["pos"][rows], mod=full["mod"][rows])
        t0 = time.perf_counter()
        oracle_step(shape, a)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    print(json.dumps({"seconds": times}))


def run_reference(args, rank, world) -> dict | None:
    if rank != 0:
        return None
    rows_per_step = 64
    d = _run_child(["--reference-child", str(args.steps), str(args.warmup), str(rows_per_step)],
                   timeout=max(900, 20 * (args.steps + args.warmup)))
    sec = statistics.fmean(d["seconds"])
    flops = QKV_FLOPS * rows_per_step / T
    value = flops / sec / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights of the BAGEL layer shape)",
            "config": bench_config(world),
            "arm": "the CPU oracle (fp64 golden: add-RMSNorm + routed QKV + QK-norm + RoPE) on the host cores, "
                   f"{rows_per_step} random rows of the pack per step; a step's time is the oracle's own time on "
                   "those rows and the rate is their flops over it",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "host": host_cpu(), "threads_env": SINGLE_THREAD_ENV,
                             "sample": f"{rows_per_step} random rows of {T} per step, single-threaded"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-baseline", dest="cpu_baseline", action="store_true", default=True)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--secondary", dest="secondary", action="store_true", default=True)
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    ap.add_argument("--profile", choices=["mlp", "cfg", "qkv_fp32", "backward", "attention", "flow"], default=None,
                    help="run only one secondary workload (mlp, cfg, backward: 5 warm-up + 50 timed steps; "
                         "qkv_fp32: 5 + 200) and print its figures; a short command for profiler captures")
    ap.add_argument("--cpu-baseline-child", nargs=2, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--reference-child", nargs=3, type=int, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_baseline_child is not None:
        cpu_baseline_child(args.cpu_baseline_child[0], int(args.cpu_baseline_child[1]))
        return
    if args.reference_child is not None:
        reference_child(*args.reference_child)
        return
    if args.profile is not None:
        import torch

        import mixture_transformers_token_gb300 as mot
        from mixture_transformers_token_gb300 import build as mot_build

        mot_build.build()
        mot.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        fn = {"mlp": run_mlp, "cfg": run_cfg_pack, "qkv_fp32": run_qkv_fp32_rope, "backward": run_backward,
              "attention": run_attention, "flow": run_flow}[args.profile]
        print(json.dumps({args.profile: fn(dev, L2Flush(dev))}), flush=True)
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
