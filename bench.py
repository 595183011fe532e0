"""Benchmark of the routed-expert MoE forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload decode|prefill|tiny]

One step = one pass of the whole routed forward (gate + top-k, dispatch
tables, row gather, grouped gate/up GEMM with SiLU, grouped down GEMM,
moe_reduce_fused) over one batch of synthetic tokens resident in HBM, through
the library's C-ABI.  L2 is flushed (a 256 MB write) before every timed step,
outside the timed events.  Each step's device time is taken with CUDA events
on the launching stream; events between the entry points give each kernel's
own duration inside the same timed region.

Prints ONE JSON line (rank 0).  ``value`` = tokens processed by all ranks /
max-over-ranks time.  ``e2e`` = the same metric through ``moe_forward`` with
host (pinned) input and output buffers, the copies inside the timed region.
``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_routed_gate_gb300 import _build, roofline, workloads  # noqa: E402

METRIC = "routed-MoE tokens/s and TFLOP/s (% roofline); reduce_fused GB/s vs HBM peak"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS_PER_STEP = 9  # gate logits, top-k, hist, scan, scatter, gather, gate/up, down, reduce
STAGES = ["gate_topk", "dispatch", "gather", "gate_up_silu", "down", "reduce"]


def describe(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T} (batch {cfg.batch} x seq {cfg.seq}), d_hidden {cfg.d_hidden}, "
            f"d_expert {cfg.d_expert}, {cfg.n_experts} routed experts, top-{cfg.top_k}, {cfg.dtype}"
            + (", Zipf(1.1) rank-order gate bias" if cfg.zipf_bias else ""))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- native arm

class NativeStep:
    """Pre-marshalled C-ABI calls of one forward step (no per-call Python checks)."""

    def __init__(self, cfg, d, dev, x_pool):
        from mixture_experts_routed_gate_gb300 import binding
        self.b = binding
        L = binding.lib()
        self.L = L
        self.cfg = cfg
        T, d_h, d_e, E, k = cfg.T, cfg.d_hidden, cfg.d_expert, cfg.n_experts, cfg.top_k
        self.T, self.k, self.E = T, k, E
        dt = d["x"].dtype
        self.code = {torch.float16: 0, torch.bfloat16: 1}[dt]
        self.ws = torch.empty(binding.forward_workspace_bytes(T, d_h, d_e, E, k, dt),
                              dtype=torch.uint8, device=dev)
        self.v = binding.forward_workspace_views(self.ws, T, d_h, d_e, E, k, dt)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty((T, d_h), dtype=dt, device=dev)
        self.d = d
        self.x_pool = x_pool
        self.mb = binding.num_m_blocks(T, k, E)
        off = lambda i: int(L.moe_forward_workspace_offset(T, d_h, d_e, E, k, self.code, i))
        self.scratch_ptr = self.ws.data_ptr() + off(10)
        self.scratch_bytes = int(L.moe_build_dispatch_workspace_bytes(T, k, E))
        self.stream = torch.cuda.current_stream(dev)
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)
        self.dev = dev

    def p(self, t):
        return ctypes.c_void_p(t.data_ptr()) if t is not None else None

    def calls(self, x):
        """The six entry points of one forward, in order."""
        cfg, v, d, L, p = self.cfg, self.v, self.d, self.L, self.p
        T, k, E, d_h, d_e = self.T, self.k, self.E, cfg.d_hidden, cfg.d_expert
        Tk = T * k
        sp = self.sp
        tables = (p(v["group_sizes"]), p(v["group_offsets"]), p(v["group_padded_offsets"]),
                  p(v["group_idx_for_bx"]))
        return [
            lambda: L.moe_gate_topk(p(x), p(d["wg"]), p(d["bias"]), T, d_h, E, k, self.code,
                                    p(v["topk_idx"]), p(v["topk_w"]), p(v["logits"]),
                                    T * E * 4, sp),
            lambda: L.moe_build_dispatch(p(v["topk_idx"]), p(v["topk_w"]), T, k, E, 128, *tables,
                                         p(v["sorted_token_idx"]), p(v["sorted_row_weight"]),
                                         p(v["token_topk_to_pos"]),
                                         ctypes.c_void_p(self.scratch_ptr), self.scratch_bytes, sp),
            lambda: L.moe_gather_rows(p(x), p(v["sorted_token_idx"]), Tk, T, d_h, self.code,
                                      p(v["a"]), sp),
            lambda: L.moe_grouped_gate_up_silu(p(v["a"]), p(d["w_gate"]), p(d["w_up"]), *tables,
                                               self.mb, Tk, d_h, d_e, E, self.code, p(v["h"]),
                                               p(self.err), sp),
            lambda: L.moe_grouped_down(p(v["h"]), p(d["w_down"]), *tables, self.mb, None, Tk, d_h,
                                       d_e, E, self.code, p(v["y"]), p(self.err), sp),
            lambda: L.moe_reduce_fused(p(v["y"]), Tk, p(v["token_topk_to_pos"]), p(v["topk_w"]), T,
                                       k, d_h, self.code, self.code, p(self.out), p(self.err), sp),
        ]


def run_native(args, cfg, rank, world, dev):
    from mixture_experts_routed_gate_gb300 import binding
    _build.build()
    binding.lib()
    torch.cuda.set_device(dev)
    d = workloads.make_moe_inputs(cfg, device=dev, seed=cfg.seed)
    n_pool = 4
    x_pool = [d["x"]] + [workloads.make_tokens(cfg, cfg.T, device=dev, seed=i) for i in range(1, n_pool)]
    step = NativeStep(cfg, d, dev, x_pool)
    call_lists = [step.calls(x) for x in x_pool]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = step.stream

    def one_step(i, evs=None):
        calls = call_lists[i % n_pool]
        if evs is not None:
            evs[0].record(stream)
        for j, c in enumerate(calls):
            st = c()
            if st != 0:
                raise RuntimeError(f"{STAGES[j]}: {binding.lib().moe_status_string(st).decode()}")
            if evs is not None:
                evs[j + 1].record(stream)

    for i in range(args.warmup):
        flush.zero_()
        one_step(i)
    torch.cuda.synchronize()
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(step.err.item())} after warm-up")

    # routing statistics of each pooled batch (for the algorithmic byte counts)
    act_experts, sizes_pool = [], []
    for i in range(n_pool):
        one_step(i)
        torch.cuda.synchronize()
        sz = step.v["group_sizes"].cpu().numpy().copy()
        sizes_pool.append(sz)
        act_experts.append(int((sz > 0).sum()))

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)]
              for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.15)
    for i in range(args.steps):
        flush.zero_()
        one_step(i, events[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    per_stage = np.array([[events[i][j].elapsed_time(events[i][j + 1]) for j in range(len(STAGES))]
                          for i in range(args.steps)])  # ms
    step_ms = per_stage.sum(axis=1)
    total_ms = float(step_ms.sum())
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(step.err.item())} in the timed region")

    e2e = measure_e2e(args, cfg, d, dev, flush, world)
    aux = measure_reduce_aux(dev, flush) if rank == 0 else None
    return dict(per_stage=per_stage, total_ms=total_ms, act_experts=act_experts,
                sizes_pool=sizes_pool, clocks=clocks, e2e=e2e, aux=aux)


def measure_e2e(args, cfg, d, dev, flush, world):
    """moe_forward through the public binding with pinned host buffers: H2D of
    the step's tokens, the forward, D2H of the output, all inside the events."""
    from mixture_experts_routed_gate_gb300 import binding
    T, d_h = cfg.T, cfg.d_hidden
    dt = d["x"].dtype
    n_pool = 4
    host_x = [workloads.make_tokens(cfg, T, device="cpu", seed=100 + i).pin_memory() for i in range(n_pool)]
    host_out = torch.empty((T, d_h), dtype=dt).pin_memory()
    x_dev = torch.empty((T, d_h), dtype=dt, device=dev)
    ws = torch.empty(binding.forward_workspace_bytes(T, d_h, cfg.d_expert, cfg.n_experts, cfg.top_k, dt),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((T, d_h), dtype=dt, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        x_dev.copy_(host_x[i % n_pool], non_blocking=True)
        binding.moe_forward(x_dev, d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k,
                            ws=ws, out=out, err=err)
        host_out.copy_(out, non_blocking=True)

    for i in range(max(args.warmup, 3)):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    total_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())} in the e2e region")
    es = x_dev.element_size()
    return dict(total_ms=total_ms, h2d=T * d_h * es, d2h=T * d_h * es)


def measure_reduce_aux(dev, flush, reps: int = 20):
    """moe_reduce_fused alone on the bf16 T x 8 x 7168 workloads (GB/s)."""
    from mixture_experts_routed_gate_gb300 import binding
    res = {}
    for name in ("reduce-512", "reduce-4096"):
        c = workloads.REDUCE_CONFIGS[name]
        r = workloads.make_reduce_inputs(c.T, c.K, c.H, c.dtype, c.seed, device=dev)
        out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            binding.moe_reduce_fused(r["x"], r["pos"], r["w"], out=out)
        ts = []
        for _ in range(reps):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            binding.moe_reduce_fused(r["x"], r["pos"], r["w"], out=out)
            e.record()
            e.synchronize()
            ts.append(s.elapsed_time(e))
        n_valid = int((r["pos"] >= 0).sum().item())
        nbytes = roofline.reduce_bytes(n_valid, c.T, c.K, c.H, 2, 2)
        ms = statistics.median(ts)
        res[name] = {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "bytes": nbytes, "bytes_pages_formula": roofline.reduce_bytes_pages(c.T, c.K, c.H, 2)}
    return res


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample(cfg, budget_s: float, min_runs: int = 1):
    """The oracle's forward on the host cores: whole steps on the small
    workloads, a few tokens of the dense per-token path on prefill."""
    from oracle import oracle
    oracle.build()
    d = workloads.make_moe_inputs(cfg, device="cpu") if cfg.name != "prefill" else None
    threads = oracle.threads(0)
    if cfg.name == "prefill":
        # routing of a 4096-token batch would need the full 22.5 GB of weights on
        # the host: time the dense per-token path over 8 experts instead
        return oracle_prefill_sample(cfg, budget_s), threads
    nb = {n: (workloads.to_numpy_bits(v) if v is not None else None) for n, v in d.items()}
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                           cfg.top_k, cfg.dtype)
        runs += 1
        el = time.perf_counter() - t0
        if runs >= min_runs and el >= budget_s:
            break
    tok_s = cfg.T * runs / el
    return dict(value=tok_s, seconds=el, sample=f"{runs} whole forward pass(es) of the {cfg.name} "
                f"workload ({cfg.T} tokens each)"), threads


def oracle_prefill_sample(cfg, budget_s):
    from oracle import oracle
    small = workloads.MoEConfig("prefill-slice", 1, 8, cfg.d_hidden, cfg.d_expert, 8, cfg.top_k,
                                cfg.dtype, cfg.seed)
    d = workloads.make_moe_inputs(small, device="cpu")
    nb = {n: (workloads.to_numpy_bits(v) if v is not None else None) for n, v in d.items()}
    idx = np.tile(np.arange(cfg.top_k, dtype=np.int32), (small.T, 1))
    w = np.full((small.T, cfg.top_k), 1.0 / cfg.top_k, np.float32)
    toks = np.arange(small.T, dtype=np.int32)
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.moe_tokens_dense(nb["x"], nb["w_gate"], nb["w_up"], nb["w_down"], idx, w, toks, cfg.dtype)
        runs += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return dict(value=small.T * runs / el, seconds=el,
                sample=f"{runs} x {small.T} tokens through the dense per-token expert path "
                       f"(8 experts of the prefill shape each); gate and dispatch not included")


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=list(workloads.MOE_CONFIGS), default="decode")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time")
    args = ap.parse_args()
    cfg = workloads.MOE_CONFIGS[args.workload]
    if args.steps is None:
        args.steps = {"decode": 2000, "tiny": 2000, "prefill": 60}[cfg.name] if args.impl == "native" else 3
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    base = {"metric": METRIC, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype,
            "data": "synthetic: seeded N(0,1) tokens, N(0,1/fan_in) random-init expert and gate weights",
            "config": {"workload": describe(cfg), "T": cfg.T, "d_hidden": cfg.d_hidden,
                       "d_expert": cfg.d_expert, "n_experts": cfg.n_experts, "top_k": cfg.top_k,
                       "l2": "flushed before every timed step (256 MB write)",
                       "parallelism": f"replicas x{args.gpus}"}}

    if args.impl == "reference":
        if rank != 0:
            return
        steps_ms = []
        budget = max(1.0, args.cpu_budget / max(1, args.steps))
        info = None
        for i in range(args.warmup + args.steps):
            res, threads = oracle_sample(cfg, budget if i >= args.warmup else 0.0)
            if i >= args.warmup:
                steps_ms.append(cfg.T / res["value"] * 1e3)
                info = res
        tok_s = cfg.T * len(steps_ms) / (sum(steps_ms) / 1e3)
        line = dict(base, impl="reference", value=tok_s, ms_per_step=statistics.mean(steps_ms),
                    cpu_baseline={"value": tok_s, "unit": "tokens/s", "cores": threads,
                                  "kind": "oracle", "sample": info["sample"]},
                    e2e={"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0})
        print(json.dumps(line))
        return

    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    dev = torch.device("cuda", local)
    res = run_native(args, cfg, rank, world, dev)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    T, k, d_h, d_e, E = cfg.T, cfg.top_k, cfg.d_hidden, cfg.d_expert, cfg.n_experts
    Tk = T * k
    per_stage = res["per_stage"]
    ms_step = res["total_ms"] / args.steps
    tokens_total = T * args.steps * world
    value = tokens_total / (res["total_ms"] / 1e3)
    e_act = float(np.mean(res["act_experts"]))
    es = 2
    flops_step = roofline.moe_forward_flops(T, k, d_h, d_e, E)
    # dominant kernel: the grouped gate/up GEMM
    gu_ms = float(per_stage[:, STAGES.index("gate_up_silu")].mean())
    gu_bytes = roofline.gate_up_bytes(Tk, d_h, d_e, round(e_act), es)
    gu_flops = roofline.gate_up_flops(Tk, d_h, d_e)
    t_bytes = gu_bytes / (peaks["hbm_gbs"] * 1e9)
    t_flops = gu_flops / (peaks["bf16_tflops"] * 1e12)
    if t_bytes >= t_flops:
        achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
        rl = {"kernel": "grouped_gemm_kernel<gate_up>", "bound": "hbm", "achieved": round(achieved, 1),
              "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
              "traffic": None, "peak_source": peak_src + " (hbm_gbs)",
              "algorithmic_bytes_per_launch": gu_bytes, "launch_us": round(gu_ms * 1e3, 2)}
    else:
        achieved = gu_flops / (gu_ms * 1e-3) / 1e12
        rl = {"kernel": "grouped_gemm_kernel<gate_up>", "bound": "tensor", "achieved": round(achieved, 1),
              "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
              "traffic": None, "peak_source": peak_src + " (bf16_tflops)",
              "algorithmic_flops_per_launch": gu_flops, "launch_us": round(gu_ms * 1e3, 2)}
    bytes_min = roofline.moe_forward_bytes_min(T, d_h, d_e, E, round(e_act), es)
    step_roof_ms = max(bytes_min / (peaks["hbm_gbs"] * 1e9), flops_step / (peaks["bf16_tflops"] * 1e12)) * 1e3
    cpu, threads = oracle_sample(cfg, args.cpu_budget)
    e2e = res["e2e"]
    line = dict(base)
    line.update({
        "value": round(value, 1), "ms_per_step": round(ms_step, 5),
        "tflops": round(flops_step * args.steps / (res["total_ms"] / 1e3) / 1e12, 3),
        "step_roofline_frac": round(step_roof_ms / ms_step, 4),
        "kernels_us": {s: round(float(per_stage[:, i].mean()) * 1e3, 2) for i, s in enumerate(STAGES)},
        "active_experts": e_act,
        "roofline": rl,
        "reduce_fused_bf16_x8_7168": res["aux"],
        "cpu_baseline": {"value": round(cpu["value"], 2), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": cpu["sample"]},
        "e2e": {"value": round(T * args.steps * world / (e2e["total_ms"] / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": res["clocks"],
    })
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
