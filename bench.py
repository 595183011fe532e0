"""Benchmark of the routed-expert MoE forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload decode|prefill|tiny]

One step = one pass of the whole routed forward (gate + top-k, dispatch
tables, row gather, grouped gate/up GEMM with SiLU, grouped down GEMM,
moe_reduce_fused) over one batch of synthetic tokens resident in HBM: one
moe_forward call through the library's C-ABI, captured once into a CUDA
graph (one per pooled token batch) and replayed.  Before every timed step L2
is evicted (a 256 MB write, then a 256 MB read of another buffer), outside
the timed events.  A second timed pass replays graphs of the six entry
points with event record nodes between them for each kernel's device time.

The headline workload is prefill (4096 tokens, d_hidden 7168, d_expert 2048,
256 experts, top-8, bf16, Zipf gate bias), the largest one-GPU workload; the
decode workload (64 tokens) follows as the ``decode`` sub-record with its own
roofline, oracle rate and end-to-end rate, and moe_reduce_fused alone on the
bf16 512 / 4096 x 8 x 7168 workloads as ``reduce_fused_bf16_x8_7168``.

Prints ONE JSON line (rank 0).  ``value`` = tokens processed by all ranks /
max-over-ranks time.  ``e2e`` = the same metric through the public
``binding.ForwardPipeline``: batches of tokens in pinned host memory, every
batch's host-to-device and device-to-host copies inside the timed region
(overlapping the neighbouring batches' forwards); ``e2e.serial_value`` the
same through ``binding.ForwardGraph`` one step at a time.
``cpu_baseline`` = the oracle's whole forward on the host cores over a
bounded sample of the same workload (for prefill: tokens of the same batch).
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


def kernels_per_step(cfg) -> int:
    """Kernels of one forward: gate (from 1024 tokens the tensor-core logits
    and the selection; below, the CUDA-core gate plus a top-k kernel when
    E > 64), dispatch (one kernel up to 16384 pairs and 256 experts, else
    two), gather (none when T <= 64: the expert MLP gathers its rows itself),
    the expert MLP (both GEMM stages in one launch) and the combine."""
    gate = 2 if cfg.T >= 1024 and cfg.d_hidden % 64 == 0 else (1 if cfg.n_experts <= 64 else 2)
    dispatch = 1 if cfg.T * cfg.top_k <= 16384 and cfg.n_experts <= 256 else 2
    gather = 0 if cfg.T <= 64 else 1
    return gate + dispatch + gather + 2


# DRAM bytes (read + write) of one expert-MLP launch from one ncu capture
# (1-pass dram__bytes_read.sum + dram__bytes_write.sum on GB300) per
# workload, valid for the kernel sources whose hash is given; any later change
# to those sources reports null.
MLP_TRAFFIC = {
    "decode": {"sources": ["mixture_experts_routed_gate_gb300/csrc/grouped_gemm.cu",
                           "mixture_experts_routed_gate_gb300/csrc/common.cuh"],
               "source_sha256_16": "5d6fd8826b004c65", "bytes": 604787712 + 2955264},
    "prefill": {"sources": ["mixture_experts_routed_gate_gb300/csrc/grouped_mlp2.cu",
                            "mixture_experts_routed_gate_gb300/csrc/common.cuh"],
                "source_sha256_16": "57ababa2a64f2460", "bytes": 15753160704 + 583650816},
}


def sources_hash(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def mlp_traffic(workload: str):
    rec = MLP_TRAFFIC.get(workload)
    if rec is None or rec["bytes"] is None or sources_hash(rec["sources"]) != rec["source_sha256_16"]:
        return None
    return rec["bytes"]


def mlp_kernel_name(cfg) -> str:
    """The expert-MLP kernel the forward launches for this workload."""
    if cfg.T <= 64:
        return "grouped_gemm_kernel<MLP_FEW> (one SM per tile, rows gathered in the kernel)"
    if cfg.d_expert % 256 == 0 and cfg.d_hidden % 512 == 0 and cfg.T * cfg.top_k // 256 + cfg.n_experts <= 512:
        return "grouped_mlp2_kernel (SM pairs, tcgen05 cta_group::2)"
    return "grouped_gemm_kernel<MLP> (one SM per tile)"


def forward_stages(T: int) -> list:
    """The entry points of one forward, in order (moe_forward makes the same
    calls; for T <= 64 the expert MLP gathers its rows and there is no gather)."""
    if T <= 64:
        return ["gate_topk", "dispatch", "expert_mlp", "reduce"]
    return ["gate_topk", "dispatch", "gather", "expert_mlp", "reduce"]


# stages `--only` can time alone: the forward's, plus the two GEMM stages as
# separate launches
ONLY_STAGES = ["gate_topk", "dispatch", "gather", "expert_mlp", "reduce", "gate_up_silu", "down",
               "w4_expert_mlp"]


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


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(total_ms: float, world: int, device=None) -> float:
    """The slowest rank's timed-region length (every rank calls this)."""
    if world <= 1:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: int, world: int, total_ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (weak scaling: each rank runs its own replica)."""
    return units_per_rank * world / (total_ms / 1e3)


# ----------------------------------------------------------------------------- native arm

class NativeStep:
    """Pre-marshalled C-ABI calls of one forward step (no per-call Python checks)."""

    def __init__(self, cfg, d, dev):
        from mixture_experts_routed_gate_gb300 import binding
        L = binding.lib()
        self.L = L
        self.cfg = cfg
        T, d_h, d_e, E, k = cfg.T, cfg.d_hidden, cfg.d_expert, cfg.n_experts, cfg.top_k
        self.T, self.k, self.E = T, k, E
        self.stages = forward_stages(T)
        dt = d["x"].dtype
        self.code = {torch.float16: 0, torch.bfloat16: 1}[dt]
        self.ws = torch.empty(binding.forward_workspace_bytes(T, d_h, d_e, E, k, dt),
                              dtype=torch.uint8, device=dev)
        self.v = binding.forward_workspace_views(self.ws, T, d_h, d_e, E, k, dt)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.out = torch.empty((T, d_h), dtype=dt, device=dev)
        self.d = d
        self.mb = binding.num_m_blocks(T, k, E)
        off = lambda i: int(L.moe_forward_workspace_offset(T, d_h, d_e, E, k, self.code, i))
        self.scratch_ptr = self.ws.data_ptr() + off(10)
        self.scratch_bytes = int(L.moe_build_dispatch_workspace_bytes(T, k, E))

    def forward_call(self, x, stream_ptr):
        """(function, argument tuple) of one moe_forward call (the product entry)."""
        cfg, d, L = self.cfg, self.d, self.L
        p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
        return (L.moe_forward, (p(x), p(d["wg"]), p(d["bias"]), p(d["w_gate"]), p(d["w_up"]),
                                p(d["w_down"]), self.T, cfg.d_hidden, cfg.d_expert, self.E, self.k,
                                self.code, p(self.ws), self.ws.numel(), p(self.out), p(self.err),
                                ctypes.c_void_p(stream_ptr)))

    def calls(self, x, stream_ptr, names=None):
        """(function, argument tuple) of the named entry points (default: the
        calls of one forward, in order)."""
        names = self.stages if names is None else names
        cfg, v, d, L = self.cfg, self.v, self.d, self.L
        p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
        T, k, E, d_h, d_e = self.T, self.k, self.E, cfg.d_hidden, cfg.d_expert
        Tk = T * k
        sp = ctypes.c_void_p(stream_ptr)
        tables = (p(v["group_sizes"]), p(v["group_offsets"]), p(v["group_padded_offsets"]),
                  p(v["group_idx_for_bx"]))
        ready = ctypes.c_void_p(self.v["mlp_ready"].data_ptr())
        by_name = {
            "gate_topk": (L.moe_gate_topk, (p(x), p(d["wg"]), p(d["bias"]), T, d_h, E, k, self.code,
                               p(v["topk_idx"]), p(v["topk_w"]), p(v["logits"]),
                               int(L.moe_gate_topk_workspace_bytes(T, E)), sp)),
            "dispatch": (L.moe_build_dispatch, (p(v["topk_idx"]), p(v["topk_w"]), T, k, E, 128, *tables,
                                    p(v["sorted_token_idx"]), p(v["sorted_row_weight"]),
                                    p(v["token_topk_to_pos"]), ctypes.c_void_p(self.scratch_ptr),
                                    self.scratch_bytes, sp)),
            # the token-order gather moe_forward runs
            "gather": (L.moe_gather_rows_by_token, (p(x), p(v["token_topk_to_pos"]), T, k, Tk, d_h, self.code,
                                                    p(v["a"]), None, sp)),
            # the gathering form for T <= 64 (rows from x), as moe_forward does
            "expert_mlp": (L.moe_grouped_mlp, (None if T <= 64 else p(v["a"]), p(d["w_gate"]), p(d["w_up"]),
                                               p(d["w_down"]), *tables, self.mb, None, Tk, d_h, d_e, E,
                                               self.code, p(v["h"]), p(v["y"]), ready,
                                               p(x) if T <= 64 else None,
                                               p(v["sorted_token_idx"]) if T <= 64 else None,
                                               T if T <= 64 else 0, p(self.err), sp)),
            "gate_up_silu": (L.moe_grouped_gate_up_silu, (p(v["a"]), p(d["w_gate"]), p(d["w_up"]), *tables, self.mb,
                                          Tk, d_h, d_e, E, self.code, p(v["h"]), p(self.err), sp)),
            "down": (L.moe_grouped_down, (p(v["h"]), p(d["w_down"]), *tables, self.mb, None, Tk, d_h, d_e, E,
                                  self.code, p(v["y"]), p(self.err), sp)),
            "reduce": (L.moe_reduce_fused, (p(v["y"]), Tk, p(v["token_topk_to_pos"]), p(v["topk_w"]), T, k, d_h,
                                  self.code, self.code, p(self.out), p(self.err), sp)),
        }
        return [by_name[n] for n in names]


def run_calls(calls, evs=None, stream=None):
    from mixture_experts_routed_gate_gb300 import binding
    if evs is not None:
        evs[0].record(stream)
    for j, (fn, args) in enumerate(calls):
        st = fn(*args)
        if st != 0:
            raise RuntimeError(f"{fn.__name__}: {binding.lib().moe_status_string(st).decode()}")
        if evs is not None:
            evs[j + 1].record(stream)


class L2Flush:
    """Evict L2 between timed steps: write a 256 MB buffer (evicts everything),
    then read a second 256 MB buffer so that L2 ends up holding clean lines of
    unrelated data (no write-backs leak into the next timed step)."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.fill_(7)
        torch.amax(self.r, dim=0, out=self.sink)


def timing_events(n):
    """Events that record inside a captured graph (external record nodes)."""
    return [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n)]


def run_native(args, cfg, rank, world, dev, with_aux=True):
    from mixture_experts_routed_gate_gb300 import binding
    _build.build()
    binding.lib()
    torch.cuda.set_device(dev)
    d = workloads.make_moe_inputs(cfg, device=dev, seed=cfg.seed)
    n_pool = 4
    x_pool = [d["x"]] + [workloads.make_tokens(cfg, cfg.T, device=dev, seed=i) for i in range(1, n_pool)]
    step = NativeStep(cfg, d, dev)
    stream = torch.cuda.Stream(dev)
    flush = L2Flush(dev)
    calls = [step.calls(x, stream.cuda_stream) for x in x_pool]
    fwd_calls = [[step.forward_call(x, stream.cuda_stream)] for x in x_pool]

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush()
            run_calls(calls[i % n_pool])
        stream.synchronize()
        if int(step.err.item()) != 0:
            raise RuntimeError(f"device error flag {int(step.err.item())} after warm-up")
        # routing statistics of each pooled batch (for the algorithmic byte counts)
        act_experts, sizes_pool = [], []
        for i in range(n_pool):
            run_calls(calls[i])
            stream.synchronize()
            sz = step.v["group_sizes"].cpu().numpy().copy()
            sizes_pool.append(sz)
            act_experts.append(int((sz > 0).sum()))

        # Two CUDA graphs per pooled batch: one moe_forward call (timed for
        # the step value) and the six entry points with event record nodes
        # between them (timed for the per-kernel breakdown).
        graphs, igraphs, gevents = [], [], []
        mode = "cuda_graph"
        try:
            for i in range(n_pool):
                run_calls(fwd_calls[i])  # first call outside capture
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    run_calls(fwd_calls[i])
                graphs.append(g)
                evs = timing_events(len(step.stages) + 1)
                gi = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gi, stream=stream):
                    run_calls(calls[i], evs, stream)
                igraphs.append(gi)
                gevents.append(evs)
            for i in range(n_pool):
                graphs[i].replay()
                igraphs[i].replay()
            stream.synchronize()
        except Exception as exc:  # capture not available: time eager launches instead
            mode = f"eager ({type(exc).__name__})"
            graphs, igraphs = [], []

        # eager timing (the host launches every kernel), for the record
        eager_ms = []
        evs_e = [torch.cuda.Event(enable_timing=True) for _ in range(len(step.stages) + 1)]
        for i in range(min(args.steps, 50)):
            flush()
            run_calls(calls[i % n_pool], evs_e, stream)
            evs_e[-1].synchronize()
            eager_ms.append(evs_e[0].elapsed_time(evs_e[-1]))

        sampler = ClockSampler(dev.index if dev.index is not None else 0)
        if world > 1:
            torch.distributed.barrier()
        stream.synchronize()
        sampler.start()
        time.sleep(0.15)
        # timed region: K steps, events around each step (the step value)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            if graphs:
                graphs[i % n_pool].replay()
            else:
                run_calls(fwd_calls[i % n_pool])
            ends[i].record(stream)
        stream.synchronize()
        t_wall = time.perf_counter() - t_wall
        step_ms = np.array([s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)])
        # the same K steps with events between the kernels (per-kernel times)
        per_stage = np.zeros((args.steps, len(step.stages)))
        for i in range(args.steps):
            flush()
            if igraphs:
                igraphs[i % n_pool].replay()
                evs = gevents[i % n_pool]
            else:
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(step.stages) + 1)]
                run_calls(calls[i % n_pool], evs, stream)
            evs[-1].synchronize()
            per_stage[i] = [evs[j].elapsed_time(evs[j + 1]) for j in range(len(step.stages))]
        stream.synchronize()
        clocks = sampler.stop()
        if world > 1:
            torch.distributed.barrier()
    total_ms = max_over_ranks(float(step_ms.sum()), world, dev)
    if int(step.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(step.err.item())} in the timed region")

    e2e = measure_e2e(args, cfg, d, dev, flush, world)
    aux = measure_reduce_aux(dev, flush) if rank == 0 and with_aux else None
    w4 = measure_w4(cfg, d, dev, flush) if rank == 0 and cfg.T <= 64 else None
    if w4 is not None:
        w4["w4a8_gemm"] = measure_w4a8(dev, flush)
    return dict(per_stage=per_stage, stages=list(step.stages), w4=w4, total_ms=total_ms, act_experts=act_experts,
                sizes_pool=sizes_pool, clocks=clocks, e2e=e2e, aux=aux, mode=mode,
                eager_ms=float(np.median(eager_ms)), wall_s=t_wall)


def quantize_int4(w):
    """Per-output-channel symmetric int4 of a stacked [E, N, K] weight:
    s = max|w| / 7 over K, q = clamp(round(w / s), -8, 7), packed two per
    byte in the pages' order ([E, N, K // 2] uint8).  Setup only."""
    wf = w.float()
    s = (wf.abs().amax(dim=2) / 7.0).clamp_min(1e-12)
    q = torch.clamp(torch.round(wf / s[..., None]), -8, 7).to(torch.int16)
    plain = ((q[..., 0::2] & 0xF) | ((q[..., 1::2] & 0xF) << 4)).to(torch.uint8).contiguous()
    return plain, s.contiguous()


def measure_w4(cfg, d, dev, flush, steps: int = 200):
    """The decode forward with int4 experts (moe_forward_w4a16; the same
    random-init weights quantised per output channel), and its expert MLP
    alone against the weight-streaming roofline."""
    from mixture_experts_routed_gate_gb300 import binding
    T, d_h, d_e, E, k = cfg.T, cfg.d_hidden, cfg.d_expert, cfg.n_experts, cfg.top_k
    qg, sg = quantize_int4(d["w_gate"])
    qu, su = quantize_int4(d["w_up"])
    qd, sd = quantize_int4(d["w_down"])
    ex = binding.Int4Experts(qg, qu, qd, sg, su, sd)
    del qg, qu, qd
    ws = torch.empty(binding.forward_workspace_bytes(T, d_h, d_e, E, k, d["x"].dtype), dtype=torch.uint8,
                     device=dev)
    out = torch.empty((T, d_h), dtype=d["x"].dtype, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    v = binding.forward_workspace_views(ws, T, d_h, d_e, E, k, d["x"].dtype)
    tables = {n: v[n] for n in ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx")}
    fwd = lambda: binding.moe_forward_w4a16(d["x"], d["wg"], d["bias"], ex, k, ws=ws, out=out, err=err)
    ready = torch.empty(tables["group_idx_for_bx"].numel() + 1, dtype=torch.int32, device=dev)
    mlp = lambda: binding.moe_grouped_mlp_w4a16(d["x"], v["sorted_token_idx"], ex, tables, h=v["h"], y=v["y"],
                                                ready=ready, err=err)
    stream = torch.cuda.Stream(dev)
    res = {}
    with torch.cuda.stream(stream):
        fwd()
        mlp()
        stream.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error flag {int(err.item())} in the int4 forward")
        sizes = v["group_sizes"].cpu().numpy()
        e_act = int((sizes > 0).sum())
        for name, fn in (("forward", fwd), ("expert_mlp", mlp)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            for _ in range(3):
                flush()
                g.replay()
            ts = []
            for _ in range(steps):
                flush()
                s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s_.record(stream)
                g.replay()
                e_.record(stream)
                e_.synchronize()
                ts.append(s_.elapsed_time(e_))
            res[name] = float(np.mean(ts))
    Tk = T * k
    w_bytes = 3 * e_act * d_e * d_h // 2 + 4 * e_act * (2 * d_e + d_h)
    mlp_bytes = w_bytes + Tk * (2 * d_h + 2 * d_e) * 2
    peaks, _ = load_peaks()
    gbs = mlp_bytes / (res["expert_mlp"] * 1e-3) / 1e9
    return {"weights": "int4 per output channel (symmetric, max|w|/7), fp32 scales", "active_experts": e_act,
            "ms_per_step": round(res["forward"], 5), "tokens_per_s": round(T / (res["forward"] * 1e-3), 1),
            "expert_mlp_us": round(res["expert_mlp"] * 1e3, 2), "expert_mlp_bytes": mlp_bytes,
            "expert_mlp_gbs": round(gbs, 1), "expert_mlp_frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "expert_mlp_note": "the standalone call includes the stream memset of its counters"}


def measure_w4a8(dev, flush, steps: int = 100):
    """The W4A8 GEMM (moe_gemm_w4a8: int4 weights x int8 activations, exact
    int32 sums) on the serving shapes beside the pages' w4a8_dequant_gemm,
    one whole call (counter memset, the K-split output memset, the int8 ->
    fp16 row kernel and the GEMM) per timed replay, against the bytes the
    product has to move (packed weights, activations, int32 result)."""
    from mixture_experts_routed_gate_gb300 import binding
    peaks, _ = load_peaks()
    stream = torch.cuda.Stream(dev)
    out = {}
    for name, (M, N, K) in workloads.W4A8_SHAPES.items():
        d = workloads.make_w4a8_inputs(M, N, K, seed=1, device=dev)
        bp = binding.moe_pack_int4_weights(d["b"], 256)
        a = d["a"]
        ct = torch.empty((N, M), dtype=torch.int32, device=dev)
        ws = torch.empty(int(binding.lib().moe_gemm_w4a8_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        fn = lambda: binding.moe_gemm_w4a8(a, bp, N, out=ct, ws=ws, err=err)
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            if int(err.item()) != 0:
                raise RuntimeError(f"device error flag {int(err.item())} in the W4A8 GEMM")
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            for _ in range(3):
                flush()
                g.replay()
            ts = []
            for _ in range(steps):
                flush()
                s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s_.record(stream)
                g.replay()
                e_.record(stream)
                e_.synchronize()
                ts.append(s_.elapsed_time(e_))
        us = float(np.mean(ts)) * 1e3
        nbytes = N * K // 2 + M * K + 4 * N * M
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"M": M, "N": N, "K": K, "us": round(us, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                     "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del d, bp, a, ct, ws, g
    return out


def measure_e2e(args, cfg, d, dev, flush, world):
    """The public API end to end, two ways, both with every step's tokens
    copied host -> device from pinned memory and its output copied back
    inside the timed region:

    * pipelined (the reported ``e2e``): binding.ForwardPipeline over K
      batches back to back, batch i + 1's copy in and batch i - 1's copy out
      overlapping batch i's forward (copy engines, two further streams); one
      timed region from before the first copy in to after the last copy out.
      No L2 eviction between batches: each batch's tokens arrive over the
      host link and every forward reads the whole expert weight set, which is
      larger than L2.
    * serial: binding.ForwardGraph with host buffers (a copy kernel reading
      the pinned tokens, the combine storing into the pinned output), one
      step per timed region after an L2 eviction."""
    from mixture_experts_routed_gate_gb300 import binding
    T, d_h = cfg.T, cfg.d_hidden
    n_pool = 4
    host_x = [workloads.make_tokens(cfg, T, device="cpu", seed=100 + i).pin_memory() for i in range(n_pool)]
    # pipelined
    pl = binding.ForwardPipeline(d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k, T)
    host_out = [torch.empty((T, d_h), dtype=host_x[0].dtype).pin_memory() for _ in range(2)]
    for i in range(max(args.warmup, 3)):
        pl.submit(host_x[i % n_pool], host_out[i % 2])
    pl.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(pl.copy_in)
    for i in range(args.steps):
        last = pl.submit(host_x[i % n_pool], host_out[i % 2])
    t1.record(pl.copy_out)
    t1.synchronize()
    pipe_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    if int(pl.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(pl.err.item())} in the pipelined e2e region")
    del pl
    # serial, one step per timed region
    fg = binding.ForwardGraph(d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k, T,
                              host_io=True)
    stream = fg.stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            flush()
            fg.x_host.copy_(host_x[i % n_pool])
            fg.replay()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        total_ms = 0.0
        for i in range(args.steps):
            fg.x_host.copy_(host_x[i % n_pool])  # host side: the caller's tokens into pinned memory
            flush()
            starts[i].record(stream)
            fg.replay()
            ends[i].record(stream)
            ends[i].synchronize()
            total_ms += starts[i].elapsed_time(ends[i])
    total_ms = max_over_ranks(total_ms, world, dev)
    if int(fg.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(fg.err.item())} in the e2e region")
    es = fg.x.element_size()
    return dict(total_ms=pipe_ms, serial_ms=total_ms, h2d=T * d_h * es, d2h=T * d_h * es)


def measure_reduce_aux(dev, flush, reps: int = 20):
    """moe_reduce_fused alone on the bf16 T x 8 x 7168 workloads (GB/s): one
    launch per timed region after an L2 eviction (the pages' protocol), and
    launches back to back on rotating cold inputs; the scaled variants at
    T = 512 (x_sf; e4m3 output; sf + e4m3 output)."""
    from mixture_experts_routed_gate_gb300 import binding

    def time_it(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush()
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record()
            fn()
            e_.record()
            e_.synchronize()
            ts.append(s_.elapsed_time(e_))
        return statistics.median(ts)

    def streamed(c, n_sets, launches):
        """Launches back to back in one CUDA graph, each on the next of n_sets
        input sets (together several times the L2), so every launch reads cold
        rows; per-launch time = replay time / launches."""
        sets = [workloads.make_reduce_inputs(c.T, c.K, c.H, c.dtype, c.seed + i, device=dev)
                for i in range(n_sets)]
        outs = [torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev) for _ in range(n_sets)]
        nb = sum(roofline.reduce_bytes(int((r["pos"] >= 0).sum().item()), c.T, c.K, c.H, 2, 2)
                 for r in sets) / n_sets
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for i in range(n_sets):  # first use outside the capture (attributes, lazy init)
                binding.moe_reduce_fused(sets[i]["x"], sets[i]["pos"], sets[i]["w"], out=outs[i])
            side.synchronize()
            with torch.cuda.graph(g, stream=side):
                for j in range(launches):
                    r = sets[j % n_sets]
                    binding.moe_reduce_fused(r["x"], r["pos"], r["w"], out=outs[j % n_sets])
        torch.cuda.current_stream(dev).wait_stream(side)
        ms = time_it(g.replay) / launches
        del g, sets, outs
        return {"streamed_us": round(ms * 1e3, 2), "streamed_gbs": round(nb / (ms * 1e-3) / 1e9, 1),
                "streamed_sets": n_sets, "streamed_launches": launches}

    res = {}
    for name in ("reduce-512", "reduce-4096"):
        c = workloads.REDUCE_CONFIGS[name]
        r = workloads.make_reduce_inputs(c.T, c.K, c.H, c.dtype, c.seed, device=dev, scales=True)
        out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev)
        n_valid = int((r["pos"] >= 0).sum().item())
        nbytes = roofline.reduce_bytes(n_valid, c.T, c.K, c.H, 2, 2)
        ms = time_it(lambda: binding.moe_reduce_fused(r["x"], r["pos"], r["w"], out=out))
        res[name] = {"us": round(ms * 1e3, 2), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "bytes": nbytes, "bytes_pages_formula": roofline.reduce_bytes_pages(c.T, c.K, c.H, 2)}
        res[name].update(streamed(c, 8, 32) if c.T <= 512 else streamed(c, 2, 8))
        if name != "reduce-512":
            continue
        out8 = torch.empty((c.T, c.H), dtype=torch.float8_e4m3fn, device=dev)
        variants = {
            "with_x_sf": (lambda: binding.moe_reduce_fused_scaled(r["x"], r["pos"], r["w"], x_sf=r["x_sf"], out=out),
                          nbytes + n_valid * 4),
            "fp8_out": (lambda: binding.moe_reduce_fused_scaled(r["x"], r["pos"], r["w"], out=out8),
                        nbytes - c.T * c.H),
            "quantized": (lambda: binding.moe_reduce_fused_scaled(r["x"], r["pos"], r["w"], sf=r["sf"], out=out8),
                          nbytes - c.T * c.H + c.T * 4),
        }
        for vname, (fn, vb) in variants.items():
            ms = time_it(fn)
            res[f"{name}-{vname}"] = {"us": round(ms * 1e3, 2), "gbs": round(vb / (ms * 1e-3) / 1e9, 1), "bytes": vb}
    return res


# ----------------------------------------------------------------------------- one stage alone

def run_only(args):
    """Time one stage of the forward alone on a (possibly reduced) workload;
    used to profile a single kernel with ncu on a small case.  Prints one JSON
    line with the stage's median event time; not the benchmark line."""
    import dataclasses
    from mixture_experts_routed_gate_gb300 import binding
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(dev)
    info = {}
    if args.only.startswith("reduce"):
        c = workloads.REDUCE_CONFIGS[args.only]
        r = workloads.make_reduce_inputs(c.T, c.K, c.H, c.dtype, c.seed, device=dev)
        out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev)
        def fn():
            binding.moe_reduce_fused(r["x"], r["pos"], r["w"], out=out)
        n_valid = int((r["pos"] >= 0).sum().item())
        info = {"workload": f"{c.name}: T={c.T} K={c.K} H={c.H} bf16",
                "bytes": roofline.reduce_bytes(n_valid, c.T, c.K, c.H, 2, 2)}
    elif args.only.startswith("w4a8-"):
        M, N, K = workloads.W4A8_SHAPES[args.only[len("w4a8-"):]]
        d = workloads.make_w4a8_inputs(M, N, K, seed=1, device=dev)
        bp = binding.moe_pack_int4_weights(d["b"], 256)
        ct = torch.empty((N, M), dtype=torch.int32, device=dev)
        ws = torch.empty(int(binding.lib().moe_gemm_w4a8_workspace_bytes(M, K)), dtype=torch.uint8, device=dev)
        def fn():
            binding.moe_gemm_w4a8(d["a"], bp, N, out=ct, ws=ws)
        info = {"workload": f"W4A8 GEMM M={M} N={N} K={K}", "bytes": N * K // 2 + M * K + 4 * N * M}
    elif args.only == "gate_topk":
        base = workloads.MOE_CONFIGS[args.workload]
        T = args.tokens or base.T
        cfg = dataclasses.replace(base, batch=1, seq=T, n_experts=args.experts or base.n_experts)
        d = workloads.make_moe_inputs(cfg, device=dev, with_experts=False)
        E, k = cfg.n_experts, cfg.top_k
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        ws = torch.empty(int(binding.lib().moe_gate_topk_workspace_bytes(T, E)), dtype=torch.uint8, device=dev)
        def fn():
            binding.moe_gate_topk(d["x"], d["wg"], d["bias"], k, topk_idx=idx, topk_w=w, ws=ws)
        info = {"workload": describe(cfg), "flops": roofline.gate_flops(T, cfg.d_hidden, E)}
    else:
        base = workloads.MOE_CONFIGS[args.workload]
        T = args.tokens or base.T
        cfg = dataclasses.replace(base, batch=1, seq=T, n_experts=args.experts or base.n_experts)
        d = workloads.make_moe_inputs(cfg, device=dev)
        step = NativeStep(cfg, d, dev)
        calls = step.calls(d["x"], stream.cuda_stream)
        with torch.cuda.stream(stream):
            run_calls(calls)  # produce every intermediate once
        stream.synchronize()
        if args.only == "w4_expert_mlp":
            # the int4 expert MLP on the same routing (weights quantised per channel)
            ex = binding.Int4Experts(*[quantize_int4(d[n])[0] for n in ("w_gate", "w_up", "w_down")])
            tables = {n: step.v[n] for n in ("group_sizes", "group_offsets", "group_padded_offsets",
                                              "group_idx_for_bx")}
            ready = torch.empty(tables["group_idx_for_bx"].numel() + 1, dtype=torch.int32, device=dev)
            def fn():
                binding.moe_grouped_mlp_w4a16(d["x"], step.v["sorted_token_idx"], ex, tables, h=step.v["h"],
                                              y=step.v["y"], ready=ready)
        else:
            fnc, fargs = step.calls(d["x"], stream.cuda_stream, names=[args.only])[0]
            def fn():
                st = fnc(*fargs)
                if st != 0:
                    raise RuntimeError(binding.lib().moe_status_string(st).decode())
        sizes = step.v["group_sizes"].cpu().numpy()
        info = {"workload": describe(cfg), "active_experts": int((sizes > 0).sum()),
                "max_rows": int(sizes.max())}
    ts = []
    with torch.cuda.stream(stream):
        for i in range(3 + args.steps):
            flush()
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record(stream)
            fn()
            e_.record(stream)
            e_.synchronize()
            if i >= 3:
                ts.append(s_.elapsed_time(e_))
    line = {"mode": "only", "stage": args.only, "steps": args.steps,
            "us_median": round(statistics.median(ts) * 1e3, 2), **info}
    if "bytes" in info:
        line["gbs"] = round(info["bytes"] / (statistics.median(ts) * 1e-3) / 1e9, 1)
    if "flops" in info:
        line["tflops"] = round(info["flops"] / (statistics.median(ts) * 1e-3) / 1e12, 2)
    print(json.dumps(line))


# ----------------------------------------------------------------------------- oracle arm

class OracleSample:
    """The oracle's whole forward (gate, top-k, dispatch tables, gather, both
    expert stages, combine: ``oracle.moe_forward``) on the host cores, over a
    bounded sample of a workload.

    decode / tiny: whole batches of the workload's shape (drawn on the host).
    prefill: a seeded sample of tokens of the very batch the GPU arm times
    (drawn on the GPU with the same generator, so the bits are identical),
    with the full gate (all 256 experts) and the full expert weights as
    host arrays; only the experts the sample routes to are ever read, so
    only those are copied into the (lazily committed) host arrays."""

    PREFILL_TOKENS = 32

    def __init__(self, cfg, device=None):
        from oracle import oracle
        oracle.build()
        self.oracle = oracle
        self.cfg = cfg
        if cfg.name != "prefill":
            d = workloads.make_moe_inputs(cfg, device="cpu")
            self.nb = {n: (workloads.to_numpy_bits(v) if v is not None else None) for n, v in d.items()}
            self.tokens = cfg.T
            self.sample = f"whole forward passes of the {cfg.name} workload ({cfg.T} tokens each)"
            return
        dev = device if device is not None else torch.device("cuda", 0)
        d = workloads.make_moe_inputs(cfg, device=dev)
        rng = np.random.default_rng(12345)
        tok = np.sort(rng.choice(cfg.T, self.PREFILL_TOKENS, replace=False))
        bits = workloads.to_numpy_bits
        nb = {"x": bits(d["x"][torch.from_numpy(tok).to(dev)]), "wg": bits(d["wg"]),
              "bias": d["bias"].cpu().numpy()}
        idx, _ = oracle.gate_topk(nb["x"], nb["wg"], nb["bias"], cfg.top_k, cfg.dtype)
        used = np.unique(idx)
        E, d_h, d_e = cfg.n_experts, cfg.d_hidden, cfg.d_expert
        for name, shape in (("w_gate", (E, d_e, d_h)), ("w_up", (E, d_e, d_h)), ("w_down", (E, d_h, d_e))):
            host = np.empty(shape, np.uint16)  # pages of unused experts are never touched
            for e in used:
                host[e] = bits(d[name][int(e)])
            nb[name] = host
        del d
        torch.cuda.empty_cache()
        self.nb = nb
        self.tokens = self.PREFILL_TOKENS
        self.sample = (f"whole forward passes (gate over all {E} experts, top-{cfg.top_k}, dispatch, both "
                       f"expert stages, combine) of {self.PREFILL_TOKENS} seeded tokens of the prefill "
                       f"batch, routed to {used.size} experts")

    def run_once(self):
        nb, cfg = self.nb, self.cfg
        self.oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                                cfg.top_k, cfg.dtype)

    def rate(self, budget_s: float, min_runs: int = 1):
        """tokens/s over whole forward passes filling about budget_s seconds."""
        runs, t0 = 0, time.perf_counter()
        while True:
            self.run_once()
            runs += 1
            el = time.perf_counter() - t0
            if runs >= min_runs and el >= budget_s:
                break
        return dict(value=self.tokens * runs / el, seconds=el, runs=runs,
                    sample=f"{runs} x {self.sample}"), self.oracle.threads(0)


# ----------------------------------------------------------------------------- records

def workload_record(args, cfg, res, world, steps, cpu_budget, dev):
    """The figures of one workload's timed run: tokens/s, per-kernel times,
    the expert MLP's roofline, the oracle's rate and the end-to-end rate."""
    peaks, peak_src = load_peaks()
    T, k, d_h, d_e, E = cfg.T, cfg.top_k, cfg.d_hidden, cfg.d_expert, cfg.n_experts
    Tk = T * k
    per_stage = res["per_stage"]
    ms_step = res["total_ms"] / steps
    value = aggregate_throughput(T * steps, world, res["total_ms"])
    e_act = float(np.mean(res["act_experts"]))
    es = 2
    flops_step = roofline.moe_forward_flops(T, k, d_h, d_e, E)
    stages = res["stages"]
    # dominant kernel: the expert MLP (both grouped GEMM stages in one launch);
    # its algorithmic bytes averaged over the pooled batches the steps cycle through
    gu_ms = float(per_stage[:, stages.index("expert_mlp")].mean())
    gu_bytes = float(np.mean([roofline.expert_mlp_bytes(Tk, d_h, d_e, a, es) for a in res["act_experts"]]))
    gu_flops = roofline.expert_mlp_flops(Tk, d_h, d_e)
    # a kernel inside a step of milliseconds runs at the sustained tensor rate
    tflops_key = "bf16_tflops_sustained" if ms_step > 1.0 else "bf16_tflops"
    t_bytes = gu_bytes / (peaks["hbm_gbs"] * 1e9)
    t_flops = gu_flops / (peaks[tflops_key] * 1e12)
    traffic = mlp_traffic(cfg.name)
    common = {"kernel": mlp_kernel_name(cfg), "traffic": traffic,
              "traffic_source": ("dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture of this "
                                 "kernel at this workload, stored with the hash of the kernel source it was "
                                 "taken on; null when the source differs" if traffic is not None else
                                 "null: the kernel source differs from the one the stored ncu counters "
                                 "were taken on"),
              "launch_us": round(gu_ms * 1e3, 2), "algorithmic_bytes_per_launch": round(gu_bytes),
              "algorithmic_flops_per_launch": gu_flops,
              "time_at_hbm_peak_us": round(t_bytes * 1e6, 2), "time_at_tensor_peak_us": round(t_flops * 1e6, 2)}
    if t_bytes >= t_flops:
        achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
        rl = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
              "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_src + " (hbm_gbs)", **common}
    else:
        achieved = gu_flops / (gu_ms * 1e-3) / 1e12
        rl = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks[tflops_key], "unit": "TFLOP/s",
              "frac": round(achieved / peaks[tflops_key], 4), "peak_source": f"{peak_src} ({tflops_key})",
              **common}
    rl["tensor_frac_of_" + tflops_key] = round(gu_flops / (gu_ms * 1e-3) / 1e12 / peaks[tflops_key], 4)
    bytes_min = float(np.mean([roofline.moe_forward_bytes_min(T, d_h, d_e, E, a, es) for a in res["act_experts"]]))
    step_roof_ms = max(bytes_min / (peaks["hbm_gbs"] * 1e9), flops_step / (peaks[tflops_key] * 1e12)) * 1e3
    sampler = OracleSample(cfg, dev)
    cpu, threads = sampler.rate(cpu_budget)
    del sampler
    e2e = res["e2e"]
    rec = {
        "value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(ms_step, 5), "steps": steps,
        "tflops": round(flops_step * steps / (res["total_ms"] / 1e3) / 1e12, 3),
        "step_roofline_frac": round(step_roof_ms / ms_step, 4),
        "kernels_us": {s: round(float(per_stage[:, i].mean()) * 1e3, 2) for i, s in enumerate(stages)},
        "kernels_note": "per-kernel times from replays of the same graphs with event nodes between the kernels",
        "active_experts": e_act,
        "expert_rows_max": int(max(int(s_.max()) for s_ in res["sizes_pool"])),
        "roofline": rl,
        "cpu_baseline": {"value": round(cpu["value"], 2), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": cpu["sample"]},
        "e2e": {"value": round(aggregate_throughput(T * steps, world, e2e["total_ms"]), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "mode": "binding.ForwardPipeline: K batches back to back from pinned host memory, each "
                        "batch's copy in and copy out (copy engines) overlapping the neighbouring batches' "
                        "forwards; one timed region; no L2 eviction (every forward reads the whole expert "
                        "weight set, larger than L2, and its tokens arrive over the host link)",
                "serial_value": round(aggregate_throughput(T * steps, world, e2e["serial_ms"]), 1),
                "serial_mode": "binding.ForwardGraph with host buffers, one step per timed region after an "
                               "L2 eviction"},
        "gpu_launches": kernels_per_step(cfg) * steps,
        "launch_mode": res["mode"],
        "eager_ms_per_step": round(res["eager_ms"], 5),
    }
    if res.get("aux") is not None:
        rec["reduce_fused_bf16_x8_7168"] = res["aux"]
    if res.get("w4") is not None:
        w4 = dict(res["w4"])
        w4a8 = w4.pop("w4a8_gemm", None)
        rec["w4a16"] = w4
        if w4a8 is not None:
            rec["w4a8_gemm"] = w4a8
    rec["clocks"] = res["clocks"]
    return rec


def config_of(cfg, args):
    return {"workload": describe(cfg), "T": cfg.T, "d_hidden": cfg.d_hidden, "d_expert": cfg.d_expert,
            "n_experts": cfg.n_experts, "top_k": cfg.top_k,
            "l2": "evicted before every timed step: 256 MB write, then a 256 MB read of another buffer",
            "parallelism": f"replicas x{args.gpus}"}


# ----------------------------------------------------------------------------- main

DEFAULT_STEPS = {"decode": 2000, "tiny": 2000, "prefill": 60}


def main():
    ap = argparse.ArgumentParser(
        description="Routed-expert MoE forward throughput: one JSON line with tokens/s, the dominant "
                    "kernel's roofline fraction, the end-to-end rate with host buffers and the oracle's rate "
                    "on the prefill workload (the headline), with the decode workload and the combine alone "
                    "as sub-records.")
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs (one rank each under torchrun; independent replicas, weak scaling)")
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps of the headline workload (default: 60 prefill, 2000 decode / tiny; "
                         "3 for the reference arm)")
    ap.add_argument("--warmup", type=int, default=5, help="untimed warm-up steps (at least 3)")
    ap.add_argument("--impl", choices=["native", "reference"], default="native",
                    help="native: the CUDA library; reference: the CPU oracle on the host cores")
    ap.add_argument("--workload", choices=list(workloads.MOE_CONFIGS), default="prefill",
                    help="headline workload. prefill: 4096 tokens, 7168/2048, 256 experts, top-8, bf16, Zipf "
                         "gate bias; decode: 64 tokens, 2048/768, 64 experts, top-6, fp16; tiny: 64 tokens, "
                         "256/128, 8 experts, top-2")
    ap.add_argument("--sub-steps", type=int, default=500,
                    help="timed steps of the decode sub-record (recorded with the prefill headline)")
    ap.add_argument("--no-sub", action="store_true", help="skip the decode sub-record")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time per workload")
    ap.add_argument("--only", default=None,
                    choices=ONLY_STAGES + ["reduce-512", "reduce-4096"] + ["w4a8-" + n for n in workloads.W4A8_SHAPES],
                    help="time one stage alone (profiling aid; not the benchmark line)")
    ap.add_argument("--experts", type=int, default=None, help="with --only: expert count override")
    ap.add_argument("--tokens", type=int, default=None, help="with --only: token count override")
    args = ap.parse_args()
    if args.only:
        args.steps = args.steps or 5
        run_only(args)
        return
    cfg = workloads.MOE_CONFIGS[args.workload]
    if args.steps is None:
        args.steps = DEFAULT_STEPS[cfg.name] if args.impl == "native" else 3
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    base = {"metric": METRIC, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype,
            "data": "synthetic: seeded N(0,1) tokens, N(0,1/fan_in) random-init expert and gate weights",
            "config": config_of(cfg, args)}

    if args.impl == "reference":
        if rank != 0:
            return
        dev = torch.device("cuda", local) if torch.cuda.is_available() else None
        sampler = OracleSample(cfg, dev)
        steps_ms, info, threads = [], None, 1
        budget = max(1.0, args.cpu_budget / max(1, args.steps))
        for i in range(args.warmup + args.steps):
            res, threads = sampler.rate(budget if i >= args.warmup else 0.0)
            if i >= args.warmup:
                steps_ms.append(cfg.T / res["value"] * 1e3)
                info = res
        tok_s = cfg.T * len(steps_ms) / (sum(steps_ms) / 1e3)
        line = dict(base, impl="reference", value=tok_s, ms_per_step=statistics.mean(steps_ms),
                    cpu_baseline={"value": tok_s, "unit": "tokens/s", "cores": threads,
                                  "kind": "oracle", "sample": f"per step: {info['sample']}"},
                    e2e={"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0})
        print(json.dumps(line))
        return

    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    dev = torch.device("cuda", local)
    res = run_native(args, cfg, rank, world, dev, with_aux=True)
    rec = workload_record(args, cfg, res, world, args.steps, args.cpu_budget, dev) if rank == 0 else None
    del res
    sub = None
    if cfg.name == "prefill" and not args.no_sub:
        # the decode workload, every rank (the replicas stay in step), recorded by rank 0
        dcfg = workloads.MOE_CONFIGS["decode"]
        sargs = argparse.Namespace(**vars(args))
        sargs.steps = max(args.sub_steps, args.steps)
        torch.cuda.empty_cache()
        dres = run_native(sargs, dcfg, rank, world, dev, with_aux=False)
        if rank == 0:
            sub = workload_record(sargs, dcfg, dres, world, sargs.steps, args.cpu_budget, dev)
            sub = {"config": config_of(dcfg, args), "dtype": dcfg.dtype, **sub}
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    line = dict(base)
    line.update(rec)
    if sub is not None:
        line["decode"] = sub
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
