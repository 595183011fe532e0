"""Seeded synthetic inputs for the routed-expert MoE forward and the combine.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  The CUDA path, the CPU oracle, the tests and the
benchmark all take their inputs from here, so both sides see identical bits.

Shapes and distributions (the five workloads):
  * ``tiny``     T=64 (1x64), d_hidden=256, d_expert=128, E=8, top-2, fp16, seed 0.
  * ``decode``   T=64 (64x1), d_hidden=2048, d_expert=768, E=64, top-6, fp16.
  * ``prefill``  T=4096 (4x1024), d_hidden=7168, d_expert=2048, E=256, top-8, bf16,
                 with a per-expert logit bias -1.1*ln(rank), the ranks a seeded
                 random permutation of 1..E (a Zipf(s=1.1) prior in rank order).
  * ``reduce``   moe_reduce_fused alone, bf16, K=8, H=7168, T=512 and T=4096.
  * ``reduce-edge`` (T,K,H) in {(4,2,256),(1,8,256),(8,1,256),(32,8,3072),(512,8,3072)}.
x ~ N(0,1); gate weight ~ N(0, 1/d_hidden); expert weights ~ N(0, 1/fan_in);
values are drawn in fp32 and rounded to the storage dtype by torch (RNE).
For the combine: positions are a random permutation of 0..T*K-1 laid out as
[T,K], then ceil(0.1*T*K) slots picked by a second permutation are set to -1;
weights are a row softmax of N(0,1) logits in fp32 (or absent: unit weights).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

BLOCK_M = 128

_TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
                 "e4m3": torch.float8_e4m3fn}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


@dataclass(frozen=True)
class MoEConfig:
    name: str
    batch: int
    seq: int
    d_hidden: int
    d_expert: int
    n_experts: int
    top_k: int
    dtype: str
    seed: int
    zipf_bias: bool = False

    @property
    def T(self) -> int:
        return self.batch * self.seq


@dataclass(frozen=True)
class ReduceConfig:
    name: str
    T: int
    K: int
    H: int
    dtype: str
    seed: int
    weighted: bool = True


MOE_CONFIGS = {
    "tiny": MoEConfig("tiny", 1, 64, 256, 128, 8, 2, "f16", 0),
    "decode": MoEConfig("decode", 64, 1, 2048, 768, 64, 6, "f16", 1),
    "prefill": MoEConfig("prefill", 4, 1024, 7168, 2048, 256, 8, "bf16", 2, zipf_bias=True),
}

REDUCE_CONFIGS = {
    "reduce-512": ReduceConfig("reduce-512", 512, 8, 7168, "bf16", 3),
    "reduce-4096": ReduceConfig("reduce-4096", 4096, 8, 7168, "bf16", 3),
}

# The W4A8 GEMM's serving shapes (TileLang tutorial ch.18 skeletons.py,
# SERVING_SHAPES beside w4a8_dequant_gemm): a decode step (M = 1) and a small
# batch (M = 32), N x K one weight matrix of that size.
W4A8_SHAPES = {
    "gemv_like": (1, 3584, 18944),
    "small_batch": (32, 3584, 18944),
}

REDUCE_EDGE_SHAPES = [(4, 2, 256), (1, 8, 256), (8, 1, 256), (32, 8, 3072), (512, 8, 3072)]


def reduce_edge_configs():
    out = []
    for dt in ("f16", "bf16", "f32"):
        for (T, K, H) in REDUCE_EDGE_SHAPES:
            for weighted in (True, False):
                out.append(ReduceConfig(f"edge-{T}x{K}x{H}-{dt}-{'w' if weighted else 'unit'}",
                                        T, K, H, dt, 4, weighted))
    return out


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, dtype: str, gen: torch.Generator, device) -> torch.Tensor:
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(torch_dtype(dtype))


def _stacked_normal(E: int, rows: int, cols: int, std: float, dtype: str,
                    gen: torch.Generator, device) -> torch.Tensor:
    """[E, rows, cols] drawn one expert at a time (bounded fp32 temporaries)."""
    out = torch.empty((E, rows, cols), dtype=torch_dtype(dtype), device=device)
    for e in range(E):
        out[e].copy_(_normal((rows, cols), std, dtype, gen, device))
    return out


def make_moe_inputs(cfg: MoEConfig, device="cpu", seed: int | None = None,
                    T: int | None = None, with_experts: bool = True) -> dict:
    """x [T,d_h]; wg [E,d_h]; bias [E] fp32 or None; w_gate, w_up [E,d_e,d_h];
    w_down [E,d_h,d_e].  ``T`` overrides the token count (same weights);
    ``with_experts=False`` skips the expert weights (gate-only use)."""
    seed = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    d_h, d_e, E, dt = cfg.d_hidden, cfg.d_expert, cfg.n_experts, cfg.dtype
    gen = _gen(device, seed)
    wg = _normal((E, d_h), 1.0 / math.sqrt(d_h), dt, gen, device)
    bias = None
    if cfg.zipf_bias:
        rank = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
        bias = (-1.1 * torch.log(rank)).to(torch.float32)
    w_gate = w_up = w_down = None
    if with_experts:
        w_gate = _stacked_normal(E, d_e, d_h, 1.0 / math.sqrt(d_h), dt, gen, device)
        w_up = _stacked_normal(E, d_e, d_h, 1.0 / math.sqrt(d_h), dt, gen, device)
        w_down = _stacked_normal(E, d_h, d_e, 1.0 / math.sqrt(d_e), dt, gen, device)
    xgen = _gen(device, seed * 1000003 + T)
    x = _normal((T, d_h), 1.0, dt, xgen, device)
    return dict(x=x, wg=wg, bias=bias, w_gate=w_gate, w_up=w_up, w_down=w_down)


def make_tokens(cfg: MoEConfig, T: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """A fresh batch of activations x [T, d_hidden] for the same layer."""
    gen = _gen(device, 7919 * (seed + 1) + cfg.seed)
    return _normal((T, cfg.d_hidden), 1.0, cfg.dtype, gen, device)


def make_reduce_inputs(T: int, K: int, H: int, dtype: str, seed: int, device="cpu",
                       weighted: bool = True, pad_fraction: float = 0.1, scales: bool = False) -> dict:
    """x [T*K, H]; token_topk_to_pos [T,K] int32 (-1 = padding); topk_weights [T,K] fp32 or None.
    With ``scales``: x_sf [T*K] fp32 and sf [T] fp32, both log-uniform in [1/4, 4]."""
    gen = _gen(device, seed * 7 + T * 131 + K * 17 + H)
    n = T * K
    x = _normal((n, H), 1.0, dtype, gen, device)
    pos = torch.randperm(n, generator=gen, device=device).to(torch.int32)
    n_pad = int(math.ceil(pad_fraction * n))
    pad_slots = torch.randperm(n, generator=gen, device=device)[:n_pad]
    pos[pad_slots] = -1
    pos = pos.view(T, K)
    w = None
    if weighted:
        logits = torch.randn((T, K), generator=gen, device=device, dtype=torch.float32)
        w = torch.softmax(logits, dim=1)
    out = dict(x=x, pos=pos, w=w)
    if scales:
        u = torch.rand((n + T,), generator=gen, device=device, dtype=torch.float32)
        s = torch.exp2(u * 4.0 - 2.0)
        out.update(x_sf=s[:n].contiguous(), sf=s[n:].contiguous())
    return out


def make_w4a8_inputs(M: int, N: int, K: int, seed: int, device="cpu", E: int = 1) -> dict:
    """Uniform int8 activations a [M, K] and uniform packed int4 weights b
    [E, N, K // 2] (every byte value equally likely: both nibbles uniform
    over -8..7), the layout the pages print."""
    gen = _gen(device, seed * 104729 + M * 31 + N * 7 + K)
    a = torch.randint(-128, 128, (M, K), generator=gen, device=device, dtype=torch.int32).to(torch.int8)
    b = torch.randint(0, 256, (E, N, K // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    return dict(a=a, b=b)


def to_numpy_bits(t: torch.Tensor):
    """Host numpy view of a tensor; 16-bit floats come back as uint16 bits."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def from_numpy_bits(a, dtype: str) -> torch.Tensor:
    """Inverse of :func:`to_numpy_bits` for a storage dtype name."""
    import numpy as np
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch_dtype(dtype))
