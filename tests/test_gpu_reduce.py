"""moe_reduce_fused on the GPU vs the oracle (TileOPs-Metax PR #55, sections 1-2).

The kernel accumulates in the oracle's order with the oracle's roundings
(ascending slots, acc = acc + w*x, one cast), so every case is compared bit
for bit; the page's tolerances are checked as well for the record."""
import numpy as np
import pytest
import torch

from gpu_helpers import REDUCE_TOL, assert_bits_equal, assert_close, bits, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def _run(d, dtype, out_dtype=None, err=None):
    out_dtype = out_dtype or dtype
    return binding.moe_reduce_fused(d["x"], d["pos"], d["w"],
                                    out_dtype=workloads.torch_dtype(out_dtype), err=err)


def _ref(oracle, d, dtype, out_dtype=None):
    out, err = oracle.reduce_fused(bits(d["x"]), d["pos"].cpu().numpy(),
                                   None if d["w"] is None else d["w"].cpu().numpy(),
                                   dtype, out_dtype or dtype)
    return out, err


@pytest.mark.parametrize("T", [512, 4096])
def test_reduce_full_size_bit_exact(oracle, T):
    """The bf16 combine at T x 8 x 7168 (all outputs compared)."""
    dev = require_cuda()
    cfg = workloads.REDUCE_CONFIGS[f"reduce-{T}"]
    d = workloads.make_reduce_inputs(cfg.T, cfg.K, cfg.H, cfg.dtype, cfg.seed, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = _run(d, cfg.dtype, err=err)
    torch.cuda.synchronize()
    want, _ = _ref(oracle, d, cfg.dtype)
    assert int(err.item()) == 0
    assert_bits_equal(bits(out), want, "reduce out")
    assert_close(bits(out), want, "bf16", *REDUCE_TOL["bf16"], "reduce out")


@pytest.mark.parametrize("cfg", workloads.reduce_edge_configs(), ids=lambda c: c.name)
def test_reduce_edge_sweep_bit_exact(oracle, cfg):
    dev = require_cuda()
    d = workloads.make_reduce_inputs(cfg.T, cfg.K, cfg.H, cfg.dtype, cfg.seed, device=dev,
                                     weighted=cfg.weighted)
    out = _run(d, cfg.dtype)
    torch.cuda.synchronize()
    want, err = _ref(oracle, d, cfg.dtype)
    assert err == 0
    assert_bits_equal(bits(out), want, cfg.name)


@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_reduce_f32_in_half_out(oracle, out_dtype):
    dev = require_cuda()
    d = workloads.make_reduce_inputs(64, 8, 1024, "f32", 5, device=dev)
    out = _run(d, "f32", out_dtype)
    torch.cuda.synchronize()
    want, _ = _ref(oracle, d, "f32", out_dtype)
    assert_bits_equal(bits(out), want, "f32 -> half combine")


@pytest.mark.parametrize("K", [32, 40])
def test_reduce_many_slots(oracle, K):
    """K = 32 is the widest the bulk-copy kernel takes; K = 40 goes through the
    per-thread kernel."""
    dev = require_cuda()
    d = workloads.make_reduce_inputs(16, K, 512, "bf16", 8, device=dev)
    out = _run(d, "bf16")
    torch.cuda.synchronize()
    want, _ = _ref(oracle, d, "bf16")
    assert_bits_equal(bits(out), want, f"K={K}")


def test_reduce_k1_identity_and_all_padding():
    dev = require_cuda()
    T, H = 33, 512
    x = torch.randn((T, H), device=dev).to(torch.bfloat16)
    perm = torch.randperm(T, device=dev).to(torch.int32).view(T, 1)
    out = binding.moe_reduce_fused(x, perm, None)
    assert torch.equal(out, x[perm[:, 0].long()])
    ones = torch.ones((T, 1), dtype=torch.float32, device=dev)
    assert torch.equal(binding.moe_reduce_fused(x, perm, ones), x[perm[:, 0].long()])
    pad = torch.full((T, 4), -1, dtype=torch.int32, device=dev)
    out = binding.moe_reduce_fused(x, pad, torch.rand((T, 4), device=dev))
    assert torch.count_nonzero(out.float()) == 0


def test_reduce_padding_rows_never_read():
    dev = require_cuda()
    d = workloads.make_reduce_inputs(64, 8, 768, "bf16", 9, device=dev)
    out1 = _run(d, "bf16")
    pos = d["pos"]
    used = torch.zeros(d["x"].shape[0], dtype=torch.bool, device=dev)
    used[pos[pos >= 0].long()] = True
    x2 = d["x"].clone()
    x2[~used] = float("nan")
    out2 = binding.moe_reduce_fused(x2, pos, d["w"])
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_reduce_out_of_range_flagged_and_skipped(oracle):
    dev = require_cuda()
    x = torch.ones((8, 256), dtype=torch.float16, device=dev)
    pos = torch.tensor([[0, 8], [1, -3], [2, 3]], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = binding.moe_reduce_fused(x, pos, None, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5  # MOE_ERR_DEVICE_FLAG
    assert out[0].float().eq(1).all() and out[1].float().eq(1).all() and out[2].float().eq(2).all()


def test_reduce_error_cases():
    """The page's error cases: hidden % 256 != 0, topk_weights of the wrong
    dtype, shape mismatch."""
    dev = require_cuda()
    x = torch.zeros((16, 200), dtype=torch.bfloat16, device=dev)
    pos = torch.zeros((4, 2), dtype=torch.int32, device=dev)
    with pytest.raises(binding.MoEError):
        binding.moe_reduce_fused(x, pos, None)
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device=dev)
    with pytest.raises(TypeError):
        binding.moe_reduce_fused(x, pos, torch.ones((4, 2), dtype=torch.float16, device=dev))
    with pytest.raises(ValueError):
        binding.moe_reduce_fused(x, pos, torch.ones((4, 3), dtype=torch.float32, device=dev))


def test_reduce_empty_batch():
    dev = require_cuda()
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device=dev)
    pos = torch.zeros((0, 8), dtype=torch.int32, device=dev)
    out = binding.moe_reduce_fused(x, pos, None)
    assert out.shape == (0, 256)


def _variant_cases():
    cases = []
    for (T, K, H) in [(4, 2, 256), (32, 8, 3072), (512, 8, 7168)]:
        for in_dt in ("f16", "bf16", "f32"):
            if H == 7168 and in_dt != "bf16":
                continue
            for out_dt in (in_dt, "e4m3"):
                for xs in (False, True):
                    for sf in (False, True):
                        cases.append((T, K, H, in_dt, out_dt, xs, sf))
    return cases


@pytest.mark.parametrize("T,K,H,in_dt,out_dt,use_xsf,use_sf", _variant_cases(),
                         ids=lambda v: str(v))
def test_reduce_scaled_variants_bit_exact(oracle, T, K, H, in_dt, out_dt, use_xsf, use_sf):
    """The WithXsf / Fp8 / Quantized switches (TileOPs-Metax PR #55): per-row
    x_sf, per-token sf, e4m3 output; bit for bit against the oracle (the
    e4m3 rounding included), and within the page's fp8 tolerance 0.1."""
    dev = require_cuda()
    d = workloads.make_reduce_inputs(T, K, H, in_dt, 6, device=dev, scales=True)
    xs = d["x_sf"] if use_xsf else None
    sf = d["sf"] if use_sf else None
    out = binding.moe_reduce_fused_scaled(d["x"], d["pos"], d["w"], x_sf=xs, sf=sf,
                                          out_dtype=workloads.torch_dtype(out_dt))
    torch.cuda.synchronize()
    want, err = oracle.reduce_fused_scaled(bits(d["x"]), d["pos"].cpu().numpy(), d["w"].cpu().numpy(),
                                           None if xs is None else xs.cpu().numpy(),
                                           None if sf is None else sf.cpu().numpy(), in_dt, out_dt)
    assert err == 0
    assert_bits_equal(bits(out), want, "scaled combine")
    if out_dt == "e4m3":
        assert_close(bits(out), want, "e4m3", 0.1, 0.1, "fp8 combine")
