"""Gate / top-k, dispatch tables and the row gather on the GPU vs the oracle.

Routing and tables are integer results and are compared bit for bit; the
logits too, since both sides sum them in the same fixed order; the softmax
weights within rtol 1e-5."""
import json
import os

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, bits, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gate_gpu(x, wg, bias, k):
    T, E = x.shape[0], wg.shape[0]
    ws = torch.empty(T * E * 4, dtype=torch.uint8, device=x.device)
    idx, w = binding.moe_gate_topk(x, wg, bias, k, ws=ws)
    torch.cuda.synchronize()
    logits = ws.view(torch.float32).view(T, E)
    return idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def _check_gate(oracle, x, wg, bias, k, dtype):
    idx, w, logits = _gate_gpu(x, wg, bias, k)
    ref_logits = oracle.gate_logits(bits(x), bits(wg), None if bias is None else bias.cpu().numpy(), dtype)
    ref_idx, ref_w = oracle.topk_softmax(ref_logits, k)
    assert_bits_equal(logits.view(np.uint32), ref_logits.view(np.uint32), "gate logits")
    assert_bits_equal(idx, ref_idx, "topk_idx")
    assert np.allclose(w, ref_w, rtol=1e-5, atol=1e-7), float(np.abs(w - ref_w).max())
    return idx, w


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_gate_topk_workloads(oracle, name):
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS[name]
    d = workloads.make_moe_inputs(cfg, device=dev)
    _check_gate(oracle, d["x"], d["wg"], d["bias"], cfg.top_k, cfg.dtype)


@pytest.mark.parametrize("T,d_h,E,k,dtype", [(37, 512, 40, 3, "bf16"), (1, 256, 8, 8, "f16"),
                                             (100, 768, 1, 1, "bf16"), (17, 256, 1000, 32, "f16"),
                                             # the many-token shape (T >= 512, E > 64), ragged in
                                             # both tokens and experts
                                             (601, 512, 100, 4, "f16"), (530, 768, 72, 8, "bf16")])
def test_gate_topk_ragged_shapes(oracle, T, d_h, E, k, dtype):
    dev = require_cuda()
    g = torch.Generator(device=dev).manual_seed(T + E)
    x = torch.randn((T, d_h), generator=g, device=dev).to(workloads.torch_dtype(dtype))
    wg = (torch.randn((E, d_h), generator=g, device=dev) / d_h ** 0.5).to(workloads.torch_dtype(dtype))
    bias = torch.randn(E, generator=g, device=dev) * 0.1
    _check_gate(oracle, x, wg, bias, k, dtype)


def test_gate_hand_computed_order_cases():
    """The hand-computed summation-order cases, through the GPU."""
    dev = require_cuda()
    with open(os.path.join(GOLDEN, "gate_order_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        d_h = c["d_hidden"]
        w = torch.zeros((1, d_h), dtype=torch.float32)
        for j, v in c["w_at"].items():
            w[0, int(j)] = v
        x = torch.ones((1, d_h), dtype=torch.bfloat16, device=dev)
        _, _, logits = _gate_gpu(x, w.to(torch.bfloat16).to(dev), None, 1)
        assert logits[0, 0] == np.float32(c["logit"]), c["what"]


def test_gate_ties_go_to_lower_id(oracle):
    """Experts 3, 4 and 5 share one weight row and get a dominant bias: their
    logits are bitwise equal, so the order must be 3, 4, 5."""
    dev = require_cuda()
    x = torch.randn((20, 256), device=dev).to(torch.bfloat16)
    wg = (torch.randn((8, 256), device=dev) * 0.05).to(torch.bfloat16)
    wg[4] = wg[3]
    wg[5] = wg[3]
    bias = torch.zeros(8, device=dev)
    bias[3:6] = 100.0
    idx, w = _check_gate(oracle, x, wg.contiguous(), bias, 3, "bf16")
    assert (idx == np.array([3, 4, 5])).all()
    assert (w[:, 0] == w[:, 1]).all() and (w[:, 1] == w[:, 2]).all()


@pytest.mark.parametrize("T,k,E,skew", [(64, 2, 8, False), (64, 6, 64, False),
                                        (3000, 8, 256, True), (1, 4, 4, False),
                                        (500, 1, 1, False), (4096, 8, 256, True),
                                        (1024, 1, 8, False), (2048, 8, 256, True),
                                        (2049, 8, 256, True), (40, 4, 300, False),
                                        (0, 2, 8, False)])
def test_dispatch_tables_bit_exact(oracle, T, k, E, skew):
    dev = require_cuda()
    rng = np.random.default_rng(T * 7 + E)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        idx = np.array([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)], np.int32)
    else:
        idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32)
    if T == 1024 and k == 1:
        idx[:] = np.repeat(np.arange(8), 128).reshape(T, 1)  # every count a multiple of 128
    idx = idx.reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    tab = binding.moe_build_dispatch(torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev), E)
    torch.cuda.synchronize()
    ref = oracle.build_dispatch(idx, w, E, 128)
    for name, want in ref.items():
        got = tab[name].cpu().numpy().reshape(want.shape)
        if want.dtype == np.float32:
            assert_bits_equal(got.view(np.uint32), want.view(np.uint32), name)
        else:
            assert_bits_equal(got, want, name)


def test_gather_rows_bit_exact(oracle):
    dev = require_cuda()
    x = torch.randn((77, 7168), device=dev).to(torch.bfloat16)
    st = torch.randint(0, 77, (1000,), device=dev, dtype=torch.int32)
    a = binding.moe_gather_rows(x, st)
    torch.cuda.synchronize()
    want = oracle.gather_rows(bits(x), st.cpu().numpy(), "bf16")
    assert_bits_equal(bits(a), want, "gathered rows")
    x = torch.randn((9, 256), device=dev).to(torch.float16)
    st = torch.randint(0, 9, (13,), device=dev, dtype=torch.int32)
    assert_bits_equal(bits(binding.moe_gather_rows(x, st)), oracle.gather_rows(bits(x), st.cpu().numpy(), "f16"), "f16 gather")
