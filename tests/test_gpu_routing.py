"""Gate / top-k, dispatch tables and the row gather on the GPU vs the oracle.

Routing and tables are integer results and are compared bit for bit; the
logits too, since both sides sum them in the same fixed order; the softmax
weights within rtol 1e-5."""
import json
import os

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, bits, check_gate_logits, gate_uses_tensor_cores, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gate_gpu(x, wg, bias, k):
    T, E = x.shape[0], wg.shape[0]
    need = int(binding.lib().moe_gate_topk_workspace_bytes(T, E))
    ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    idx, w = binding.moe_gate_topk(x, wg, bias, k, ws=ws)
    torch.cuda.synchronize()
    logits = ws[:T * E * 4].view(torch.float32).view(T, E)
    return idx.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def _check_gate(oracle, x, wg, bias, k, dtype):
    """Ids bit for bit, weights within rtol 1e-5, logits as check_gate_logits
    says (bit for bit, or on the tensor-core path within its bound)."""
    idx, w, logits = _gate_gpu(x, wg, bias, k)
    b = None if bias is None else bias.cpu().numpy()
    ref_logits = oracle.gate_logits(bits(x), bits(wg), b, dtype)
    ref_idx, ref_w = oracle.topk_softmax(ref_logits, k)
    assert_bits_equal(idx, ref_idx, "topk_idx")
    assert np.allclose(w, ref_w, rtol=1e-5, atol=1e-7), float(np.abs(w - ref_w).max())
    check_gate_logits(logits, ref_logits, idx, bits(x), bits(wg), b, dtype,
                      gate_uses_tensor_cores(x.shape[0], x.shape[1], wg.shape[0]))
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


@pytest.mark.parametrize("T,d_h,E,k,dtype", [(1024, 7168, 256, 8, "bf16"),  # prefill width, one N tile
                                             (1100, 512, 100, 4, "f16"),    # ragged tokens and experts
                                             (1031, 768, 72, 8, "bf16"),
                                             (2048, 2048, 64, 6, "f16"),
                                             (1024, 256, 1000, 32, "f16"),  # four N tiles, k = 32
                                             (1200, 256, 8, 2, "bf16")])    # N tile mostly past E
def test_gate_tensor_core_path_shapes(oracle, T, d_h, E, k, dtype):
    """Many tokens: logits on the tensor cores, every expert that could be
    selected recomputed in the fixed order.  Ids bit for bit, weights within
    rtol 1e-5, selected logits bit for bit, the rest within the bound."""
    assert gate_uses_tensor_cores(T, d_h, E)
    dev = require_cuda()
    g = torch.Generator(device=dev).manual_seed(T + 3 * E)
    x = torch.randn((T, d_h), generator=g, device=dev).to(workloads.torch_dtype(dtype))
    wg = (torch.randn((E, d_h), generator=g, device=dev) / d_h ** 0.5).to(workloads.torch_dtype(dtype))
    rank = torch.randperm(E, generator=g, device=dev).to(torch.float64) + 1.0
    bias = (-1.1 * torch.log(rank)).to(torch.float32)
    _check_gate(oracle, x, wg, bias, k, dtype)


def test_gate_tensor_core_path_ties_and_near_ties(oracle):
    """Many tokens on the tensor-core path: (a) experts 3, 4, 5 share one row
    and a dominant bias, so their logits tie exactly and the order must be
    3, 4, 5 with equal weights; (b) expert 2j + 1 equals expert 2j but for one
    element one bf16 step away, so pairs of logits nearly tie and only the
    fixed-order recompute separates them; (c) zero tokens: every logit equals
    its bias, all experts tie, the first k ids win with weight 1/E."""
    dev = require_cuda()
    T, d_h, E = 1024, 1024, 64
    g = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn((T, d_h), generator=g, device=dev).to(torch.bfloat16)
    wg = (torch.randn((E, d_h), generator=g, device=dev) * 0.05).to(torch.bfloat16)
    wg[4] = wg[3]
    wg[5] = wg[3]
    bias = torch.zeros(E, device=dev)
    bias[3:6] = 100.0
    idx, w = _check_gate(oracle, x, wg.contiguous(), bias, 3, "bf16")
    assert (idx == np.array([3, 4, 5])).all()
    assert (w[:, 0] == w[:, 1]).all() and (w[:, 1] == w[:, 2]).all()

    wn = wg.clone()
    wn[1::2] = wn[0::2]
    j = torch.randint(0, d_h, (E // 2,), generator=g, device=dev)
    bumped = wn[1::2].view(torch.int16)
    rows = torch.arange(E // 2, device=dev)
    bumped[rows, j] = bumped[rows, j] + 1  # one step of the bf16 encoding
    _check_gate(oracle, x, wn.contiguous(), None, 8, "bf16")

    x0 = torch.zeros((T, d_h), dtype=torch.bfloat16, device=dev)
    idx, w = _check_gate(oracle, x0, wg.contiguous(), None, 6, "bf16")
    assert (idx == np.arange(6)).all()
    assert np.allclose(w, 1.0 / E, rtol=1e-6)


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


@pytest.mark.parametrize("T,k,E,d_h,dtype", [(4096, 8, 256, 7168, "bf16"),  # the prefill shape
                                             (301, 3, 17, 256, "f16"),
                                             (70, 32, 40, 512, "f32"),      # k at its limit
                                             (5, 1, 3, 64, "bf16"),
                                             (20000, 2, 9, 64, "bf16"),     # two tokens per warp, both buffers
                                             (3, 2, 4, 24576, "f32"),       # 96 KB rows: one warp per CTA
                                             (9, 2, 5, 26624, "f32")])      # 104 KB rows: the register form
def test_gather_rows_by_token_bit_exact(oracle, T, k, E, d_h, dtype):
    """The token-order gather moe_forward runs gives the row-order gather's
    rows bit for bit: against the oracle's gather with the same dispatch's
    sorted_token_idx; a position of -1 (a dropped pair) is skipped and a row
    no position names keeps its contents."""
    dev = require_cuda()
    rng = np.random.default_rng(T + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    tab = oracle.build_dispatch(idx, None, E, 128)
    td = workloads.torch_dtype(dtype)
    x = torch.randn((T, d_h), generator=torch.Generator().manual_seed(T), dtype=torch.float32).to(td).to(dev)
    pos = torch.from_numpy(tab["token_topk_to_pos"].reshape(T, k).copy()).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    a = binding.moe_gather_rows_by_token(x, pos, T * k, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.gather_rows(bits(x), tab["sorted_token_idx"], dtype)
    assert_bits_equal(bits(a), want, "rows gathered in token order")
    # drop one pair: its row is not written
    pos[T // 2, 0] = -1
    r_dropped = int(tab["token_topk_to_pos"].reshape(T, k)[T // 2, 0])
    a2 = torch.zeros_like(a)
    binding.moe_gather_rows_by_token(x, pos, T * k, out=a2)
    torch.cuda.synchronize()
    got = bits(a2)
    keep = np.arange(T * k) != r_dropped
    assert_bits_equal(got[keep], want[keep], "rows of the kept pairs")
    assert not got[r_dropped].any()


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
