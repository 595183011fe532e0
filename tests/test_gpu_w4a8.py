"""The W4A8 GEMM (int4 weights x int8 activations, int32 sums) on the GPU vs
the oracle, bit for bit (TileLang tutorial ch.18 skeletons.py,
w4a8_dequant_gemm: the weight unpacked and sign-extended on chip, the
products summed in an int32 accumulator, the result written transposed).

Inputs are uniform int8 activations and uniform packed bytes (both nibbles
uniform over -8..7) in the pages' int4 layout, repacked on the device by
moe_pack_int4_weights; the oracle reads the pages' layout directly."""
import numpy as np
import pytest
import torch

from gpu_helpers import require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def _tables_to(dev, tab):
    return {n: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for n, v in tab.items()}


def _dense(dev, a, b, N):
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bp = binding.moe_pack_int4_weights(b.to(dev), 256)
    ct = binding.moe_gemm_w4a8(a.to(dev), bp, N, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ct.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(1, 3584, 18944),   # the pages' gemv-like serving shape
                                   (32, 3584, 18944),  # the pages' small-batch shape
                                   (1, 256, 64),       # one tile, one sub-step
                                   (5, 300, 1984),     # partial N tile, odd sub-step count (31)
                                   (64, 700, 4096),    # the most rows
                                   (17, 255, 16448)])  # K past one exact chunk
def test_gemm_w4a8_matches_oracle_bit_for_bit(oracle, M, N, K):
    dev = require_cuda()
    d = workloads.make_w4a8_inputs(M, N, K, seed=3)
    got = _dense(dev, d["a"], d["b"], N)
    want = oracle.gemm_w4a8(d["a"].numpy(), d["b"][0].numpy())
    assert got.shape == (N, M)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(3, 38912, 16384),  # one tile per SM: one K chunk of 16384, sums 2^24
                                   (2, 512, 18944),    # sums above 2^24: several chunks added as integers
                                   (1, 3584, 18944),
                                   (2, 256, 1 << 20)])  # the largest K: 64 chunks, sums up to 2^30
def test_gemm_w4a8_extremes_are_exact(M, N, K):
    """Rows of -128 and 127 against weight rows of -8, 7 and 0: every product
    at its extreme, Ct = K * a_m * b_n in closed form (up to 1024 K)."""
    dev = require_cuda()
    av = np.where(np.arange(M) % 2 == 0, -128, 127).astype(np.int64)
    bv = np.array([-8, 7, 0], np.int64)[np.arange(N) % 3]
    a = torch.from_numpy(np.repeat(av[:, None], K, axis=1).astype(np.int8))
    byte = np.array([0x88, 0x77, 0x00], np.uint8)[np.arange(N) % 3]
    b = torch.from_numpy(np.repeat(byte[:, None], K // 2, axis=1)[None])
    got = _dense(dev, a, b, N)
    assert np.array_equal(got, (K * np.outer(bv, av)).astype(np.int32))


def _routing(rng, T, k, E, skew):
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,k,E,N,K,skew", [(64, 6, 64, 2048, 768, False),   # decode stage-2 shape
                                            (64, 6, 64, 768, 2048, True),    # decode stage-1 shape, skewed
                                            (7, 2, 5, 300, 128, False),      # ragged N, empty experts
                                            (64, 8, 16, 256, 18944, False),  # K split into chunks
                                            (300, 4, 6, 512, 256, True)])     # 64-row units of larger blocks
def test_grouped_gemm_w4a8_matches_oracle(oracle, T, k, E, N, K, skew):
    """Rows gathered from x by sorted_token_idx, every routed row against the
    oracle's block walk over the same tables, bit for bit."""
    dev = require_cuda()
    rng = np.random.default_rng(T + E + N)
    idx = _routing(rng, T, k, E, skew)
    tab = oracle.build_dispatch(idx, None, E, 128)
    d = workloads.make_w4a8_inputs(T, N, K, seed=11, E=E)
    x, b = d["a"], d["b"]
    tabd = _tables_to(dev, tab)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bp = binding.moe_pack_int4_weights(b.to(dev), 256)
    c = binding.moe_grouped_gemm_w4a8(x.to(dev), tabd["sorted_token_idx"], bp, tabd, N, E, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = x.numpy()[tab["sorted_token_idx"]]
    want = oracle.grouped_gemm_w4a8(rows, b.numpy(), tab)
    assert np.array_equal(c.cpu().numpy(), want)


def test_grouped_gemm_w4a8_rows_in_place_and_bad_index(oracle):
    """Without sorted_token_idx the rows are x's own; an index outside [0, T)
    is reported (MOE_ERR_DEVICE_FLAG = 5) and its row summed from zeros."""
    dev = require_cuda()
    rng = np.random.default_rng(5)
    T, E, N, K = 40, 3, 512, 256
    idx = rng.integers(0, E, (T, 1)).astype(np.int32)
    tab = oracle.build_dispatch(idx, None, E, 128)
    d = workloads.make_w4a8_inputs(T, N, K, seed=12, E=E)
    rows = d["a"].numpy()[tab["sorted_token_idx"]]
    tabd = _tables_to(dev, tab)
    bp = binding.moe_pack_int4_weights(d["b"].to(dev), 256)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    c = binding.moe_grouped_gemm_w4a8(torch.from_numpy(rows).to(dev), None, bp, tabd, N, E, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.grouped_gemm_w4a8(rows, d["b"].numpy(), tab)
    assert np.array_equal(c.cpu().numpy(), want)
    bad = tabd["sorted_token_idx"].clone()
    bad[3] = T
    c2 = binding.moe_grouped_gemm_w4a8(d["a"].to(dev), bad, bp, tabd, N, E, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
    c2 = c2.cpu().numpy()
    assert (c2[3] == 0).all()
    keep = np.arange(T) != 3
    assert np.array_equal(c2[keep], want[keep])


def test_gemm_w4a8_argument_checks():
    dev = require_cuda()
    a = torch.zeros((65, 64), dtype=torch.int8, device=dev)
    bp = binding.moe_pack_int4_weights(torch.zeros((1, 256, 32), dtype=torch.uint8, device=dev), 256)
    with pytest.raises((ValueError, RuntimeError)):
        binding.moe_gemm_w4a8(a, bp, 256)  # M > 64
    with pytest.raises((ValueError, RuntimeError)):
        binding.moe_gemm_w4a8(torch.zeros((4, 96), dtype=torch.int8, device=dev), bp, 256)  # K % 64
    L = binding.lib()
    assert L.moe_gemm_w4a8_workspace_bytes(65, 64) == -1
    assert L.moe_gemm_w4a8_workspace_bytes(1, 100) == -1
    assert L.moe_gemm_w4a8_workspace_bytes(1, 64) > 0
