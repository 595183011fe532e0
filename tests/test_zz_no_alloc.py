"""moe_build_dispatch_noalloc: the dispatch entry point for callers that may
not allocate device memory (code inside a CUDA graph capture, engines whose
memory is planned up front).  Its scratch is a fixed array inside the
library; its tables must equal those of moe_build_dispatch, which takes a
caller-provided workspace, and those of the oracle.  Collected last on
purpose."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, require_cuda
from mixture_experts_routed_gate_gb300 import binding

pytestmark = pytest.mark.gpu

# counters in the library's fixed scratch array (1 MiB of int32)
SCRATCH_COUNTERS = 262144
CHUNK = 2048  # token-expert pairs per histogram chunk


def _routing(seed, T, k, E, dev, distinct=True):
    """Zipf-skewed expert ids (distinct per token, like a top-k, or drawn with
    replacement for very large cases) and random fp32 weights."""
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    if distinct:
        idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    else:
        idx = rng.choice(E, size=(T, k), p=p)
    idx = idx.astype(np.int32).reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    return torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)


def _as_bits(a):
    a = np.asarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _assert_tables_equal(got, want, what):
    for name in want:
        g = got[name].cpu().numpy() if torch.is_tensor(got[name]) else got[name]
        w = want[name].cpu().numpy() if torch.is_tensor(want[name]) else want[name]
        assert_bits_equal(_as_bits(g).reshape(np.shape(w)), _as_bits(w), f"{what}: {name}")


def test_noalloc_dispatch_matches_workspace_dispatch_and_oracle_twice(oracle):
    """Two calls in a row, through the C-ABI, each compared table by table,
    bit for bit, with the workspace entry point and with the oracle.  Both
    calls take the multi-kernel path that uses the fixed scratch (32768
    pairs; then 300 experts, more than the one-CTA path handles) with a
    different size and routing, so stale counters left by the first call
    would show."""
    dev = require_cuda()
    for seed, (T, k, E) in enumerate([(4096, 8, 256), (300, 6, 300)]):
        idx, w = _routing(seed, T, k, E, dev)
        want = binding.moe_build_dispatch(idx, w, E)
        got = binding.moe_build_dispatch_noalloc(idx, w, E)
        torch.cuda.synchronize()
        _assert_tables_equal(got, want, f"call {seed + 1} vs workspace entry")
        ref = oracle.build_dispatch(idx.cpu().numpy(), w.cpu().numpy(), E, 128)
        _assert_tables_equal(got, ref, f"call {seed + 1} vs oracle")


def test_noalloc_dispatch_at_the_exact_scratch_limit(oracle):
    """ceil(T*k / 2048) * E == 262144 exactly (1024 experts, 524288 pairs):
    accepted, and the last counter of the array is used; the tables equal
    the workspace entry point's and the oracle's bit for bit."""
    dev = require_cuda()
    T, k, E = 65536, 8, 1024
    assert -(-T * k // CHUNK) * E == SCRATCH_COUNTERS
    idx, w = _routing(11, T, k, E, dev, distinct=False)
    got = binding.moe_build_dispatch_noalloc(idx, w, E)
    want = binding.moe_build_dispatch(idx, w, E)
    torch.cuda.synchronize()
    _assert_tables_equal(got, want, "limit vs workspace entry")
    ref = oracle.build_dispatch(idx.cpu().numpy(), w.cpu().numpy(), E, 128)
    _assert_tables_equal(got, ref, "limit vs oracle")


def test_noalloc_dispatch_rejects_problems_beyond_its_scratch():
    """One chunk past the limit (65537 tokens x 8 = 257 chunks of 1024
    counters) and a clearly oversized problem both return MOE_ERR_WORKSPACE
    without launching."""
    dev = require_cuda()
    for T, k, E in [(65537, 8, 1024), (75000, 8, 1024)]:
        assert -(-T * k // CHUNK) * E > SCRATCH_COUNTERS
        idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
        with pytest.raises(binding.MoEError, match="WORKSPACE"):
            binding.moe_build_dispatch_noalloc(idx, None, E)


def test_noalloc_dispatch_with_no_tokens_and_many_experts(oracle):
    """T = 0 with 300 experts (the table kernel still runs: every expert
    empty, each owning its one padding block), against the oracle."""
    dev = require_cuda()
    T, k, E = 0, 4, 300
    idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
    got = binding.moe_build_dispatch_noalloc(idx, None, E)
    torch.cuda.synchronize()
    ref = oracle.build_dispatch(np.zeros((T, k), np.int32), None, E, 128)
    _assert_tables_equal(got, ref, "T = 0")
    assert (got["group_sizes"].cpu().numpy() == 0).all()
