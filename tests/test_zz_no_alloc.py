"""moe_build_dispatch_noalloc: the dispatch entry point for callers that may
not allocate device memory (code inside a CUDA graph capture, engines whose
memory is planned up front).  Its scratch is a fixed array inside the
library; its tables must equal those of moe_build_dispatch, which takes a
caller-provided workspace.  Collected last on purpose."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bits_equal, require_cuda
from mixture_experts_routed_gate_gb300 import binding

pytestmark = pytest.mark.gpu


def _routing(seed, T, k, E, dev):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    """Two calls in a row, through the C-ABI, each compared table by table
    (bit for bit, the tolerance the dispatch tests use) with the workspace
    entry point.  Both calls take the multi-kernel path that uses the fixed
    scratch (32768 pairs; then 300 experts, more than the one-CTA path
    handles) with a different size and routing, so stale counters left by
    the first call would show."""
    dev = require_cuda()
    for seed, (T, k, E) in enumerate([(4096, 8, 256), (300, 6, 300)]):
        idx, w = _routing(seed, T, k, E, dev)
        want = binding.moe_build_dispatch(idx, w, E)
        got = binding.moe_build_dispatch_noalloc(idx, w, E)
        torch.cuda.synchronize()
        for name in want:
            a, b = got[name].cpu().numpy(), want[name].cpu().numpy()
            if a.dtype == np.float32:
                a, b = a.view(np.uint32), b.view(np.uint32)
            assert_bits_equal(a, b, f"call {seed + 1}: {name}")


def test_noalloc_dispatch_rejects_problems_beyond_its_scratch():
    """ceil(T*k / 2048) * E must stay within the 262,144 fixed counters."""
    dev = require_cuda()
    T, k, E = 75000, 8, 1024  # 293 chunks x 1024 experts > 262144
    idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
    with pytest.raises(binding.MoEError, match="WORKSPACE"):
        binding.moe_build_dispatch_noalloc(idx, None, E)
