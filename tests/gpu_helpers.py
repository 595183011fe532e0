"""Helpers shared by the GPU parity tests (not a test module)."""
import numpy as np
import pytest
import torch

from mixture_experts_routed_gate_gb300 import workloads

# fp16 MoE output tolerance (stated with the workloads), bf16 reading (the
# combine's bf16 figure from TileOPs-Metax PR #55, section 2), and the combine's
# own tolerances from the same section.
MOE_TOL = {"f16": (2e-2, 2e-3), "bf16": (1.6e-2, 1.6e-2)}
REDUCE_TOL = {"f16": (1e-3, 1e-3), "f32": (1e-3, 1e-3), "bf16": (1.6e-2, 1.6e-2), "e4m3": (0.1, 0.1)}


def require_cuda():
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but CUDA is not available")
    return torch.device("cuda:0")


def bits(t: torch.Tensor) -> np.ndarray:
    return workloads.to_numpy_bits(t)


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    from oracle import oracle
    return oracle.decode(a, dtype)


def assert_close(got_bits, want_bits, dtype: str, rtol: float, atol: float, what: str):
    got = as_f32(np.asarray(got_bits), dtype).astype(np.float64)
    want = as_f32(np.asarray(want_bits), dtype).astype(np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    bad = ~(np.abs(got - want) <= atol + rtol * np.abs(want))
    bad |= np.isnan(got) != np.isnan(want)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements outside rtol {rtol} atol {atol}; "
            f"first at {tuple(i)}: got {got[tuple(i)]} want {want[tuple(i)]}")


def assert_bits_equal(got, want, what: str):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if not np.array_equal(got, want):
        diff = np.argwhere(got != want)
        i = tuple(diff[0])
        raise AssertionError(f"{what}: {len(diff)} elements differ; first at {i}: "
                             f"got {got[i]} want {want[i]}")
