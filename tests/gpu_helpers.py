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


def gate_uses_tensor_cores(T: int, d_h: int, E: int) -> bool:
    """Whether moe_gate_topk takes the tensor-core path for this shape (many
    tokens; the select kernel's per-warp shared memory within its limit)."""
    return T >= 1024 and d_h % 64 == 0 and E <= 1024 and d_h * 2 + E * 12 + 32 <= 200 * 1024


def gate_tc_bound(x_bits, wg_bits, bias, ref_logits, dtype: str) -> np.ndarray:
    """The tensor-core gate's bound on |logit~ - logit| per (token, expert),
    restated from its error model: 2 (18 G 2^-23 + (d_h/32 + 6) 2^-24 +
    (S + 2) 2^-24) (1 + 2^-9)^2 (|x_t| |w_e| + |bias_e|) + 2^-22 |logit|, with
    G = 4 K steps per split and S splits as the launch chooses them (the
    logit's magnitude taken from the fixed-order value, doubled)."""
    from oracle import oracle
    xf = oracle.decode(x_bits, dtype).astype(np.float64)
    wf = oracle.decode(wg_bits, dtype).astype(np.float64)
    T, d_h = xf.shape
    E = wf.shape[0]
    nk = d_h // 64
    tiles = -(-T // 128) * -(-E // 256)
    S = max(1, min(8, 128 // tiles))
    S = min(S, nk)
    ks = -(-nk // S)
    S = -(-nk // ks)
    u = 2.0 ** -24
    coef = 2 * (18 * 4 * ks * 2 * u + (d_h / 32 + 6) * u + (S + 2) * u) * (1 + 2.0 ** -9) ** 2
    b = np.zeros(E) if bias is None else np.abs(np.asarray(bias, np.float64))
    mag = np.linalg.norm(xf, axis=1)[:, None] * np.linalg.norm(wf, axis=1)[None, :] + b[None, :]
    return coef * mag + 2.0 ** -21 * np.abs(ref_logits.astype(np.float64))


def check_gate_logits(logits, ref_logits, idx, x_bits, wg_bits, bias, dtype: str, tensor_cores: bool):
    """Logits of the fixed summation order are compared bit for bit.  On the
    tensor-core path only the experts the kernel recomputed in that order
    carry those bits: the selected ones always (checked bit for bit), the
    others either carry them too or lie within the path's bound (checked)."""
    if not tensor_cores:
        assert_bits_equal(logits.view(np.uint32), ref_logits.view(np.uint32), "gate logits")
        return
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    sel_ref = np.take_along_axis(ref_logits, idx.astype(np.int64), axis=1)
    assert_bits_equal(sel.view(np.uint32), sel_ref.view(np.uint32), "logits of the selected experts")
    bound = gate_tc_bound(x_bits, wg_bits, bias, ref_logits, dtype)
    diff = np.abs(logits.astype(np.float64) - ref_logits.astype(np.float64))
    bad = diff > bound
    assert not bad.any(), (f"{int(bad.sum())} logits outside the tensor-core bound; worst "
                           f"{float((diff / bound).max())} of it")
    # the bound is loose by design; the real differences sit far inside it
    ratio = np.where(bound > 0, diff / np.where(bound > 0, bound, 1.0), 0.0)
    assert float(ratio.max()) < 0.25, float(ratio.max())
