"""Algorithmic FLOP and byte counts of each step (host arithmetic only).

These are the numerators of the roofline fractions the benchmark reports:
achieved = algorithmic bytes (or FLOPs) of one launch / its measured duration.
"""
from __future__ import annotations

ELEM_BYTES = {"f16": 2, "bf16": 2, "f32": 4}


def reduce_bytes_pages(T: int, K: int, H: int, elem_bytes: int) -> int:
    """The combine's byte count as TileOPs-Metax PR #55 section 3 (Roofline)
    states it: every one of the T*K slot rows read, T rows written, plus the
    int32 positions and fp32 weights: (T*K*H + T*H)*e + T*K*4 + T*K*4."""
    return (T * K * H + T * H) * elem_bytes + T * K * 4 + T * K * 4


def reduce_bytes(n_valid: int, T: int, K: int, H: int, in_bytes: int, out_bytes: int,
                 weighted: bool = True) -> int:
    """Bytes the combine must move: only the n_valid non-padding rows are read."""
    return n_valid * H * in_bytes + T * H * out_bytes + T * K * 4 + (T * K * 4 if weighted else 0)


def reduce_flops(T: int, K: int, H: int) -> int:
    return 2 * T * K * H


def gate_up_flops(n_rows: int, d_h: int, d_e: int) -> int:
    """Stage 1: two GEMMs [n_rows, d_h] x [d_h, d_e]."""
    return 2 * n_rows * d_h * (2 * d_e)


def down_flops(n_rows: int, d_h: int, d_e: int) -> int:
    return 2 * n_rows * d_e * d_h


def gate_up_bytes(n_rows: int, d_h: int, d_e: int, active_experts: int, e: int) -> int:
    """Stage 1 minimum traffic: W_gate and W_up of every expert that owns a row,
    the gathered activations once, h written once."""
    return 2 * active_experts * d_e * d_h * e + n_rows * d_h * e + n_rows * d_e * e


def down_bytes(n_rows: int, d_h: int, d_e: int, active_experts: int, e: int) -> int:
    return active_experts * d_h * d_e * e + n_rows * d_e * e + n_rows * d_h * e


def expert_mlp_bytes(n_rows: int, d_h: int, d_e: int, active_experts: int, e: int) -> int:
    """Both stages in one launch: the three weight matrices of every active
    expert, the gathered rows read, h written and read back, y written."""
    return gate_up_bytes(n_rows, d_h, d_e, active_experts, e) + down_bytes(n_rows, d_h, d_e, active_experts, e)


def expert_mlp_flops(n_rows: int, d_h: int, d_e: int) -> int:
    return gate_up_flops(n_rows, d_h, d_e) + down_flops(n_rows, d_h, d_e)


def gate_flops(T: int, d_h: int, E: int) -> int:
    return 2 * T * E * d_h


def moe_forward_flops(T: int, k: int, d_h: int, d_e: int, E: int) -> int:
    Tk = T * k
    return gate_flops(T, d_h, E) + gate_up_flops(Tk, d_h, d_e) + down_flops(Tk, d_h, d_e) \
        + reduce_flops(T, k, d_h)


def moe_forward_bytes_min(T: int, d_h: int, d_e: int, E: int, active_experts: int, e: int) -> int:
    """Least traffic of the whole forward: the three weight matrices of every
    active expert, the gate weight, x read and out written once."""
    return 3 * active_experts * d_e * d_h * e + E * d_h * e + 2 * T * d_h * e
