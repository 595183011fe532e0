"""The C-ABI library loads and exports every entry point the public header
declares; host-side sizing and argument checks work without a GPU (none of
these calls reaches a kernel)."""
import ctypes
import os
import re

import pytest

from mixture_experts_routed_gate_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_routed_gate.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API[^;(]*?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for required in ("moe_gate_topk", "moe_build_dispatch", "moe_grouped_gate_up_silu",
                     "moe_grouped_down", "moe_reduce_fused", "moe_forward"):
        assert required in names
    assert sorted(binding.exported_symbols()) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_sizing_helpers(lib, oracle):
    for T, k, E in [(64, 2, 8), (64, 6, 64), (4096, 8, 256), (0, 2, 8), (1, 1, 1)]:
        assert lib.moe_num_m_blocks(T, k, E, 128) == oracle.num_m_blocks(T, k, E, 128)
    assert lib.moe_num_m_blocks(4096, 8, 256, 128) == 512
    assert lib.moe_num_m_blocks(-1, 2, 8, 128) == -1
    assert lib.moe_gate_topk_workspace_bytes(64, 8) == 64 * 8 * 4
    ws = lib.moe_forward_workspace_bytes(4096, 7168, 2048, 256, 8, 1)
    # the gathered rows, h and y dominate: Tk*(2*d_h + d_e)*2 bytes
    assert ws >= 32768 * (2 * 7168 + 2048) * 2
    assert ws % 256 == 0
    offs = [lib.moe_forward_workspace_offset(4096, 7168, 2048, 256, 8, 1, i) for i in range(15)]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    # the last section holds one int32 counter per M block
    assert ws - offs[14] >= 512 * 4
    assert lib.moe_forward_workspace_offset(4096, 7168, 2048, 256, 8, 1, 15) == -1


def test_status_strings(lib):
    for s in range(7):
        assert lib.moe_status_string(s).startswith(b"MOE_")
    assert lib.moe_status_string(99) == b"unknown moe status"


def test_argument_errors_without_launch(lib):
    """The pages' error cases (hidden % 256 != 0 for the combine) and others are
    rejected on the host, before any CUDA call."""
    P = ctypes.c_void_p
    fake = P(0x1000)
    # reduce: H % 256 != 0
    assert lib.moe_reduce_fused(fake, 8, fake, None, 4, 2, 200, 1, 1, fake, None, None) == MOE_ERR_INVALID_ARG
    # reduce: unsupported dtype pair (bf16 in, f32 out)
    assert lib.moe_reduce_fused(fake, 8, fake, None, 4, 2, 256, 1, 2, fake, None, None) == MOE_ERR_UNSUPPORTED
    # reduce: null output
    assert lib.moe_reduce_fused(fake, 8, fake, None, 4, 2, 256, 1, 1, None, None, None) == MOE_ERR_INVALID_ARG
    # gate: d_hidden % 256 != 0, k > E, f32 activations
    assert lib.moe_gate_topk(fake, fake, None, 4, 200, 8, 2, 1, fake, fake, fake, 1 << 20, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_gate_topk(fake, fake, None, 4, 256, 8, 9, 1, fake, fake, fake, 1 << 20, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_gate_topk(fake, fake, None, 4, 256, 8, 2, 2, fake, fake, fake, 1 << 20, None) == MOE_ERR_UNSUPPORTED
    # gate: workspace too small
    assert lib.moe_gate_topk(fake, fake, None, 4, 256, 8, 2, 1, fake, fake, fake, 16, None) == MOE_ERR_WORKSPACE
    # dispatch: block_m other than 128, workspace too small
    assert lib.moe_build_dispatch(fake, None, 4, 2, 8, 64, fake, fake, fake, fake, fake, fake, fake,
                                  fake, 1 << 20, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_build_dispatch(fake, None, 4, 2, 8, 128, fake, fake, fake, fake, fake, fake, fake,
                                  fake, 0, None) == MOE_ERR_WORKSPACE
    # grouped GEMMs: misaligned d_expert, m_blocks larger than the table space
    assert lib.moe_grouped_gate_up_silu(fake, fake, fake, fake, fake, fake, fake, 3, 8, 256, 100, 8, 1,
                                        fake, None, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_down(fake, fake, fake, fake, fake, fake, 99, None, 8, 256, 128, 8, 1,
                                fake, None, None) == MOE_ERR_INVALID_ARG
    # expert MLP in one launch: no counter buffer, misaligned d_expert
    assert lib.moe_grouped_mlp(fake, fake, fake, fake, fake, fake, fake, fake, 3, None, 8, 256, 128, 8, 1,
                               fake, fake, None, None, None, 0, None, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp(fake, fake, fake, fake, fake, fake, fake, fake, 3, None, 8, 256, 100, 8, 1,
                               fake, fake, fake, None, None, 0, None, None) == MOE_ERR_INVALID_ARG
    # gathering form: no token rows, more rows than int32 indices reach, or no tokens given
    assert lib.moe_grouped_mlp(None, fake, fake, fake, fake, fake, fake, fake, 3, None, 8, 256, 128, 8, 1,
                               fake, fake, fake, fake, fake, 0, None, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp(None, fake, fake, fake, fake, fake, fake, fake, 3, None, 8, 256, 128, 8, 1,
                               fake, fake, fake, fake, fake, 1 << 31, None, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_mlp(None, fake, fake, fake, fake, fake, fake, fake, 3, None, 8, 256, 128, 8, 1,
                               fake, fake, fake, None, fake, 8, None, None) == MOE_ERR_INVALID_ARG
    # forward: workspace too small, misaligned workspace
    assert lib.moe_forward(fake, fake, None, fake, fake, fake, 64, 256, 128, 8, 2, 0, P(0x100000), 16,
                           fake, None, None) == MOE_ERR_WORKSPACE
    assert lib.moe_forward(fake, fake, None, fake, fake, fake, 64, 256, 128, 8, 2, 0, P(0x100010),
                           1 << 30, fake, None, None) == MOE_ERR_INVALID_ARG
    # empty problems are valid no-ops
    assert lib.moe_reduce_fused(fake, 0, fake, None, 0, 2, 256, 1, 1, fake, None, None) == MOE_OK
    assert lib.moe_gather_rows(fake, fake, 0, 4, 256, 1, fake, None) == MOE_OK
    assert lib.moe_copy(fake, P(0x200000), 0, None) == MOE_OK
    # copy: size not a 16-byte multiple, misaligned, overlapping ranges
    assert lib.moe_copy(fake, P(0x200000), 24, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_copy(P(0x100008), P(0x200000), 32, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_copy(P(0x100000), P(0x100010), 64, None) == MOE_ERR_INVALID_ARG
    # bounded flag wait: no flag, no error word, timeout out of range
    assert lib.moe_wait_flag(None, 1, 1000, fake, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_wait_flag(fake, 1, 1000, None, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_wait_flag(fake, 1, 0, fake, None) == MOE_ERR_INVALID_ARG
    assert lib.moe_wait_flag(fake, 1, 10_000_000_001, fake, None) == MOE_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def test_header_is_plain_c_and_links(tmp_path):
    """A C11 program that includes only the header and the CUDA runtime
    compiles (-Wall -Werror) and links against the library."""
    import c_caller
    exe = c_caller.build(str(tmp_path))
    assert os.path.exists(exe)


@pytest.mark.parametrize("T,d_h,d_e,E,k", [(1, 256, 64, 1, 1), (64, 2048, 768, 64, 6), (65, 256, 192, 8, 2),
                                           (4096, 7168, 2048, 256, 8), (300, 512, 320, 1000, 32)])
def test_forward_workspace_sections_are_disjoint(lib, T, d_h, d_e, E, k):
    """Every intermediate of moe_forward gets its own 256-byte aligned range
    inside the workspace, large enough for its shape (checked on a host
    buffer: only the library's sizing functions run)."""
    import torch
    for dtype in (torch.float16, torch.bfloat16):
        need = binding.forward_workspace_bytes(T, d_h, d_e, E, k, dtype)
        ws = torch.empty(need, dtype=torch.uint8)
        views = binding.forward_workspace_views(ws, T, d_h, d_e, E, k, dtype)
        base = ws.data_ptr()
        ranges = []
        for name, v in views.items():
            lo = v.data_ptr() - base
            hi = lo + v.numel() * v.element_size()
            assert lo % 256 == 0, name
            assert 0 <= lo and hi <= need, (name, lo, hi, need)
            ranges.append((lo, hi, name))
        ranges.sort()
        for (lo0, hi0, n0), (lo1, hi1, n1) in zip(ranges, ranges[1:]):
            assert hi0 <= lo1, f"{n0} [{lo0}, {hi0}) overlaps {n1} [{lo1}, {hi1})"
        # the dispatch scratch sits between token_topk_to_pos and the rows A
        off = [lib.moe_forward_workspace_offset(T, d_h, d_e, E, k, 0 if dtype == torch.float16 else 1, i)
               for i in range(15)]
        scratch = lib.moe_build_dispatch_workspace_bytes(T, k, E)
        assert off[11] - off[10] >= scratch
