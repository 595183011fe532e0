"""Thin Python binding of ``libmoe_routed_gb300.so`` (argument marshalling only).

Every function here has the name of the C-ABI entry point it calls, takes
CUDA tensors, checks their dtype/shape/contiguity, and passes raw pointers and
``torch.cuda.current_stream()`` to the library.  All computation happens in
the library's kernels; there is no fallback: if the library is missing or a
call fails, a ``MoEError`` is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.float8_e4m3fn: 3}
_DT_NAME = {0: "f16", 1: "bf16", 2: "f32", 3: "e4m3"}
_lib = None

BLOCK_M = 128
WS_NAMES = ["logits", "topk_idx", "topk_w", "group_sizes", "group_offsets",
            "group_padded_offsets", "group_idx_for_bx", "sorted_token_idx", "sorted_row_weight",
            "token_topk_to_pos", "dispatch_scratch", "a", "h", "y", "mlp_ready"]


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = lib().moe_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the CUDA library (build it first with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P, I64, SZ, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    sigs = {
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_num_m_blocks": (I64, [I64, I64, I64, I64]),
        "moe_gate_topk_workspace_bytes": (SZ, [I64, I64]),
        "moe_build_dispatch_workspace_bytes": (SZ, [I64, I64, I64]),
        "moe_forward_workspace_bytes": (SZ, [I64, I64, I64, I64, I64, I]),
        "moe_forward_workspace_offset": (I64, [I64, I64, I64, I64, I64, I, I]),
        "moe_gate_topk": (I, [P, P, P, I64, I64, I64, I64, I, P, P, P, SZ, P]),
        "moe_build_dispatch": (I, [P, P, I64, I64, I64, I64, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_build_dispatch_noalloc": (I, [P, P, I64, I64, I64, I64, P, P, P, P, P, P, P, P]),
        "moe_copy": (I, [P, P, I64, P]),
        "moe_wait_flag": (I, [P, ctypes.c_int32, I64, P, P]),
        "moe_gather_rows": (I, [P, P, I64, I64, I64, I, P, P]),
        "moe_gather_rows_by_token": (I, [P, P, I64, I64, I64, I64, I, P, P, P]),
        "moe_grouped_gate_up_silu": (I, [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I, P, P, P]),
        "moe_grouped_down": (I, [P, P, P, P, P, P, I64, P, I64, I64, I64, I64, I, P, P, P]),
        "moe_grouped_mlp": (I, [P, P, P, P, P, P, P, P, I64, P, I64, I64, I64, I64, I, P, P, P, P, P, I64, P, P]),
        "moe_reduce_fused": (I, [P, I64, P, P, I64, I64, I64, I, I, P, P, P]),
        "moe_reduce_fused_scaled": (I, [P, I64, P, P, P, P, I64, I64, I64, I, I, P, P, P]),
        "moe_forward": (I, [P, P, P, P, P, P, I64, I64, I64, I64, I64, I, P, SZ, P, P, P]),
        "moe_pack_int4_bytes": (I64, [I64, I64, I64, I64]),
        "moe_pack_int4_weights": (I, [P, I64, I64, I64, I64, P, P]),
        "moe_grouped_mlp_w4a16": (I, [P, P, I64, P, P, P, P, P, P, P, P, P, P, I64, P, I64, I64, I64, I64, I,
                                      P, P, P, P, P]),
        "moe_forward_w4a16": (I, [P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I, P, SZ, P, P, P]),
        "moe_gemm_w4a8_workspace_bytes": (I64, [I64, I64]),
        "moe_gemm_w4a8": (I, [P, P, I64, I64, I64, P, P, I64, P, P]),
        "moe_grouped_gemm_w4a8_workspace_bytes": (I64, [I64, I64, I64]),
        "moe_grouped_gemm_w4a8": (I, [P, P, I64, P, P, P, P, P, I64, I64, I64, I64, I64, P, P, I64, P, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def exported_symbols():
    return ["moe_status_string", "moe_num_m_blocks", "moe_gate_topk_workspace_bytes",
            "moe_build_dispatch_workspace_bytes", "moe_forward_workspace_bytes",
            "moe_forward_workspace_offset", "moe_gate_topk", "moe_build_dispatch",
            "moe_build_dispatch_noalloc",
            "moe_copy", "moe_wait_flag", "moe_gather_rows", "moe_gather_rows_by_token",
            "moe_grouped_gate_up_silu", "moe_grouped_down",
            "moe_grouped_mlp", "moe_pack_int4_bytes", "moe_pack_int4_weights", "moe_grouped_mlp_w4a16",
            "moe_forward_w4a16", "moe_gemm_w4a8_workspace_bytes", "moe_gemm_w4a8",
            "moe_grouped_gemm_w4a8_workspace_bytes", "moe_grouped_gemm_w4a8", "moe_reduce_fused",
            "moe_reduce_fused_scaled", "moe_forward"]


# --------------------------------------------------------------------------- helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _cuda(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _cuda_or_pinned(t, name, dtype=None):
    """A CUDA tensor, or a pinned host tensor: with unified addressing its
    address is valid on the device, which stores to it directly."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        return t
    return _cuda(t, name, dtype=dtype)


def _dtype_code(t, name):
    if t.dtype not in _DT:
        raise TypeError(f"{name}: unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _check(status, what):
    if status != 0:
        raise MoEError(status, what)


def num_m_blocks(T: int, k: int, E: int, block_m: int = BLOCK_M) -> int:
    return int(lib().moe_num_m_blocks(T, k, E, block_m))


moe_num_m_blocks = num_m_blocks


# --------------------------------------------------------------------------- entry points

def moe_gate_topk(x, w_g, bias, k: int, topk_idx=None, topk_w=None, ws=None):
    """Routing: returns (topk_idx [T,k] int32, topk_w [T,k] fp32)."""
    _cuda(x, "x", ndim=2)
    _cuda(w_g, "w_g", dtype=x.dtype, ndim=2)
    T, d_h = x.shape
    E = w_g.shape[0]
    if w_g.shape[1] != d_h:
        raise ValueError("w_g must be [E, d_hidden]")
    if bias is not None:
        _cuda(bias, "bias", dtype=torch.float32, ndim=1)
        if bias.numel() != E:
            raise ValueError("bias must be [E]")
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    _cuda(topk_idx, "topk_idx", dtype=torch.int32)
    _cuda(topk_w, "topk_w", dtype=torch.float32)
    need = lib().moe_gate_topk_workspace_bytes(T, E)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().moe_gate_topk(_ptr(x), _ptr(w_g), _ptr(bias), T, d_h, E, k,
                                   _dtype_code(x, "x"), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(dev)), "moe_gate_topk")
    return topk_idx, topk_w


def moe_build_dispatch(topk_idx, topk_w, E: int, block_m: int = BLOCK_M, out=None, ws=None):
    """Dispatch tables: returns a dict of device tensors (names as in the C-ABI)."""
    _cuda(topk_idx, "topk_idx", dtype=torch.int32, ndim=2)
    T, k = topk_idx.shape
    if topk_w is not None:
        _cuda(topk_w, "topk_w", dtype=torch.float32)
        if topk_w.shape != topk_idx.shape:
            raise ValueError("topk_w must match topk_idx")
    dev = topk_idx.device
    mb = num_m_blocks(T, k, E, block_m)
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = dict(group_sizes=torch.empty(E, **i32), group_offsets=torch.empty(E, **i32),
                   group_padded_offsets=torch.empty(E, **i32),
                   group_idx_for_bx=torch.empty(max(mb, 0), **i32),
                   sorted_token_idx=torch.empty(T * k, **i32),
                   sorted_row_weight=torch.empty(T * k, dtype=torch.float32, device=dev),
                   token_topk_to_pos=torch.empty((T, k), **i32))
    need = lib().moe_build_dispatch_workspace_bytes(T, k, E)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().moe_build_dispatch(
            _ptr(topk_idx), _ptr(topk_w), T, k, E, block_m, _ptr(out["group_sizes"]),
            _ptr(out["group_offsets"]), _ptr(out["group_padded_offsets"]),
            _ptr(out["group_idx_for_bx"]), _ptr(out["sorted_token_idx"]),
            _ptr(out["sorted_row_weight"]), _ptr(out["token_topk_to_pos"]), _ptr(ws),
            ws.numel() * ws.element_size(), _stream(dev)), "moe_build_dispatch")
    return out


def _dispatch_outputs(T, k, E, block_m, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    mb = num_m_blocks(T, k, E, block_m)
    return dict(group_sizes=torch.empty(E, **i32), group_offsets=torch.empty(E, **i32),
                group_padded_offsets=torch.empty(E, **i32),
                group_idx_for_bx=torch.empty(max(mb, 0), **i32),
                sorted_token_idx=torch.empty(T * k, **i32),
                sorted_row_weight=torch.empty(T * k, dtype=torch.float32, device=dev),
                token_topk_to_pos=torch.empty((T, k), **i32))


def moe_build_dispatch_noalloc(topk_idx, topk_w, E: int, block_m: int = BLOCK_M, out=None):
    """moe_build_dispatch with the library's fixed scratch array instead of a
    workspace (for callers that may not allocate device memory).  The output
    tables are still the caller's: pass preallocated ones in ``out`` to make
    the call itself allocation-free."""
    _cuda(topk_idx, "topk_idx", dtype=torch.int32, ndim=2)
    T, k = topk_idx.shape
    if topk_w is not None:
        _cuda(topk_w, "topk_w", dtype=torch.float32)
        if topk_w.shape != topk_idx.shape:
            raise ValueError("topk_w must match topk_idx")
    dev = topk_idx.device
    if out is None:
        out = _dispatch_outputs(T, k, E, block_m, dev)
    with torch.cuda.device(dev):
        _check(lib().moe_build_dispatch_noalloc(
            _ptr(topk_idx), _ptr(topk_w), T, k, E, block_m, _ptr(out["group_sizes"]),
            _ptr(out["group_offsets"]), _ptr(out["group_padded_offsets"]),
            _ptr(out["group_idx_for_bx"]), _ptr(out["sorted_token_idx"]),
            _ptr(out["sorted_row_weight"]), _ptr(out["token_topk_to_pos"]), _stream(dev)),
            "moe_build_dispatch_noalloc")
    return out


def moe_copy(src, dst):
    """dst[:] = src by a kernel on dst's device stream; either may be a pinned
    host tensor (same number of bytes, 16-byte multiple)."""
    dev_t = dst if dst.is_cuda else src
    if not dev_t.is_cuda:
        raise ValueError("moe_copy: one side must be a CUDA tensor")
    _cuda_or_pinned(src, "src")
    _cuda_or_pinned(dst, "dst")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("moe_copy: src and dst sizes differ")
    with torch.cuda.device(dev_t.device):
        _check(lib().moe_copy(_ptr(src), _ptr(dst), nbytes, _stream(dev_t.device)), "moe_copy")
    return dst


def moe_wait_flag(flag, expected: int, timeout_s: float, err, device=None):
    """Stream-ordered bounded wait until flag[0] >= expected (flag: int32 CUDA
    tensor or pinned host tensor); on a timeout err[0] becomes MOE_ERR_TIMEOUT."""
    _cuda_or_pinned(flag, "flag", dtype=torch.int32)
    _cuda(err, "err", dtype=torch.int32)
    dev = err.device if device is None else device
    with torch.cuda.device(dev):
        _check(lib().moe_wait_flag(_ptr(flag), int(expected), int(timeout_s * 1e9), _ptr(err), _stream(dev)),
               "moe_wait_flag")


def moe_gather_rows(x, sorted_token_idx, out=None):
    _cuda(x, "x", ndim=2)
    _cuda(sorted_token_idx, "sorted_token_idx", dtype=torch.int32)
    T, d_h = x.shape
    n = sorted_token_idx.numel()
    if out is None:
        out = torch.empty((n, d_h), dtype=x.dtype, device=x.device)
    _cuda(out, "out", dtype=x.dtype)
    with torch.cuda.device(x.device):
        _check(lib().moe_gather_rows(_ptr(x), _ptr(sorted_token_idx), n, T, d_h,
                                     _dtype_code(x, "x"), _ptr(out), _stream(x.device)),
               "moe_gather_rows")
    return out


def moe_gather_rows_by_token(x, token_topk_to_pos, n_rows: int, out=None, err=None):
    """The gather in token order: out[token_topk_to_pos[t, j]] = x[t] (positions
    outside [0, n_rows) skipped); with a dispatch's positions, moe_gather_rows'
    result."""
    _cuda(x, "x", ndim=2)
    _cuda(token_topk_to_pos, "token_topk_to_pos", dtype=torch.int32, ndim=2)
    T, d_h = x.shape
    k = token_topk_to_pos.shape[1]
    if token_topk_to_pos.shape[0] != T:
        raise ValueError("token_topk_to_pos must be [T, k]")
    if out is None:
        out = torch.empty((n_rows, d_h), dtype=x.dtype, device=x.device)
    _cuda(out, "out", dtype=x.dtype)
    with torch.cuda.device(x.device):
        _check(lib().moe_gather_rows_by_token(_ptr(x), _ptr(token_topk_to_pos), T, k, n_rows, d_h,
                                              _dtype_code(x, "x"), _ptr(out), _ptr(err), _stream(x.device)),
               "moe_gather_rows_by_token")
    return out


def _tables(t):
    names = ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx")
    for n in names:
        _cuda(t[n], n, dtype=torch.int32)
    return [t[n] for n in names]


def moe_grouped_gate_up_silu(a, w_gate, w_up, tables, h=None, err=None):
    _cuda(a, "a", ndim=2)
    _cuda(w_gate, "w_gate", dtype=a.dtype, ndim=3)
    _cuda(w_up, "w_up", dtype=a.dtype, ndim=3)
    n_rows, d_h = a.shape
    E, d_e, d_h2 = w_gate.shape
    if d_h2 != d_h or w_up.shape != w_gate.shape:
        raise ValueError("w_gate / w_up must be [E, d_expert, d_hidden]")
    s, o, p, g = _tables(tables)
    if h is None:
        h = torch.empty((n_rows, d_e), dtype=a.dtype, device=a.device)
    _cuda(h, "h", dtype=a.dtype)
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(a.device):
        _check(lib().moe_grouped_gate_up_silu(
            _ptr(a), _ptr(w_gate), _ptr(w_up), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.numel(),
            n_rows, d_h, d_e, E, _dtype_code(a, "a"), _ptr(h), _ptr(err), _stream(a.device)),
            "moe_grouped_gate_up_silu")
    return h


def moe_grouped_down(h, w_down, tables, row_weights=None, y=None, err=None):
    _cuda(h, "h", ndim=2)
    _cuda(w_down, "w_down", dtype=h.dtype, ndim=3)
    n_rows, d_e = h.shape
    E, d_h, d_e2 = w_down.shape
    if d_e2 != d_e:
        raise ValueError("w_down must be [E, d_hidden, d_expert]")
    s, o, p, g = _tables(tables)
    if row_weights is not None:
        _cuda(row_weights, "row_weights", dtype=torch.float32)
    if y is None:
        y = torch.empty((n_rows, d_h), dtype=h.dtype, device=h.device)
    _cuda(y, "y", dtype=h.dtype)
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(h.device):
        _check(lib().moe_grouped_down(
            _ptr(h), _ptr(w_down), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.numel(),
            _ptr(row_weights), n_rows, d_h, d_e, E, _dtype_code(h, "h"), _ptr(y), _ptr(err),
            _stream(h.device)), "moe_grouped_down")
    return y


def moe_grouped_mlp(a, w_gate, w_up, w_down, tables, row_weights=None, h=None, y=None,
                    ready=None, err=None, x=None, sorted_token_idx=None):
    """Stage 1 and stage 2 in one launch; returns (h, y).  With x and
    sorted_token_idx (and a=None), stage 1 gathers its rows from the tokens x."""
    gathering = sorted_token_idx is not None
    if gathering:
        _cuda(x, "x", ndim=2)
        _cuda(sorted_token_idx, "sorted_token_idx", dtype=torch.int32)
        src, n_rows, d_h = x, sorted_token_idx.numel(), x.shape[1]
    else:
        _cuda(a, "a", ndim=2)
        src = a
        n_rows, d_h = a.shape
    for n, t in (("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down)):
        _cuda(t, n, dtype=src.dtype, ndim=3)
    E, d_e, d_h2 = w_gate.shape
    if d_h2 != d_h or w_up.shape != w_gate.shape:
        raise ValueError("w_gate / w_up must be [E, d_expert, d_hidden]")
    if tuple(w_down.shape) != (E, d_h, d_e):
        raise ValueError("w_down must be [E, d_hidden, d_expert]")
    s, o, p, g = _tables(tables)
    if row_weights is not None:
        _cuda(row_weights, "row_weights", dtype=torch.float32)
    if h is None:
        h = torch.empty((n_rows, d_e), dtype=src.dtype, device=src.device)
    if y is None:
        y = torch.empty((n_rows, d_h), dtype=src.dtype, device=src.device)
    if ready is None:
        ready = torch.empty(g.numel() + 1, dtype=torch.int32, device=src.device)
    _cuda(h, "h", dtype=src.dtype)
    _cuda(y, "y", dtype=src.dtype)
    _cuda(ready, "ready", dtype=torch.int32)
    if ready.numel() < g.numel() + 1:
        raise ValueError("ready needs one int32 per M block plus one")
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(src.device):
        _check(lib().moe_grouped_mlp(
            _ptr(a) if not gathering else None, _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(s), _ptr(o),
            _ptr(p), _ptr(g), g.numel(), _ptr(row_weights), n_rows, d_h, d_e, E, _dtype_code(src, "x"),
            _ptr(h), _ptr(y), _ptr(ready), _ptr(x) if gathering else None,
            _ptr(sorted_token_idx), x.shape[0] if gathering else 0, _ptr(err), _stream(src.device)),
            "moe_grouped_mlp")
    return h, y


def moe_pack_int4_weights(plain, tile_rows: int):
    """A stacked int4 weight in the pages' format (uint8 [E, N, K // 2]: two
    per byte, element j in byte j // 2 at nibble j % 2 from the low end) ->
    the tiled layout the int4 kernels read (tile_rows 128 for W_gate / W_up,
    256 for W_down); returns a flat uint8 tensor."""
    _cuda(plain, "plain", dtype=torch.uint8, ndim=3)
    E, N, half = plain.shape
    nbytes = int(lib().moe_pack_int4_bytes(E, N, 2 * half, tile_rows))
    if nbytes < 0:
        raise ValueError("K must be a multiple of 64 and tile_rows 128 or 256")
    packed = torch.empty(nbytes, dtype=torch.uint8, device=plain.device)
    with torch.cuda.device(plain.device):
        _check(lib().moe_pack_int4_weights(_ptr(plain), E, N, 2 * half, tile_rows, _ptr(packed),
                                           _stream(plain.device)), "moe_pack_int4_weights")
    return packed


class Int4Experts:
    """The three expert weights of a layer in the int4 kernels' layout, with
    their per-channel scales (or None)."""

    def __init__(self, q_gate, q_up, q_down, s_gate=None, s_up=None, s_down=None):
        """q_gate, q_up: uint8 [E, d_e, d_h // 2]; q_down: [E, d_h, d_e // 2] in
        the pages' int4 format; s_*: fp32 [E, d_e], [E, d_e], [E, d_h] or None."""
        self.E, self.d_e, half = q_gate.shape
        self.d_h = 2 * half
        if tuple(q_up.shape) != tuple(q_gate.shape) or tuple(q_down.shape) != (self.E, self.d_h, self.d_e // 2):
            raise ValueError("q_gate / q_up must be [E, d_e, d_h // 2] and q_down [E, d_h, d_e // 2]")
        self.q_gate = moe_pack_int4_weights(q_gate, 128)
        self.q_up = moe_pack_int4_weights(q_up, 128)
        self.q_down = moe_pack_int4_weights(q_down, 256)
        self.s_gate = _scale(s_gate, "s_gate", (self.E, self.d_e))
        self.s_up = _scale(s_up, "s_up", (self.E, self.d_e))
        self.s_down = _scale(s_down, "s_down", (self.E, self.d_h))


def _scale(t, name, shape):
    if t is None:
        return None
    _cuda(t, name, dtype=torch.float32)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {tuple(shape)}")
    return t


def moe_grouped_mlp_w4a16(x, sorted_token_idx, experts: "Int4Experts", tables, row_weights=None, h=None,
                          y=None, ready=None, err=None):
    """Both expert stages with int4 weights, rows gathered from x [T, d_h];
    returns (h, y)."""
    _cuda(x, "x", ndim=2)
    _cuda(sorted_token_idx, "sorted_token_idx", dtype=torch.int32)
    T, d_h = x.shape
    E, d_e = experts.E, experts.d_e
    if d_h != experts.d_h:
        raise ValueError("x and the experts disagree on d_hidden")
    s, o, p, g = _tables(tables)
    n_rows = sorted_token_idx.numel()
    if row_weights is not None:
        _cuda(row_weights, "row_weights", dtype=torch.float32)
    if h is None:
        h = torch.empty((n_rows, d_e), dtype=x.dtype, device=x.device)
    if y is None:
        y = torch.empty((n_rows, d_h), dtype=x.dtype, device=x.device)
    if ready is None:
        ready = torch.empty(g.numel() + 1, dtype=torch.int32, device=x.device)
    _cuda(h, "h", dtype=x.dtype)
    _cuda(y, "y", dtype=x.dtype)
    _cuda(ready, "ready", dtype=torch.int32)
    if ready.numel() < g.numel() + 1:
        raise ValueError("ready needs one int32 per M block plus one")
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    q = experts
    with torch.cuda.device(x.device):
        _check(lib().moe_grouped_mlp_w4a16(
            _ptr(x), _ptr(sorted_token_idx), T, _ptr(q.q_gate), _ptr(q.q_up), _ptr(q.q_down), _ptr(q.s_gate),
            _ptr(q.s_up), _ptr(q.s_down), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.numel(), _ptr(row_weights),
            n_rows, d_h, d_e, E, _dtype_code(x, "x"), _ptr(h), _ptr(y), _ptr(ready), _ptr(err),
            _stream(x.device)), "moe_grouped_mlp_w4a16")
    return h, y


def moe_gemm_w4a8(a, b_packed, N: int, out=None, ws=None, err=None):
    """W4A8 GEMM: a int8 [M <= 64, K], b_packed = moe_pack_int4_weights(b [1, N, K // 2], 256);
    returns Ct int32 [N, M], the exact sums int4(b) @ a.T."""
    _cuda(a, "a", dtype=torch.int8, ndim=2)
    _cuda(b_packed, "b_packed", dtype=torch.uint8)
    M, K = a.shape
    nws = int(lib().moe_gemm_w4a8_workspace_bytes(M, K))
    if nws < 0:
        raise ValueError("need 1 <= M <= 64, K % 64 == 0, 64 <= K <= 2^20")
    if out is None:
        out = torch.empty((N, M), dtype=torch.int32, device=a.device)
    if ws is None:
        ws = torch.empty(nws, dtype=torch.uint8, device=a.device)
    _cuda(out, "out", dtype=torch.int32)
    _cuda(ws, "ws", dtype=torch.uint8)
    if tuple(out.shape) != (N, M):
        raise ValueError("out must be [N, M]")
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(a.device):
        _check(lib().moe_gemm_w4a8(_ptr(a), _ptr(b_packed), M, N, K, _ptr(out), _ptr(ws), ws.numel(), _ptr(err),
                                   _stream(a.device)), "moe_gemm_w4a8")
    return out


def moe_grouped_gemm_w4a8(x, sorted_token_idx, b_packed, tables, N: int, E: int, n_rows=None, out=None,
                          ws=None, err=None):
    """Grouped W4A8 over the dispatch tables: x int8 [T, K], rows
    x[sorted_token_idx[r]] (None: x's own rows), b_packed the [E, N, K] weight
    packed with tile_rows 256; returns C int32 [n_rows, N]."""
    _cuda(x, "x", dtype=torch.int8, ndim=2)
    _cuda(b_packed, "b_packed", dtype=torch.uint8)
    T, K = x.shape
    if sorted_token_idx is not None:
        _cuda(sorted_token_idx, "sorted_token_idx", dtype=torch.int32)
        n_rows = sorted_token_idx.numel()
    elif n_rows is None:
        n_rows = T
    s, o, p, g = _tables(tables)
    nws = int(lib().moe_grouped_gemm_w4a8_workspace_bytes(max(n_rows, 1), K, max(g.numel(), 1)))
    if nws < 0:
        raise ValueError("need K % 64 == 0, 64 <= K <= 2^20")
    if out is None:
        out = torch.empty((n_rows, N), dtype=torch.int32, device=x.device)
    if ws is None:
        ws = torch.empty(nws, dtype=torch.uint8, device=x.device)
    _cuda(out, "out", dtype=torch.int32)
    _cuda(ws, "ws", dtype=torch.uint8)
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(x.device):
        _check(lib().moe_grouped_gemm_w4a8(
            _ptr(x), _ptr(sorted_token_idx), T, _ptr(b_packed), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.numel(),
            n_rows, N, K, E, _ptr(out), _ptr(ws), ws.numel(), _ptr(err), _stream(x.device)),
            "moe_grouped_gemm_w4a8")
    return out


def moe_forward_w4a16(x, w_g, bias, experts: "Int4Experts", k: int, ws=None, out=None, err=None):
    """The routed forward with int4 experts; returns out [T, d_hidden]."""
    _cuda(x, "x", ndim=2)
    _cuda(w_g, "w_g", dtype=x.dtype)
    if bias is not None:
        _cuda(bias, "bias", dtype=torch.float32, ndim=1)
    T, d_h = x.shape
    E, d_e = experts.E, experts.d_e
    if d_h != experts.d_h:
        raise ValueError("x and the experts disagree on d_hidden")
    need = forward_workspace_bytes(T, d_h, d_e, E, k, x.dtype)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    _cuda(ws, "ws", dtype=torch.uint8)
    if out is None:
        out = torch.empty((T, d_h), dtype=x.dtype, device=x.device)
    _cuda(out, "out", dtype=x.dtype)
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    q = experts
    with torch.cuda.device(x.device):
        _check(lib().moe_forward_w4a16(
            _ptr(x), _ptr(w_g), _ptr(bias), _ptr(q.q_gate), _ptr(q.q_up), _ptr(q.q_down), _ptr(q.s_gate),
            _ptr(q.s_up), _ptr(q.s_down), T, d_h, d_e, E, k, _dtype_code(x, "x"), _ptr(ws), ws.numel(),
            _ptr(out), _ptr(err), _stream(x.device)), "moe_forward_w4a16")
    return out


def moe_reduce_fused(x, token_topk_to_pos, topk_weights=None, out_dtype=None, out=None, err=None):
    """out[t] = cast(sum_k w[t,k] * x[pos[t,k]]) over pos >= 0, fp32 accumulation."""
    _cuda(x, "x", ndim=2)
    _cuda(token_topk_to_pos, "token_topk_to_pos", dtype=torch.int32, ndim=2)
    if topk_weights is not None:
        if topk_weights.dtype != torch.float32:
            raise TypeError(f"topk_weights must be torch.float32, got {topk_weights.dtype}")
        _cuda(topk_weights, "topk_weights", dtype=torch.float32, ndim=2)
        if topk_weights.shape != token_topk_to_pos.shape:
            raise ValueError("topk_weights and token_topk_to_pos shapes differ")
    n_rows, H = x.shape
    T, K = token_topk_to_pos.shape
    if out_dtype is None:
        out_dtype = x.dtype if out is None else out.dtype
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=x.device)
    _cuda(out, "out", dtype=out_dtype)
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(x.device):
        _check(lib().moe_reduce_fused(_ptr(x), n_rows, _ptr(token_topk_to_pos), _ptr(topk_weights),
                                      T, K, H, _dtype_code(x, "x"), _dtype_code(out, "out"),
                                      _ptr(out), _ptr(err), _stream(x.device)),
               "moe_reduce_fused")
    return out


def moe_reduce_fused_scaled(x, token_topk_to_pos, topk_weights=None, x_sf=None, sf=None,
                            out_dtype=None, out=None, err=None):
    """The combine with an optional per-row scale x_sf [n_rows], an optional
    per-token scale sf [T] and an optional float8 e4m3fn output."""
    _cuda(x, "x", ndim=2)
    _cuda(token_topk_to_pos, "token_topk_to_pos", dtype=torch.int32, ndim=2)
    n_rows, H = x.shape
    T, K = token_topk_to_pos.shape
    if topk_weights is not None:
        if topk_weights.dtype != torch.float32:
            raise TypeError(f"topk_weights must be torch.float32, got {topk_weights.dtype}")
        _cuda(topk_weights, "topk_weights", dtype=torch.float32, ndim=2)
        if topk_weights.shape != token_topk_to_pos.shape:
            raise ValueError("topk_weights and token_topk_to_pos shapes differ")
    if x_sf is not None:
        _cuda(x_sf, "x_sf", dtype=torch.float32, ndim=1)
        if x_sf.numel() != n_rows:
            raise ValueError("x_sf must have one entry per row of x")
    if sf is not None:
        _cuda(sf, "sf", dtype=torch.float32, ndim=1)
        if sf.numel() != T:
            raise ValueError("sf must have one entry per token")
    if out_dtype is None:
        out_dtype = x.dtype if out is None else out.dtype
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=x.device)
    _cuda(out, "out", dtype=out_dtype)
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(x.device):
        _check(lib().moe_reduce_fused_scaled(
            _ptr(x), n_rows, _ptr(token_topk_to_pos), _ptr(topk_weights), _ptr(x_sf), _ptr(sf), T, K,
            H, _dtype_code(x, "x"), _dtype_code(out, "out"), _ptr(out), _ptr(err), _stream(x.device)),
            "moe_reduce_fused_scaled")
    return out


def forward_workspace_bytes(T, d_h, d_e, E, k, dtype) -> int:
    return int(lib().moe_forward_workspace_bytes(T, d_h, d_e, E, k, _DT[dtype]))


def forward_workspace_views(ws, T, d_h, d_e, E, k, dtype) -> dict:
    """Typed views of moe_forward's intermediates inside its workspace."""
    L = lib()
    code = _DT[dtype]
    Tk = T * k
    mb = num_m_blocks(T, k, E)
    shapes = {"logits": ((T, E), torch.float32), "topk_idx": ((T, k), torch.int32),
              "topk_w": ((T, k), torch.float32), "group_sizes": ((E,), torch.int32),
              "group_offsets": ((E,), torch.int32), "group_padded_offsets": ((E,), torch.int32),
              "group_idx_for_bx": ((mb,), torch.int32), "sorted_token_idx": ((Tk,), torch.int32),
              "sorted_row_weight": ((Tk,), torch.float32),
              "token_topk_to_pos": ((T, k), torch.int32), "a": ((Tk, d_h), dtype),
              "h": ((Tk, d_e), dtype), "y": ((Tk, d_h), dtype), "mlp_ready": ((mb + 1,), torch.int32)}
    out = {}
    for i, name in enumerate(WS_NAMES):
        if name not in shapes:
            continue
        shape, dt = shapes[name]
        off = int(L.moe_forward_workspace_offset(T, d_h, d_e, E, k, code, i))
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        out[name] = ws[off:off + nbytes].view(dt).view(shape)
    return out


def moe_forward(x, w_g, bias, w_gate, w_up, w_down, k: int, ws=None, out=None, err=None):
    """The whole routed forward; returns out [T, d_hidden].  ``out`` may be a
    pinned host tensor: the combine kernel then stores the result straight
    into host memory (no separate device-to-host copy)."""
    _cuda(x, "x", ndim=2)
    for n, t in (("w_g", w_g), ("w_gate", w_gate), ("w_up", w_up), ("w_down", w_down)):
        _cuda(t, n, dtype=x.dtype)
    if bias is not None:
        _cuda(bias, "bias", dtype=torch.float32, ndim=1)
    T, d_h = x.shape
    E, d_e, _ = w_gate.shape
    need = forward_workspace_bytes(T, d_h, d_e, E, k, x.dtype)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    _cuda(ws, "ws", dtype=torch.uint8)
    if out is None:
        out = torch.empty((T, d_h), dtype=x.dtype, device=x.device)
    _cuda_or_pinned(out, "out", dtype=x.dtype)
    if tuple(out.shape) != (T, d_h):
        raise ValueError(f"out must be [{T}, {d_h}], got {tuple(out.shape)}")
    if err is not None:
        _cuda(err, "err", dtype=torch.int32)
    with torch.cuda.device(x.device):
        _check(lib().moe_forward(_ptr(x), _ptr(w_g), _ptr(bias), _ptr(w_gate), _ptr(w_up),
                                 _ptr(w_down), T, d_h, d_e, E, k, _dtype_code(x, "x"), _ptr(ws),
                                 ws.numel(), _ptr(out), _ptr(err), _stream(x.device)),
               "moe_forward")
    return out


class ForwardPipeline:
    """Back-to-back forwards over a sequence of token batches that live in
    pinned host memory, each result returned to pinned host memory.  Batch
    i's copy in runs on one copy stream while the forward of batch i - 1 runs
    on the compute stream, and batch i - 1's copy out on a second copy stream
    while batch i is computed: two device token buffers and two device
    outputs, ordered by events, each forward one replay of a CUDA graph of
    ``moe_forward``.  Every batch crosses the host link once each way; only
    those copies and the forwards of neighbouring batches overlap.

    :meth:`submit` queues one batch and returns at once; the host must not
    write that batch's ``x_host`` before its copy in has run, nor read its
    ``out_host`` before the returned event has completed."""

    def __init__(self, w_g, bias, w_gate, w_up, w_down, k: int, T: int):
        dev = w_gate.device
        dt = w_gate.dtype
        E, d_e, d_h = w_gate.shape
        self.params = (w_g, bias, w_gate, w_up, w_down, k)
        self.T, self.d_h = T, d_h
        self.x = [torch.zeros((T, d_h), dtype=dt, device=dev) for _ in range(2)]
        self.out = [torch.empty((T, d_h), dtype=dt, device=dev) for _ in range(2)]
        self.ws = torch.empty(forward_workspace_bytes(T, d_h, d_e, E, k, dt), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.compute = torch.cuda.Stream(dev)
        self.copy_in = torch.cuda.Stream(dev)
        self.copy_out = torch.cuda.Stream(dev)
        # the buffers were filled on the caller's stream
        for st in (self.compute, self.copy_in, self.copy_out):
            st.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(self.compute):
            for p in range(2):
                self._body(p)  # first calls on the device outside capture (one-time set-up)
        self.compute.synchronize()
        self.graphs = []
        for p in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.compute):
                self._body(p)
            self.graphs.append(g)
        self.in_done = [torch.cuda.Event() for _ in range(2)]
        self.fwd_done = [torch.cuda.Event() for _ in range(2)]
        self.out_done = [torch.cuda.Event() for _ in range(2)]
        self.issued = 0

    def _body(self, p):
        w_g, bias, w_gate, w_up, w_down, k = self.params
        moe_forward(self.x[p], w_g, bias, w_gate, w_up, w_down, k, ws=self.ws, out=self.out[p], err=self.err)

    def submit(self, x_host, out_host):
        """Queue one batch: x_host and out_host pinned [T, d_hidden] host
        tensors.  Returns the event that completes when out_host holds the
        result."""
        for t, name in ((x_host, "x_host"), (out_host, "out_host")):
            if t.is_cuda or not t.is_pinned() or tuple(t.shape) != (self.T, self.d_h) or t.dtype != self.x[0].dtype:
                raise ValueError(f"{name} must be a pinned host tensor [{self.T}, {self.d_h}] of the weights' dtype")
        p = self.issued % 2
        again = self.issued >= 2
        # copy in: the device buffer is free once the forward two batches back is done
        if again:
            self.copy_in.wait_event(self.fwd_done[p])
        with torch.cuda.stream(self.copy_in):
            self.x[p].copy_(x_host, non_blocking=True)
        self.in_done[p].record(self.copy_in)
        # forward: its tokens are in, and its output buffer has been copied out
        self.compute.wait_event(self.in_done[p])
        if again:
            self.compute.wait_event(self.out_done[p])
        with torch.cuda.stream(self.compute):
            self.graphs[p].replay()
        self.fwd_done[p].record(self.compute)
        # copy out
        self.copy_out.wait_event(self.fwd_done[p])
        with torch.cuda.stream(self.copy_out):
            out_host.copy_(self.out[p], non_blocking=True)
        self.out_done[p].record(self.copy_out)
        self.issued += 1
        return self.out_done[p]

    def synchronize(self):
        for s in (self.copy_in, self.compute, self.copy_out):
            s.synchronize()


class ForwardGraph:
    """``moe_forward`` captured once into a CUDA graph for a fixed token count,
    with static device buffers (and, with ``host_io``, pinned host buffers: a
    copy kernel in the graph reads the tokens from ``x_host``, and the combine
    kernel stores the output straight into ``out_host``).

    Fill ``x`` (or ``x_host``), call :meth:`replay`, and read ``out`` (or
    ``out_host`` after synchronising).  One replay is one launch from the host,
    which removes the per-kernel launch cost of a small decode step."""

    def __init__(self, w_g, bias, w_gate, w_up, w_down, k: int, T: int, host_io: bool = False):
        dev = w_gate.device
        dt = w_gate.dtype
        E, d_e, d_h = w_gate.shape
        self.params = (w_g, bias, w_gate, w_up, w_down, k)
        self.x = torch.zeros((T, d_h), dtype=dt, device=dev)
        self.out = torch.empty((T, d_h), dtype=dt, device=dev)
        self.ws = torch.empty(forward_workspace_bytes(T, d_h, d_e, E, k, dt), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.x_host = torch.zeros((T, d_h), dtype=dt).pin_memory() if host_io else None
        self.out_host = torch.empty((T, d_h), dtype=dt).pin_memory() if host_io else None
        self.stream = torch.cuda.Stream(dev)
        self.stream.wait_stream(torch.cuda.current_stream(dev))  # the buffers were filled on the caller's stream
        with torch.cuda.stream(self.stream):
            self._body()  # first call on the device outside capture (one-time set-up)
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._body()

    def _body(self):
        w_g, bias, w_gate, w_up, w_down, k = self.params
        if self.x_host is not None:
            moe_copy(self.x_host, self.x)  # a kernel, not a memcpy node
        out = self.out_host if self.out_host is not None else self.out
        moe_forward(self.x, w_g, bias, w_gate, w_up, w_down, k, ws=self.ws, out=out, err=self.err)

    def replay(self):
        self.graph.replay()
