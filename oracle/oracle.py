"""ctypes wrapper around the plain C oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` import this module.  It shares
nothing with the CUDA library: it builds and loads its own ``libmoe_oracle.so``
from ``moe_oracle.c`` and never imports the product package.

Arrays are numpy arrays.  16-bit floating point tensors travel as their raw
bits: ``np.float16`` arrays or ``np.uint16`` bit arrays together with a dtype
name (``"f16"``, ``"bf16"``); fp32 tensors as ``np.float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

DTYPE_CODES = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libmoe_oracle.so`` next to its source (gcc, strict fp)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                   "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    sig = {
        "oracle_decode": (None, [P, I, I64, P]),
        "oracle_encode": (None, [P, I, I64, P]),
        "oracle_resolve_threads": (I, [I]),
        "oracle_gate_logits": (I, [P, P, P, I64, I64, I64, I, P, I]),
        "oracle_topk_softmax": (I, [P, I64, I64, I64, P, P]),
        "oracle_num_m_blocks": (I64, [I64, I64, I64, I64]),
        "oracle_build_dispatch": (I, [P, P, I64, I64, I64, I64, P, P, P, P, I64, P, P, P]),
        "oracle_gather_rows": (I, [P, P, I64, I64, I64, I, P]),
        "oracle_grouped_gate_up_silu": (I, [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I64, I, P, I]),
        "oracle_grouped_down": (I, [P, P, P, P, P, P, I64, I64, P, I64, I64, I64, I64, I, P, I]),
        "oracle_reduce_fused": (I, [P, I64, P, P, I64, I64, I64, I, I, P, P, I]),
        "oracle_reduce_fused_scaled": (I, [P, I64, P, P, P, P, I64, I64, I64, I, I, P, P, I]),
        "oracle_moe_tokens_dense": (I, [P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I64, I, P, I]),
        "oracle_rows_gate_up_silu": (I, [P, P, I64, P, P, I64, I64, I64, I, P, I]),
        "oracle_rows_down": (I, [P, P, I64, P, P, I64, I64, I64, I, P, I]),
        "oracle_unpack_int4": (None, [P, I64, P]),
        "oracle_grouped_gate_up_silu_w4": (I, [P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, I64,
                                               I, P, I]),
        "oracle_grouped_down_w4": (I, [P, P, P, P, P, P, P, I64, I64, P, I64, I64, I64, I64, I, P, I]),
        "oracle_gemm_w4a8": (I, [P, P, I64, I64, I64, P, I]),
        "oracle_grouped_gemm_w4a8": (I, [P, P, P, P, P, P, I64, I64, I64, I64, I64, I64, P, I]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a: np.ndarray, dtype: str) -> np.ndarray:
    """Contiguous storage array for ``dtype`` (uint16 bits for f16/bf16)."""
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "e4m3":
        return np.ascontiguousarray(a).view(np.uint8)
    if a.dtype == np.float16:
        if dtype != "f16":
            raise ValueError("np.float16 array passed as bf16")
        return np.ascontiguousarray(a).view(np.uint16)
    if a.dtype in (np.uint16, np.int16):
        return np.ascontiguousarray(a).view(np.uint16)
    raise TypeError(f"expected 16-bit storage for {dtype}, got {a.dtype}")


def _empty(shape, dtype: str) -> np.ndarray:
    if dtype == "e4m3":
        return np.empty(shape, dtype=np.uint8)
    return np.empty(shape, dtype=np.float32 if dtype == "f32" else np.uint16)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def threads(n: int = 0) -> int:
    return _load().oracle_resolve_threads(n)


def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage values -> fp32 (exact widening)."""
    src = _bits(a, dtype)
    out = np.empty(src.shape, dtype=np.float32)
    _load().oracle_decode(_ptr(src), DTYPE_CODES[dtype], src.size, _ptr(out))
    return out


def encode(a: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 -> storage bits, round-to-nearest-even."""
    src = np.ascontiguousarray(a, dtype=np.float32)
    out = _empty(src.shape, dtype)
    _load().oracle_encode(_ptr(src), DTYPE_CODES[dtype], src.size, _ptr(out))
    return out


def gate_logits(x, wg, bias, dtype: str, nthreads: int = 0) -> np.ndarray:
    xb, wb = _bits(x, dtype), _bits(wg, dtype)
    T, d_h = xb.shape
    E = wb.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _check(_load().oracle_gate_logits(_ptr(xb), _ptr(wb), _ptr(b), T, d_h, E,
                                      DTYPE_CODES[dtype], _ptr(out), nthreads), "gate_logits")
    return out


def topk_softmax(logits: np.ndarray, k: int):
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _check(_load().oracle_topk_softmax(_ptr(lg), T, E, k, _ptr(idx), _ptr(w)), "topk_softmax")
    return idx, w


def gate_topk(x, wg, bias, k: int, dtype: str, nthreads: int = 0):
    return topk_softmax(gate_logits(x, wg, bias, dtype, nthreads), k)


def num_m_blocks(T: int, k: int, E: int, block_m: int = 128) -> int:
    return int(_load().oracle_num_m_blocks(T, k, E, block_m))


def build_dispatch(topk_idx: np.ndarray, topk_w, E: int, block_m: int = 128) -> dict:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    w = None if topk_w is None else np.ascontiguousarray(topk_w, dtype=np.float32)
    mb = num_m_blocks(T, k, E, block_m)
    out = {
        "group_sizes": np.empty(E, np.int32),
        "group_offsets": np.empty(E, np.int32),
        "group_padded_offsets": np.empty(E, np.int32),
        "group_idx_for_bx": np.empty(mb, np.int32),
        "sorted_token_idx": np.empty(T * k, np.int32),
        "sorted_row_weight": np.empty(T * k, np.float32),
        "token_topk_to_pos": np.empty((T, k), np.int32),
    }
    _check(_load().oracle_build_dispatch(
        _ptr(idx), _ptr(w), T, k, E, block_m, _ptr(out["group_sizes"]), _ptr(out["group_offsets"]),
        _ptr(out["group_padded_offsets"]), _ptr(out["group_idx_for_bx"]), mb,
        _ptr(out["sorted_token_idx"]), _ptr(out["sorted_row_weight"]),
        _ptr(out["token_topk_to_pos"])), "build_dispatch")
    return out


def gather_rows(x, sorted_token_idx, dtype: str) -> np.ndarray:
    xb = _bits(x, dtype)
    T, d_h = xb.shape
    st = np.ascontiguousarray(sorted_token_idx, dtype=np.int32)
    out = _empty((st.size, d_h), dtype)
    _check(_load().oracle_gather_rows(_ptr(xb), _ptr(st), st.size, T, d_h,
                                      DTYPE_CODES[dtype], _ptr(out)), "gather_rows")
    return out


def _tables(t: dict):
    return [np.ascontiguousarray(t[n], dtype=np.int32) for n in
            ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx")]


def grouped_gate_up_silu(a, w_gate, w_up, tables: dict, dtype: str, block_m: int = 128,
                         nthreads: int = 0) -> np.ndarray:
    ab, wg, wu = _bits(a, dtype), _bits(w_gate, dtype), _bits(w_up, dtype)
    n_rows, d_h = ab.shape
    E, d_e, _ = wg.shape
    s, o, p, g = _tables(tables)
    h = _empty((n_rows, d_e), dtype)
    _check(_load().oracle_grouped_gate_up_silu(
        _ptr(ab), _ptr(wg), _ptr(wu), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.size, block_m,
        n_rows, d_h, d_e, E, DTYPE_CODES[dtype], _ptr(h), nthreads), "grouped_gate_up_silu")
    return h


def grouped_down(h, w_down, tables: dict, dtype: str, row_weights=None, block_m: int = 128,
                 nthreads: int = 0) -> np.ndarray:
    hb, wd = _bits(h, dtype), _bits(w_down, dtype)
    n_rows, d_e = hb.shape
    E, d_h, _ = wd.shape
    s, o, p, g = _tables(tables)
    rw = None if row_weights is None else np.ascontiguousarray(row_weights, dtype=np.float32)
    y = _empty((n_rows, d_h), dtype)
    _check(_load().oracle_grouped_down(
        _ptr(hb), _ptr(wd), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.size, block_m, _ptr(rw),
        n_rows, d_h, d_e, E, DTYPE_CODES[dtype], _ptr(y), nthreads), "grouped_down")
    return y


def unpack_int4(packed: np.ndarray, n: int) -> np.ndarray:
    """int8 values of n int4 elements packed two per byte (element j: byte
    j // 2, nibble j % 2 from the low end, two's complement)."""
    pk = np.ascontiguousarray(packed, dtype=np.uint8)
    if pk.size * 2 < n:
        raise ValueError("not enough packed bytes")
    out = np.empty(n, dtype=np.int8)
    _load().oracle_unpack_int4(_ptr(pk), n, _ptr(out))
    return out


def _f32_or_none(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def grouped_gate_up_silu_w4(a, q_gate, q_up, tables: dict, dtype: str, s_gate=None, s_up=None,
                            block_m: int = 128, nthreads: int = 0) -> np.ndarray:
    """Stage 1 with int4 weights: q_gate / q_up [E, d_e, d_h // 2] uint8 packed
    as the pages print it; s_gate / s_up [E, d_e] fp32 or None."""
    ab = _bits(a, dtype)
    qg, qu = np.ascontiguousarray(q_gate, np.uint8), np.ascontiguousarray(q_up, np.uint8)
    n_rows, d_h = ab.shape
    E, d_e, half = qg.shape
    if half * 2 != d_h or qu.shape != qg.shape:
        raise ValueError("q_gate / q_up must be [E, d_e, d_h // 2]")
    sg, su = _f32_or_none(s_gate), _f32_or_none(s_up)
    s, o, p, g = _tables(tables)
    h = _empty((n_rows, d_e), dtype)
    _check(_load().oracle_grouped_gate_up_silu_w4(
        _ptr(ab), _ptr(qg), _ptr(qu), _ptr(sg), _ptr(su), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.size,
        block_m, n_rows, d_h, d_e, E, DTYPE_CODES[dtype], _ptr(h), nthreads), "grouped_gate_up_silu_w4")
    return h


def grouped_down_w4(h, q_down, tables: dict, dtype: str, s_down=None, row_weights=None,
                    block_m: int = 128, nthreads: int = 0) -> np.ndarray:
    """Stage 2 with int4 weights: q_down [E, d_h, d_e // 2] uint8; s_down [E, d_h] or None."""
    hb = _bits(h, dtype)
    qd = np.ascontiguousarray(q_down, np.uint8)
    n_rows, d_e = hb.shape
    E, d_h, half = qd.shape
    if half * 2 != d_e:
        raise ValueError("q_down must be [E, d_h, d_e // 2]")
    sd = _f32_or_none(s_down)
    rw = _f32_or_none(row_weights)
    s, o, p, g = _tables(tables)
    y = _empty((n_rows, d_h), dtype)
    _check(_load().oracle_grouped_down_w4(
        _ptr(hb), _ptr(qd), _ptr(sd), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.size, block_m, _ptr(rw),
        n_rows, d_h, d_e, E, DTYPE_CODES[dtype], _ptr(y), nthreads), "grouped_down_w4")
    return y


def gemm_w4a8(a, b, nthreads: int = 0) -> np.ndarray:
    """W4A8 GEMM of skeletons.py ``w4a8_dequant_gemm``: a int8 [M, K], b uint8
    [N, K // 2] (int4 two per byte, element j in byte j // 2 at nibble j % 2
    from the low end); returns Ct int32 [N, M] = int4(b) @ a.T, summed exactly."""
    av = np.ascontiguousarray(a, dtype=np.int8)
    bv = np.ascontiguousarray(b, dtype=np.uint8)
    M, K = av.shape
    N, half = bv.shape
    if half * 2 != K:
        raise ValueError("b must be [N, K // 2]")
    ct = np.empty((N, M), dtype=np.int32)
    _check(_load().oracle_gemm_w4a8(_ptr(av), _ptr(bv), M, N, K, _ptr(ct), nthreads), "gemm_w4a8")
    return ct


def grouped_gemm_w4a8(a, b, tables: dict, block_m: int = 128, nthreads: int = 0) -> np.ndarray:
    """The grouped W4A8 GEMM over the dispatch tables: a int8 [n_rows, K] in
    expert order, b uint8 [E, N, K // 2]; returns C int32 [n_rows, N]."""
    av = np.ascontiguousarray(a, dtype=np.int8)
    bv = np.ascontiguousarray(b, dtype=np.uint8)
    n_rows, K = av.shape
    E, N, half = bv.shape
    if half * 2 != K:
        raise ValueError("b must be [E, N, K // 2]")
    s, o, p, g = _tables(tables)
    c = np.zeros((n_rows, N), dtype=np.int32)
    _check(_load().oracle_grouped_gemm_w4a8(
        _ptr(av), _ptr(bv), _ptr(s), _ptr(o), _ptr(p), _ptr(g), g.size, block_m, n_rows, N, K, E, _ptr(c),
        nthreads), "grouped_gemm_w4a8")
    return c


def rows_gate_up_silu(a_rows, row_expert, w_gate, w_up, dtype: str, nthreads: int = 0):
    """Stage 1 for a list of rows; row i uses expert row_expert[i]."""
    ab, wg, wu = _bits(a_rows, dtype), _bits(w_gate, dtype), _bits(w_up, dtype)
    n, d_h = ab.shape
    E, d_e, _ = wg.shape
    re = np.ascontiguousarray(row_expert, dtype=np.int32)
    h = _empty((n, d_e), dtype)
    _check(_load().oracle_rows_gate_up_silu(_ptr(ab), _ptr(re), n, _ptr(wg), _ptr(wu), d_h, d_e, E,
                                            DTYPE_CODES[dtype], _ptr(h), nthreads), "rows_gate_up_silu")
    return h


def rows_down(h_rows, row_expert, w_down, dtype: str, row_weights=None, nthreads: int = 0):
    """Stage 2 for a list of rows; row i uses expert row_expert[i]."""
    hb, wd = _bits(h_rows, dtype), _bits(w_down, dtype)
    n, d_e = hb.shape
    E, d_h, _ = wd.shape
    re = np.ascontiguousarray(row_expert, dtype=np.int32)
    rw = None if row_weights is None else np.ascontiguousarray(row_weights, dtype=np.float32)
    y = _empty((n, d_h), dtype)
    _check(_load().oracle_rows_down(_ptr(hb), _ptr(re), n, _ptr(wd), _ptr(rw), d_h, d_e, E,
                                    DTYPE_CODES[dtype], _ptr(y), nthreads), "rows_down")
    return y


def reduce_fused(x, token_topk_to_pos, topk_weights, in_dtype: str, out_dtype: str,
                 nthreads: int = 0):
    """Returns (out, err_flag)."""
    pos = np.ascontiguousarray(token_topk_to_pos, dtype=np.int32)
    T, K = pos.shape
    xb = _bits(x, in_dtype)
    n_rows, H = xb.shape
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32)
    out = _empty((T, H), out_dtype)
    err = np.zeros(1, np.int32)
    _check(_load().oracle_reduce_fused(_ptr(xb), n_rows, _ptr(pos), _ptr(w), T, K, H,
                                       DTYPE_CODES[in_dtype], DTYPE_CODES[out_dtype], _ptr(out),
                                       _ptr(err), nthreads), "reduce_fused")
    return out, int(err[0])


def reduce_fused_scaled(x, token_topk_to_pos, topk_weights, x_sf, sf, in_dtype: str,
                        out_dtype: str, nthreads: int = 0):
    """The combine with the optional per-row x_sf and per-token sf scales and
    e4m3 output.  Returns (out, err_flag)."""
    pos = np.ascontiguousarray(token_topk_to_pos, dtype=np.int32)
    T, K = pos.shape
    xb = _bits(x, in_dtype)
    n_rows, H = xb.shape
    f32 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float32)
    w, xs, s = f32(topk_weights), f32(x_sf), f32(sf)
    out = _empty((T, H), out_dtype)
    err = np.zeros(1, np.int32)
    _check(_load().oracle_reduce_fused_scaled(_ptr(xb), n_rows, _ptr(pos), _ptr(w), _ptr(xs),
                                              _ptr(s), T, K, H, DTYPE_CODES[in_dtype],
                                              DTYPE_CODES[out_dtype], _ptr(out), _ptr(err),
                                              nthreads), "reduce_fused_scaled")
    return out, int(err[0])


def moe_tokens_dense(x, w_gate, w_up, w_down, topk_idx, topk_w, tokens, dtype: str,
                     nthreads: int = 0) -> np.ndarray:
    """Brute-force forward of the listed tokens, no dispatch tables involved."""
    xb = _bits(x, dtype)
    wg, wu, wd = _bits(w_gate, dtype), _bits(w_up, dtype), _bits(w_down, dtype)
    T, d_h = xb.shape
    E, d_e, _ = wg.shape
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    k = idx.shape[1]
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    out = _empty((tok.size, d_h), dtype)
    _check(_load().oracle_moe_tokens_dense(
        _ptr(xb), _ptr(wg), _ptr(wu), _ptr(wd), _ptr(idx), _ptr(w), _ptr(tok), tok.size, T, d_h,
        d_e, E, k, DTYPE_CODES[dtype], _ptr(out), nthreads), "moe_tokens_dense")
    return out


def moe_forward(x, wg, bias, w_gate, w_up, w_down, k: int, dtype: str, block_m: int = 128,
                nthreads: int = 0) -> dict:
    """The whole path through the dispatch tables: gate, top-k, tables, gather,
    stage 1, stage 2 and the fp32 combine.  Returns every intermediate."""
    E = _bits(wg, dtype).shape[0]
    logits = gate_logits(x, wg, bias, dtype, nthreads)
    idx, w = topk_softmax(logits, k)
    tab = build_dispatch(idx, w, E, block_m)
    a = gather_rows(x, tab["sorted_token_idx"], dtype)
    h = grouped_gate_up_silu(a, w_gate, w_up, tab, dtype, block_m, nthreads)
    y = grouped_down(h, w_down, tab, dtype, None, block_m, nthreads)
    out, err = reduce_fused(y, tab["token_topk_to_pos"], w, dtype, dtype, nthreads)
    res = dict(tab)
    res.update(logits=logits, topk_idx=idx, topk_w=w, a=a, h=h, y=y, out=out, err=err)
    return res
