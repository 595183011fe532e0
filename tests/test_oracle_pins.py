"""Pins of the CPU oracle against things other than itself: values the pages
print, hand-computed cases, closed forms, brute force and library routines.

These run without a GPU (``-m "not gpu"``)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

from mixture_experts_routed_gate_gb300 import roofline, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_f16(a):
    return np.asarray(a, np.float32).astype(np.float16).view(np.uint16)


def _enc(a, dtype):
    if dtype == "bf16":
        return _bits_bf16(a)
    if dtype == "f16":
        return _bits_f16(a)
    return np.asarray(a, np.float32)


# --------------------------------------------------------------------------- #
# storage conversions vs numpy float16 and torch bfloat16
# --------------------------------------------------------------------------- #

def test_decode_all_half_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_decode_all_bf16_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _encode_probe_values():
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000).astype(np.float32) * s for s in (1e-6, 1e-3, 1, 1e3, 6e4)]
    # exact halfway points and their neighbours for both formats
    h = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)
    h = h[np.isfinite(h)]
    nxt = np.nextafter(h.astype(np.float16), np.float16(np.inf)).astype(np.float32)
    mid = ((h.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)
    b = (np.arange(0, 65536, 5, dtype=np.uint32) << 16).view(np.float32)
    b = b[np.isfinite(b)]
    bmid = (b.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.99, 65520, 65536, 6.1e-5,
                        5.96e-8, 2.98e-8, 2.99e-8, 1e-9, 3.4e38, -3.4e38], np.float32)
    allv = np.concatenate(vals + [h, mid, np.nextafter(mid, np.float32(np.inf)),
                                  np.nextafter(mid, np.float32(-np.inf)), b, bmid, special])
    return allv[np.isfinite(allv) | np.isinf(allv)]


def test_encode_half_matches_numpy(oracle):
    v = _encode_probe_values()
    got = oracle.encode(v, "f16")
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_encode_bf16_matches_torch(oracle):
    v = _encode_probe_values()
    got = oracle.encode(v, "bf16")
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------- #
# o1 gate logits
# --------------------------------------------------------------------------- #

def test_gate_logits_hand_computed_order(oracle):
    """The two hand-computed cases pin the chunk ownership, the in-lane order
    and the butterfly order (see the fixture for the arithmetic)."""
    with open(os.path.join(GOLDEN, "gate_order_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        d_h = c["d_hidden"]
        w = np.zeros((1, d_h), np.float32)
        for j, v in c["w_at"].items():
            w[0, int(j)] = v
        x = np.ones((1, d_h), np.float32)
        got = oracle.gate_logits(_bits_bf16(x), _bits_bf16(w), None, "bf16")
        assert got[0, 0] == np.float32(c["logit"]), c["what"]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gate_logits_integer_inputs_exact(oracle, dtype):
    """Small integers: every partial sum is exact, so any order gives the
    integer matmul."""
    rng = np.random.default_rng(1)
    T, d_h, E = 7, 512, 5
    x = rng.integers(-4, 5, (T, d_h)).astype(np.float32)
    w = rng.integers(-4, 5, (E, d_h)).astype(np.float32)
    bias = rng.integers(-3, 4, E).astype(np.float32)
    got = oracle.gate_logits(_enc(x, dtype), _enc(w, dtype), bias, dtype)
    ref = (x.astype(np.int64) @ w.astype(np.int64).T + bias.astype(np.int64)).astype(np.float32)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gate_logits_random_within_fp32_bound(oracle, dtype):
    rng = np.random.default_rng(2)
    T, d_h, E = 9, 1024, 16
    xs = _enc(rng.standard_normal((T, d_h)), dtype)
    ws = _enc(rng.standard_normal((E, d_h)) / 32, dtype)
    xf, wf = oracle.decode(xs, dtype).astype(np.float64), oracle.decode(ws, dtype).astype(np.float64)
    got = oracle.gate_logits(xs, ws, None, dtype)
    ref = xf @ wf.T
    bound = (d_h // 256 * 8 + 5) * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T) * 1.01
    assert np.all(np.abs(got - ref) <= bound)


def test_gate_logits_rejects_bad_hidden(oracle):
    with pytest.raises(ValueError):
        oracle.gate_logits(np.zeros((2, 200), np.uint16), np.zeros((3, 200), np.uint16), None, "bf16")


# --------------------------------------------------------------------------- #
# o2 top-k + softmax
# --------------------------------------------------------------------------- #

def _brute_topk(l, k):
    """Enumerate every k-subset; keep the one that no outside expert beats,
    then order it.  'a beats b' = larger logit, or equal logit and lower id."""
    E = len(l)
    beats = lambda a, b: l[a] > l[b] or (l[a] == l[b] and a < b)
    for sub in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in sub]
        if all(beats(s, r) for s in sub for r in rest):
            chosen = list(sub)
            # order: position of s = number of chosen experts that beat s
            return sorted(chosen, key=lambda s: sum(beats(o, s) for o in chosen))
    raise AssertionError


def test_topk_brute_force_small(oracle):
    rng = np.random.default_rng(3)
    E, k, T = 8, 2, 300
    logits = rng.integers(-3, 4, (T, E)).astype(np.float32)  # many ties
    idx, w = oracle.topk_softmax(logits, k)
    for t in range(T):
        assert list(idx[t]) == _brute_topk(logits[t], k)
    for k in (1, 3, 8):
        idx, _ = oracle.topk_softmax(logits, k)
        for t in range(0, T, 17):
            assert list(idx[t]) == _brute_topk(logits[t], k)


def test_topk_ties_go_to_lower_id(oracle):
    logits = np.array([[1.0, 5.0, 5.0, 2.0, 5.0]], np.float32)
    idx, w = oracle.topk_softmax(logits, 3)
    assert list(idx[0]) == [1, 2, 4]
    assert w[0, 0] == w[0, 1] == w[0, 2]


def test_topk_weights_are_softmax_probabilities(oracle):
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal((50, 64)) * 3).astype(np.float32)
    idx, w = oracle.topk_softmax(logits, 6)
    p = sp_softmax(logits.astype(np.float64), axis=1)
    ref = np.take_along_axis(p, idx.astype(np.int64), axis=1).astype(np.float32)
    assert np.allclose(w, ref, rtol=2e-7, atol=0)
    idx_all, w_all = oracle.topk_softmax(logits, 64)
    assert np.allclose(w_all.astype(np.float64).sum(1), 1.0, atol=1e-6)


# --------------------------------------------------------------------------- #
# o3 dispatch
# --------------------------------------------------------------------------- #

def test_dispatch_worked_examples_from_pages(oracle):
    with open(os.path.join(GOLDEN, "dispatch_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    c0, c1 = cases
    # example 1: counts [2,2,2] -> offsets [0,2,4]
    idx = np.repeat(np.arange(3), c0["counts"]).astype(np.int32).reshape(3, 2)
    tab = oracle.build_dispatch(idx, None, 3, 128)
    assert list(tab["group_sizes"]) == c0["counts"]
    assert list(tab["group_offsets"]) == c0["group_offsets"]
    assert list(np.cumsum(tab["group_sizes"])) == c0["cumsum"]
    # example 2: padded starts [0,3,6] with block 1; bx=1 -> expert 0
    idx = np.repeat(np.arange(3), c1["counts"]).astype(np.int32).reshape(3, 2)
    tab = oracle.build_dispatch(idx, None, 3, c1["block_m"])
    assert list(tab["group_padded_offsets"]) == c1["group_padded_offsets"]
    assert tab["group_idx_for_bx"][c1["bx"]] == c1["expert_for_bx"]
    assert list(tab["group_idx_for_bx"]) == [0, 0, 0, 1, 1, 1, 2, 2, 2]


def _dispatch_invariants(idx, w, tab, E, block_m):
    T, k = idx.shape
    Tk = T * k
    sizes, off, po, gidx = (tab[n] for n in ("group_sizes", "group_offsets",
                                               "group_padded_offsets", "group_idx_for_bx"))
    assert sizes.sum() == Tk
    assert np.array_equal(np.bincount(idx.ravel(), minlength=E), sizes)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(sizes)[:-1]]))
    assert np.all(po % block_m == 0) and po[0] == 0
    steps = np.diff(po)
    assert np.array_equal(steps, ((sizes[:-1] + 1 + block_m - 1) // block_m) * block_m)
    assert np.all(steps > 0)
    mb = len(gidx)
    assert mb == math.ceil(Tk / block_m) + E
    assert po[-1] + ((sizes[-1] + block_m) // block_m) * block_m <= block_m * mb
    assert np.all(np.diff(gidx) >= 0)
    assert set(gidx.tolist()) == set(range(E))          # every expert owns a block
    # brute-force block lookup: bisect over the starts
    for bx in range(mb):
        assert gidx[bx] == np.searchsorted(po, bx * block_m, side="right") - 1
    pos = tab["token_topk_to_pos"].ravel()
    assert np.array_equal(np.sort(pos), np.arange(Tk))
    st, sw = tab["sorted_token_idx"], tab["sorted_row_weight"]
    flat = idx.ravel()
    # brute force stable rank: rank(f) = #{f' < f with the same expert}
    for f in range(Tk):
        e = flat[f]
        rank = int(np.count_nonzero(flat[:f] == e))
        assert pos[f] == off[e] + rank
        assert st[pos[f]] == f // k
        if w is not None:
            assert sw[pos[f]] == w.ravel()[f]
    for e in range(E):
        seg = st[off[e]:off[e] + sizes[e]]
        assert np.all(np.diff(seg) >= 0)


@pytest.mark.parametrize("T,k,E,block_m", [(64, 2, 8, 128), (37, 6, 64, 128), (300, 8, 16, 32),
                                           (5, 4, 4, 1), (0, 2, 8, 128)])
def test_dispatch_invariants_random(oracle, T, k, E, block_m):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], np.int32).reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    tab = oracle.build_dispatch(idx, w, E, block_m)
    _dispatch_invariants(idx, w, tab, E, block_m)


def test_dispatch_exact_multiple_and_empty_experts(oracle):
    """count % block == 0 still gets a whole padding block (the +1), and an
    empty expert owns one block."""
    T, k, E = 128, 1, 4
    idx = np.full((T, k), 2, np.int32)         # expert 2 gets exactly 128 rows
    tab = oracle.build_dispatch(idx, None, E, 128)
    assert list(tab["group_sizes"]) == [0, 0, 128, 0]
    assert list(tab["group_padded_offsets"]) == [0, 128, 256, 512]
    assert list(tab["group_idx_for_bx"]) == [0, 1, 2, 2, 3]
    _dispatch_invariants(idx, None, tab, E, 128)


def test_gather_rows_is_fancy_indexing(oracle):
    rng = np.random.default_rng(5)
    x = rng.integers(0, 65535, (11, 16)).astype(np.uint16)
    st = rng.integers(0, 11, 30).astype(np.int32)
    assert np.array_equal(oracle.gather_rows(x, st, "bf16"), x[st])


# --------------------------------------------------------------------------- #
# o4 grouped GEMMs
# --------------------------------------------------------------------------- #

def _random_tables(oracle, rng, T, k, E, block_m=128):
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    return idx, oracle.build_dispatch(idx, None, E, block_m)


def test_grouped_gemms_integer_closed_form(oracle):
    """fp32 storage, integer operands, gate logits >= 40: silu(G) rounds to G
    in fp32, so h = G*U and y = h W_down^T exactly (all sums < 2^24).  With
    400 rows over 3 experts, experts span several 128-row blocks."""
    rng = np.random.default_rng(6)
    T, k, E, d_h, d_e = 200, 2, 3, 32, 16
    idx, tab = _random_tables(oracle, rng, T, k, E)
    Tk = T * k
    a = rng.integers(0, 3, (Tk, d_h)).astype(np.float32)
    a[:, 0] = 1
    wg = rng.integers(0, 2, (E, d_e, d_h)).astype(np.float32)
    wg[:, :, 0] = 40
    wu = rng.integers(-2, 3, (E, d_e, d_h)).astype(np.float32)
    wd = rng.integers(-1, 2, (E, d_h, d_e)).astype(np.float32)
    h = oracle.grouped_gate_up_silu(a, wg, wu, tab, "f32")
    y = oracle.grouped_down(h, wd, tab, "f32")
    expert_of_row = np.repeat(np.arange(E), tab["group_sizes"])
    ai = a.astype(np.int64)
    G = np.einsum("rj,rnj->rn", ai, wg.astype(np.int64)[expert_of_row])
    U = np.einsum("rj,rnj->rn", ai, wu.astype(np.int64)[expert_of_row])
    assert G.min() >= 40
    H = G * U
    assert np.array_equal(h, H.astype(np.float32))
    assert tab["group_sizes"].max() > 128
    Y = np.einsum("rn,ron->ro", H, wd.astype(np.int64)[expert_of_row])
    assert np.abs(Y).max() < 2 ** 24
    assert np.array_equal(y, Y.astype(np.float32))
    rw = rng.choice([0.5, 1.0, 2.0, 0.25], Tk).astype(np.float32)
    y2 = oracle.grouped_down(h, wd, tab, "f32", row_weights=rw)
    assert np.array_equal(y2, (Y * rw[:, None]).astype(np.float32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_grouped_gemms_random_vs_float64(oracle, dtype):
    """Per-expert definition in float64 (no tables: the expert of a row is found
    from sizes alone) vs the oracle's block walk, within fp32 accumulation
    error plus one storage rounding."""
    rng = np.random.default_rng(7)
    T, k, E, d_h, d_e = 50, 3, 6, 256, 64
    idx, tab = _random_tables(oracle, rng, T, k, E)
    Tk = T * k
    a = _enc(rng.standard_normal((Tk, d_h)), dtype)
    wg = _enc(rng.standard_normal((E, d_e, d_h)) / 16, dtype)
    wu = _enc(rng.standard_normal((E, d_e, d_h)) / 16, dtype)
    wd = _enc(rng.standard_normal((E, d_h, d_e)) / 8, dtype)
    h = oracle.grouped_gate_up_silu(a, wg, wu, tab, dtype)
    y = oracle.grouped_down(h, wd, tab, dtype)
    af, gf, uf, df = (oracle.decode(v, dtype).astype(np.float64) for v in (a, wg, wu, wd))
    hf, yf = oracle.decode(h, dtype).astype(np.float64), oracle.decode(y, dtype).astype(np.float64)
    eps = 2.0 ** -11 if dtype == "f16" else 2.0 ** -8
    for r in range(Tk):
        e = int(np.searchsorted(np.cumsum(tab["group_sizes"]), r, side="right"))
        G = gf[e] @ af[r]
        U = uf[e] @ af[r]
        ref_h = G / (1 + np.exp(-G)) * U
        tol_h = eps * np.abs(ref_h) + 1e-5 * (np.abs(gf[e]) @ np.abs(af[r]) + np.abs(uf[e]) @ np.abs(af[r])) + 1e-6
        assert np.all(np.abs(hf[r] - ref_h) <= tol_h)
        ref_y = df[e] @ hf[r]
        tol_y = eps * np.abs(ref_y) + 1e-5 * (np.abs(df[e]) @ np.abs(hf[r])) + 1e-6
        assert np.all(np.abs(yf[r] - ref_y) <= tol_y)


def test_row_forms_integer_closed_form(oracle):
    """rows_gate_up_silu / rows_down (row i uses expert row_expert[i], the
    forms the full-size tests sample with): fp32 storage, integer operands,
    gate logits >= 40 so silu(G) rounds to G, a shuffled row -> expert map
    that is neither sorted nor the identity, and power-of-two row weights.
    Every sum is an integer below 2^24, so h = G*U and y = (h W_down^T) * rw
    hold exactly against an int64 einsum."""
    rng = np.random.default_rng(16)
    n, E, d_h, d_e = 97, 5, 32, 16
    row_expert = rng.integers(0, E, n).astype(np.int32)
    assert not np.all(np.diff(row_expert) >= 0)
    a = rng.integers(0, 3, (n, d_h)).astype(np.float32)
    a[:, 0] = 1
    wg = rng.integers(0, 2, (E, d_e, d_h)).astype(np.float32)
    wg[:, :, 0] = 40
    wu = rng.integers(-2, 3, (E, d_e, d_h)).astype(np.float32)
    wd = rng.integers(-1, 2, (E, d_h, d_e)).astype(np.float32)
    rw = rng.choice([0.5, 1.0, 2.0, 0.25], n).astype(np.float32)
    h = oracle.rows_gate_up_silu(a, row_expert, wg, wu, "f32")
    y = oracle.rows_down(h, row_expert, wd, "f32", row_weights=rw)
    y1 = oracle.rows_down(h, row_expert, wd, "f32")
    ai = a.astype(np.int64)
    G = np.einsum("rj,rnj->rn", ai, wg.astype(np.int64)[row_expert])
    U = np.einsum("rj,rnj->rn", ai, wu.astype(np.int64)[row_expert])
    assert G.min() >= 40
    H = G * U
    assert np.array_equal(h, H.astype(np.float32))
    Y = np.einsum("rn,ron->ro", H, wd.astype(np.int64)[row_expert])
    assert np.abs(Y).max() < 2 ** 24
    assert np.array_equal(y1, Y.astype(np.float32))
    assert np.array_equal(y, (Y * rw[:, None]).astype(np.float32))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_row_forms_equal_the_block_walk_on_shuffled_rows(oracle, dtype):
    """The rows of a dispatch fed to the per-row forms in a shuffled order,
    each with the expert its block belongs to, give the table-driven
    stages' rows bit for bit (random 16-bit inputs, rows spanning several
    128-row blocks and a ragged tail, row weights in stage 2)."""
    rng = np.random.default_rng(17)
    T, k, E, d_h, d_e = 300, 2, 3, 64, 32
    idx, tab = _random_tables(oracle, rng, T, k, E)
    Tk = T * k
    assert tab["group_sizes"].max() > 128
    a = _enc(rng.standard_normal((Tk, d_h)), dtype)
    wg = _enc(rng.standard_normal((E, d_e, d_h)) / 8, dtype)
    wu = _enc(rng.standard_normal((E, d_e, d_h)) / 8, dtype)
    wd = _enc(rng.standard_normal((E, d_h, d_e)) / 6, dtype)
    rw = rng.random(Tk).astype(np.float32)
    h = oracle.grouped_gate_up_silu(a, wg, wu, tab, dtype)
    y = oracle.grouped_down(h, wd, tab, dtype, row_weights=rw)
    expert_of_row = np.repeat(np.arange(E, dtype=np.int32), tab["group_sizes"])
    perm = rng.permutation(Tk)
    h_rows = oracle.rows_gate_up_silu(a[perm], expert_of_row[perm], wg, wu, dtype)
    assert np.array_equal(h_rows, h[perm])
    y_rows = oracle.rows_down(h[perm], expert_of_row[perm], wd, dtype, row_weights=rw[perm])
    assert np.array_equal(y_rows, y[perm])


def test_grouped_gemms_zero_weights(oracle):
    rng = np.random.default_rng(8)
    T, k, E, d_h, d_e = 20, 2, 4, 64, 32
    idx, tab = _random_tables(oracle, rng, T, k, E)
    a = _bits_bf16(rng.standard_normal((T * k, d_h)))
    wg = _bits_bf16(rng.standard_normal((E, d_e, d_h)))
    zero_u = np.zeros((E, d_e, d_h), np.uint16)
    h = oracle.grouped_gate_up_silu(a, wg, zero_u, tab, "bf16")
    assert np.all(oracle.decode(h, "bf16") == 0)
    wu = _bits_bf16(rng.standard_normal((E, d_e, d_h)))
    h = oracle.grouped_gate_up_silu(a, wg, wu, tab, "bf16")
    y = oracle.grouped_down(h, np.zeros((E, d_h, d_e), np.uint16), tab, "bf16")
    assert np.all(oracle.decode(y, "bf16") == 0)


def test_silu_special_values(oracle):
    """fp32 operands with W_up = identity-like selector: h = silu(G) * 1.
    silu(0) = 0; silu(G) = G for large G; silu(-G) ~ -G e^-G."""
    Gs = np.array([0.0, 1.0, -1.0, 40.0, -20.0, 3.5], np.float32)
    n = len(Gs)
    T, k, E, d_h, d_e = n, 1, 1, 8, 1
    idx = np.zeros((T, k), np.int32)
    tab = oracle.build_dispatch(idx, None, E, 128)
    a = np.zeros((n, d_h), np.float32)
    a[:, 0] = Gs
    a[:, 1] = 1.0
    wg = np.zeros((1, 1, d_h), np.float32); wg[0, 0, 0] = 1.0
    wu = np.zeros((1, 1, d_h), np.float32); wu[0, 0, 1] = 1.0
    h = oracle.grouped_gate_up_silu(a, wg, wu, tab, "f32")[:, 0]
    ref = (Gs.astype(np.float64) / (1 + np.exp(-Gs.astype(np.float64)))).astype(np.float32)
    assert np.array_equal(h, ref)
    assert h[0] == 0 and h[3] == 40.0


# --------------------------------------------------------------------------- #
# o5 reduce
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_reduce_k1_unit_weight_identity(oracle, dtype):
    rng = np.random.default_rng(9)
    T, H = 13, 256
    x = _enc(rng.standard_normal((T, H)), dtype)
    perm = rng.permutation(T).astype(np.int32).reshape(T, 1)
    out, err = oracle.reduce_fused(x, perm, None, dtype, dtype)
    assert err == 0
    assert np.array_equal(out, x[perm[:, 0]])
    out, _ = oracle.reduce_fused(x, perm, np.ones((T, 1), np.float32), dtype, dtype)
    assert np.array_equal(out, x[perm[:, 0]])


def test_reduce_all_padding_is_zero(oracle):
    x = _bits_bf16(np.ones((4, 256)))
    pos = np.full((3, 2), -1, np.int32)
    out, err = oracle.reduce_fused(x, pos, np.ones((3, 2), np.float32), "bf16", "bf16")
    assert err == 0 and np.all(out == 0)


def test_reduce_padding_rows_never_read(oracle):
    """Rows that only padding slots pointed at may hold NaN or huge values."""
    d = workloads.make_reduce_inputs(32, 8, 512, "bf16", seed=1)
    x = workloads.to_numpy_bits(d["x"]).copy()
    pos = d["pos"].numpy()
    w = d["w"].numpy()
    out1, _ = oracle.reduce_fused(x, pos, w, "bf16", "bf16")
    unused = np.setdiff1d(np.arange(x.shape[0]), pos[pos >= 0])
    assert unused.size > 0
    x[unused[::2]] = 0x7FC0   # NaN
    x[unused[1::2]] = 0x7F7F  # ~3.4e38
    out2, _ = oracle.reduce_fused(x, pos, w, "bf16", "bf16")
    assert np.array_equal(out1, out2)


def test_reduce_integer_pow2_weights_exact(oracle):
    rng = np.random.default_rng(10)
    T, K, H = 16, 8, 256
    x = rng.integers(-8, 9, (T * K, H)).astype(np.float32)
    pos = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    pos[rng.random((T, K)) < 0.2] = -1
    w = rng.choice([0.25, 0.5, 1.0, 2.0], (T, K)).astype(np.float32)
    out, _ = oracle.reduce_fused(x, pos, w, "f32", "f32")
    ref = np.zeros((T, H))
    for t in range(T):
        for kk in range(K):
            if pos[t, kk] >= 0:
                ref[t] += w[t, kk] * x[pos[t, kk]]
    assert np.array_equal(out, ref.astype(np.float32))


def test_reduce_random_vs_float64(oracle):
    d = workloads.make_reduce_inputs(64, 8, 1024, "bf16", seed=2)
    x = workloads.to_numpy_bits(d["x"])
    pos, w = d["pos"].numpy(), d["w"].numpy()
    out, _ = oracle.reduce_fused(x, pos, w, "bf16", "f32")
    xf = oracle.decode(x, "bf16").astype(np.float64)
    ref = np.zeros((64, 1024))
    mag = np.zeros((64, 1024))
    for t in range(64):
        for kk in range(8):
            if pos[t, kk] >= 0:
                ref[t] += w[t, kk] * xf[pos[t, kk]]
                mag[t] += abs(w[t, kk]) * np.abs(xf[pos[t, kk]])
    assert np.all(np.abs(out - ref) <= 9 * 2.0 ** -24 * mag + 1e-30)


def test_reduce_flags_out_of_range(oracle):
    x = _bits_bf16(np.ones((4, 256)))
    pos = np.array([[0, 4], [1, -2]], np.int32)
    out, err = oracle.reduce_fused(x, pos, None, "bf16", "bf16")
    assert err == 1
    assert np.all(oracle.decode(out, "bf16") == 1.0)


def test_reduce_byte_formula_matches_pages():
    """TileOPs-Metax PR #55, section 3 (Roofline): 66.09 MB at 512x8x7168 bf16,
    58.72 MB read + 7.34 MB write + 32.8 KB metadata."""
    T, K, H = 512, 8, 7168
    total = roofline.reduce_bytes_pages(T, K, H, 2)
    assert round(total / 1e6, 2) == 66.09
    assert round(T * K * H * 2 / 1e6, 2) == 58.72
    assert round(T * H * 2 / 1e6, 2) == 7.34
    assert round((T * K * 8) / 1e3, 1) == 32.8


# --------------------------------------------------------------------------- #
# o6 brute force vs the composition through the tables
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_dense_brute_force_equals_table_path(oracle, dtype):
    cfg = workloads.MoEConfig("t", 1, 48, 256, 64, 8, 3, dtype, 11)
    d = workloads.make_moe_inputs(cfg)
    nb = {kk: (workloads.to_numpy_bits(v) if v is not None else None) for kk, v in d.items()}
    res = oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"],
                             nb["w_down"], cfg.top_k, dtype)
    tokens = np.arange(cfg.T, dtype=np.int32)
    dense = oracle.moe_tokens_dense(nb["x"], nb["w_gate"], nb["w_up"], nb["w_down"],
                                    res["topk_idx"], res["topk_w"], tokens, dtype)
    assert np.array_equal(dense, res["out"])
    assert res["err"] == 0


# --------------------------------------------------------------------------- #
# combine variants: x_sf / sf scales and float8 e4m3fn output
# --------------------------------------------------------------------------- #

def test_decode_all_e4m3_patterns(oracle):
    bits = np.arange(256, dtype=np.uint8)
    got = oracle.decode(bits, "e4m3")
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_encode_e4m3_matches_torch_in_range_and_saturates(oracle):
    rng = np.random.default_rng(20)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 30, 200)]).astype(np.float32)
    grid = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    grid = np.sort(grid[np.isfinite(grid)])
    mids = ((grid[1:].astype(np.float64) + grid[:-1]) / 2).astype(np.float32)  # exact ties
    v = np.concatenate([v, grid, mids, np.nextafter(mids, np.float32(1e9)), np.nextafter(mids, np.float32(-1e9))])
    v = v[np.abs(v) < 464]
    got = oracle.encode(v, "e4m3")
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # past the largest finite value the saturating reading gives +-448 (0x7e / 0xfe)
    big = np.array([464.0, 500.0, 1e30, -464.0, -1e30], np.float32)
    assert list(oracle.encode(big, "e4m3")) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.encode(np.array([np.nan], np.float32), "e4m3")[0] & 0x7F == 0x7F


def test_scaled_combine_reduces_to_plain_and_closed_forms(oracle):
    d = workloads.make_reduce_inputs(24, 8, 512, "bf16", seed=21)
    x = workloads.to_numpy_bits(d["x"])
    pos, w = d["pos"].numpy(), d["w"].numpy()
    base, _ = oracle.reduce_fused(x, pos, w, "bf16", "bf16")
    ones_r, ones_t = np.ones(x.shape[0], np.float32), np.ones(24, np.float32)
    for xs, sf in ((None, None), (ones_r, None), (None, ones_t), (ones_r, ones_t)):
        got, _ = oracle.reduce_fused_scaled(x, pos, w, xs, sf, "bf16", "bf16")
        assert np.array_equal(got, base)
    # integer rows, power-of-two weights and scales: every product and sum exact
    rng = np.random.default_rng(22)
    T, K, H = 12, 4, 256
    xi = rng.integers(-6, 7, (T * K, H)).astype(np.float32)
    pos = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    pos[0, 1] = -1
    wi = rng.choice([0.5, 1.0, 2.0], (T, K)).astype(np.float32)
    xs = rng.choice([0.25, 1.0, 4.0], T * K).astype(np.float32)
    sf = rng.choice([0.5, 2.0], T).astype(np.float32)
    got, _ = oracle.reduce_fused_scaled(xi, pos, wi, xs, sf, "f32", "f32")
    ref = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            if pos[t, k] >= 0:
                ref[t] += wi[t, k] * xs[pos[t, k]] * xi[pos[t, k]]
        ref[t] *= sf[t]
    assert np.array_equal(got, ref.astype(np.float32))


def test_e4m3_output_is_the_rounded_fp32_result(oracle):
    """With fp32 in, the e4m3 output equals rounding the fp32 output once."""
    d = workloads.make_reduce_inputs(16, 8, 256, "f32", seed=23)
    x, pos, w = d["x"].numpy(), d["pos"].numpy(), d["w"].numpy()
    sf = np.full(16, 8.0, np.float32)
    f32, _ = oracle.reduce_fused_scaled(x, pos, w, None, sf, "f32", "f32")
    f8, _ = oracle.reduce_fused_scaled(x, pos, w, None, sf, "f32", "e4m3")
    assert np.array_equal(f8, oracle.encode(f32, "e4m3"))


# --------------------------------------------------------------------------- #
# int4 weights (skeletons.py w4a8_dequant_gemm; weight-only W4A16)
# --------------------------------------------------------------------------- #

def _pack_int4(q: np.ndarray) -> np.ndarray:
    """Test-side packer, the inverse of the pages' layout: element 2i in the
    low nibble of byte i, element 2i + 1 in the high nibble."""
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    u = u.reshape(*q.shape[:-1], q.shape[-1] // 2, 2)
    return (u[..., 0] | (u[..., 1] << 4)).astype(np.uint8)


def test_unpack_int4_hand_decoded_bytes(oracle):
    with open(os.path.join(GOLDEN, "int4_unpack_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = oracle.unpack_int4(np.array(c["bytes"], np.uint8), len(c["values"]))
        assert got.tolist() == c["values"], c


def test_unpack_int4_inverts_packing_of_every_pair(oracle):
    vals = np.array([(a, b) for a in range(-8, 8) for b in range(-8, 8)], np.int8).reshape(-1)
    packed = _pack_int4(vals)
    assert packed.size == 256 and len(set(packed.tolist())) == 256
    assert np.array_equal(oracle.unpack_int4(packed, vals.size), vals)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_w4_stages_equal_fp_stages_on_the_same_integers(oracle, dtype):
    """Unscaled int4 weights are integers -8..7, exact in fp16 and bf16: the
    int4 stages must give the bits of the plain stages fed those integers."""
    rng = np.random.default_rng(21)
    T, k, E, d_h, d_e = 150, 2, 4, 64, 32
    _, tab = _random_tables(oracle, rng, T, k, E)
    a = _enc(rng.standard_normal((T * k, d_h)) * 0.5, dtype)
    qg = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qu = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qd = rng.integers(-8, 8, (E, d_h, d_e)).astype(np.int8)
    h_q = oracle.grouped_gate_up_silu_w4(a, _pack_int4(qg), _pack_int4(qu), tab, dtype)
    h_f = oracle.grouped_gate_up_silu(a, _enc(qg, dtype), _enc(qu, dtype), tab, dtype)
    assert np.array_equal(h_q, h_f)
    y_q = oracle.grouped_down_w4(h_q, _pack_int4(qd), tab, dtype)
    y_f = oracle.grouped_down(h_q, _enc(qd, dtype), tab, dtype)
    assert np.array_equal(y_q, y_f)
    ones_e = np.ones((E, d_e), np.float32)
    assert np.array_equal(oracle.grouped_gate_up_silu_w4(a, _pack_int4(qg), _pack_int4(qu), tab, dtype,
                                                         s_gate=ones_e, s_up=ones_e), h_q)


def test_w4_stages_integer_closed_form_and_pow2_scales(oracle):
    """fp16, integer operands, gate logits >= 40 (silu(G) = G in fp32):
    h = G * U and y = h Q_down^T exactly; a power-of-two scale per output
    channel scales h (through up) and y exactly."""
    rng = np.random.default_rng(22)
    T, k, E, d_h, d_e = 200, 2, 3, 16, 16
    _, tab = _random_tables(oracle, rng, T, k, E)
    Tk = T * k
    a = rng.integers(0, 2, (Tk, d_h)).astype(np.float32)
    a[:, 0] = 6
    qg = rng.integers(0, 2, (E, d_e, d_h)).astype(np.int8)
    qg[:, :, 0] = 7
    qu = rng.integers(-1, 2, (E, d_e, d_h)).astype(np.int8)
    qu[:, :, 0] = 0
    h = oracle.grouped_gate_up_silu_w4(_bits_f16(a), _pack_int4(qg), _pack_int4(qu), tab, "f16")
    expert_of_row = np.repeat(np.arange(E), tab["group_sizes"])
    ai = a.astype(np.int64)
    G = np.einsum("rj,rnj->rn", ai, qg.astype(np.int64)[expert_of_row])
    U = np.einsum("rj,rnj->rn", ai, qu.astype(np.int64)[expert_of_row])
    assert G.min() >= 40 and np.abs(G * U).max() < 2048
    assert np.array_equal(oracle.decode(h, "f16"), (G * U).astype(np.float32))
    s_up = rng.choice([0.5, 2.0, 4.0], (E, d_e)).astype(np.float32)
    h2 = oracle.grouped_gate_up_silu_w4(_bits_f16(a), _pack_int4(qg), _pack_int4(qu), tab, "f16", s_up=s_up)
    assert np.array_equal(oracle.decode(h2, "f16"), (G * U * s_up[expert_of_row]).astype(np.float32))
    hi = rng.integers(-2, 3, (Tk, d_e)).astype(np.float32)
    qd = rng.integers(-8, 8, (E, d_h, d_e)).astype(np.int8)
    y = oracle.grouped_down_w4(_bits_f16(hi), _pack_int4(qd), tab, "f16")
    Y = np.einsum("rn,ron->ro", hi.astype(np.int64), qd.astype(np.int64)[expert_of_row])
    assert np.abs(Y).max() <= 2048
    assert np.array_equal(oracle.decode(y, "f16"), Y.astype(np.float32))
    s_down = rng.choice([0.25, 1.0, 2.0], (E, d_h)).astype(np.float32)
    y2 = oracle.grouped_down_w4(_bits_f16(hi), _pack_int4(qd), tab, "f16", s_down=s_down)
    assert np.array_equal(oracle.decode(y2, "f16"), (Y * s_down[expert_of_row]).astype(np.float32))


# --------------------------------------------------------------------------- #
# W4A8: int4 weights x int8 activations, int32 sums (skeletons.py w4a8_dequant_gemm)
# --------------------------------------------------------------------------- #

def _int4_by_hand(byte: int, j: int) -> int:
    """Element j % 2 of one packed byte, decoded with Python integers."""
    v = (byte >> 4) if j % 2 else (byte & 15)
    return v - 16 if v & 8 else v


def test_w4a8_brute_force_tiny(oracle):
    """Pure-Python loops over the bytes against the oracle, M != N so that a
    transposed result or a swapped operand fails."""
    rng = np.random.default_rng(31)
    for M, N, K in [(1, 1, 2), (3, 5, 10), (7, 2, 34), (4, 9, 64)]:
        a = rng.integers(-128, 128, (M, K)).astype(np.int8)
        b = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
        ref = [[sum(int(a[m, k]) * _int4_by_hand(int(b[n, k // 2]), k) for k in range(K))
                for m in range(M)] for n in range(N)]
        got = oracle.gemm_w4a8(a, b)
        assert got.shape == (N, M) and got.dtype == np.int32
        assert got.tolist() == ref


def test_w4a8_extreme_closed_forms(oracle):
    """Every element at its extreme: the sums are 1024 K, 889 K and -896 K,
    here up to 2^30 (the int32 accumulator of the pages cannot wrap)."""
    for K in (64, 4096, 1 << 20):
        a = np.full((2, K), -128, np.int8)
        b = np.full((3, K // 2), 0x88, np.uint8)  # every nibble -8
        assert (oracle.gemm_w4a8(a, b) == 1024 * K).all()
        assert (oracle.gemm_w4a8(np.full((1, K), 127, np.int8), np.full((1, K // 2), 0x77, np.uint8))
                == 889 * K).all()
        assert (oracle.gemm_w4a8(a[:1], np.full((2, K // 2), 0x77, np.uint8)) == -896 * K).all()
    with pytest.raises(ValueError):
        oracle.gemm_w4a8(np.zeros((1, (1 << 20) + 2), np.int8), np.zeros((1, (1 << 19) + 1), np.uint8))


def test_w4a8_basis_rows_read_the_weights(oracle):
    """A row that is the unit vector e_k gives column k of the unpacked
    weight (unpack_int4 is pinned on hand-decoded bytes), for every k."""
    rng = np.random.default_rng(32)
    N, K = 6, 32
    b = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    a = np.eye(K, dtype=np.int8) * np.int8(-1)
    q = oracle.unpack_int4(b.reshape(-1), N * K).reshape(N, K).astype(np.int32)
    assert np.array_equal(oracle.gemm_w4a8(a, b), -q)


def test_w4a8_grouped_is_the_dense_product_per_expert(oracle):
    """The grouped form over random dispatch tables equals the dense product
    of each expert's rows with that expert's weight (transposed back)."""
    rng = np.random.default_rng(33)
    T, k, E, N, K = 300, 3, 5, 24, 96
    _, tab = _random_tables(oracle, rng, T, k, E)
    n_rows = T * k
    a = rng.integers(-128, 128, (n_rows, K)).astype(np.int8)
    b = rng.integers(0, 256, (E, N, K // 2)).astype(np.uint8)
    c = oracle.grouped_gemm_w4a8(a, b, tab)
    sizes, offs = tab["group_sizes"], tab["group_offsets"]
    assert sizes.max() > 128  # several blocks per expert
    for g in range(E):
        r0, r1 = int(offs[g]), int(offs[g]) + int(sizes[g])
        if r1 > r0:
            assert np.array_equal(c[r0:r1], oracle.gemm_w4a8(a[r0:r1], b[g]).T)
