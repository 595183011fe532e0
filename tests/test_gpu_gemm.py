"""The two grouped GEMM stages (tcgen05 kernels) vs the oracle's block walk.

Tables and gathered rows come from the oracle and are copied to the device,
so both sides see the same inputs.  Random inputs are compared within the
MoE tolerances; integer-valued inputs make every fp32 sum exact and are
compared bit for bit."""
import numpy as np
import pytest
import torch

from gpu_helpers import MOE_TOL, assert_bits_equal, assert_close, bits, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def _tables_to(dev, tab):
    return {n: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for n, v in tab.items()}


def _routing(rng, T, k, E, skew=False):
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def _from_bits(a, dtype, dev):
    return workloads.from_numpy_bits(a, dtype).to(dev)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T,k,E,d_h,d_e,skew", [(300, 4, 6, 512, 256, False),
                                                (200, 8, 32, 256, 192, True),
                                                (1, 1, 4, 256, 64, False)])
def test_grouped_gemms_vs_oracle(oracle, dtype, T, k, E, d_h, d_e, skew):
    """Several 128-row blocks per expert with ragged tails, empty experts,
    several N tiles, a partial last N tile (d_e = 192), and a single row."""
    dev = require_cuda()
    rng = np.random.default_rng(T + E + d_e)
    idx = _routing(rng, T, k, E, skew)
    tab = oracle.build_dispatch(idx, None, E, 128)
    td = workloads.torch_dtype(dtype)
    x = torch.randn((T, d_h), generator=torch.Generator().manual_seed(1)).to(td)
    w_gate = (torch.randn((E, d_e, d_h), generator=torch.Generator().manual_seed(2)) / d_h ** 0.5).to(td)
    w_up = (torch.randn((E, d_e, d_h), generator=torch.Generator().manual_seed(3)) / d_h ** 0.5).to(td)
    w_down = (torch.randn((E, d_h, d_e), generator=torch.Generator().manual_seed(4)) / d_e ** 0.5).to(td)
    a = oracle.gather_rows(bits(x), tab["sorted_token_idx"], dtype)
    h_ref = oracle.grouped_gate_up_silu(a, bits(w_gate), bits(w_up), tab, dtype)
    y_ref = oracle.grouped_down(h_ref, bits(w_down), tab, dtype)
    rw = rng.random(T * k).astype(np.float32)
    yw_ref = oracle.grouped_down(h_ref, bits(w_down), tab, dtype, row_weights=rw)

    tabd = _tables_to(dev, tab)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    a_d = _from_bits(a, dtype, dev)
    h = binding.moe_grouped_gate_up_silu(a_d, w_gate.to(dev), w_up.to(dev), tabd, err=err)
    h_in = _from_bits(h_ref, dtype, dev)  # stage 2 from the oracle's h: isolates stage 2
    y = binding.moe_grouped_down(h_in, w_down.to(dev), tabd, err=err)
    yw = binding.moe_grouped_down(h_in, w_down.to(dev), tabd, row_weights=torch.from_numpy(rw).to(dev), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rtol, atol = MOE_TOL[dtype]
    assert_close(bits(h), h_ref, dtype, rtol, atol, "h")
    assert_close(bits(y), y_ref, dtype, rtol, atol, "y")
    assert_close(bits(yw), yw_ref, dtype, rtol, atol, "y with row weights")


def test_grouped_gemms_integer_inputs_bit_exact(oracle):
    """fp16, small integers, gate logits >= 40 (silu(g) = g in fp32): every
    sum is exact, so h = rt(G*U) and y = rt(h W_down^T) match bit for bit."""
    dev = require_cuda()
    rng = np.random.default_rng(11)
    T, k, E, d_h, d_e = 260, 2, 3, 256, 128
    idx = _routing(rng, T, k, E)
    tab = oracle.build_dispatch(idx, None, E, 128)
    x = rng.integers(0, 3, (T, d_h)).astype(np.float16)
    x[:, 0] = 1
    wg = rng.integers(0, 2, (E, d_e, d_h)).astype(np.float16)
    wg[:, :, 0] = 40
    wu = rng.integers(-1, 2, (E, d_e, d_h)).astype(np.float16)
    wd = rng.integers(-1, 2, (E, d_h, d_e)).astype(np.float16)
    a = oracle.gather_rows(x.view(np.uint16), tab["sorted_token_idx"], "f16")
    h_ref = oracle.grouped_gate_up_silu(a, wg.view(np.uint16), wu.view(np.uint16), tab, "f16")
    # exact small-integer h for stage 2 so that y stays exact in fp16 (|y| < 2048)
    h_int = rng.integers(-2, 3, (T * k, d_e)).astype(np.float16).view(np.uint16)
    y_ref = oracle.grouped_down(h_int, wd.view(np.uint16), tab, "f16")
    tabd = _tables_to(dev, tab)
    h = binding.moe_grouped_gate_up_silu(_from_bits(a, "f16", dev), torch.from_numpy(wg).to(dev),
                                         torch.from_numpy(wu).to(dev), tabd)
    y = binding.moe_grouped_down(_from_bits(h_int, "f16", dev), torch.from_numpy(wd).to(dev), tabd)
    torch.cuda.synchronize()
    assert_bits_equal(bits(h), h_ref, "integer h")
    assert_bits_equal(bits(y), y_ref, "integer y")


def test_grouped_gemms_zero_weights():
    dev = require_cuda()
    from oracle import oracle
    rng = np.random.default_rng(12)
    T, k, E, d_h, d_e = 150, 2, 4, 256, 128
    tab = _tables_to(dev, oracle.build_dispatch(_routing(rng, T, k, E), None, E, 128))
    a = torch.randn((T * k, d_h), device=dev).to(torch.bfloat16)
    wg = torch.randn((E, d_e, d_h), device=dev).to(torch.bfloat16)
    zero_u = torch.zeros((E, d_e, d_h), device=dev, dtype=torch.bfloat16)
    h = binding.moe_grouped_gate_up_silu(a, wg, zero_u, tab)
    assert torch.count_nonzero(h.float()) == 0
    y = binding.moe_grouped_down(torch.randn((T * k, d_e), device=dev).to(torch.bfloat16),
                                 torch.zeros((E, d_h, d_e), device=dev, dtype=torch.bfloat16), tab)
    assert torch.count_nonzero(y.float()) == 0


def test_grouped_gemm_rows_outside_the_tables_untouched(oracle):
    """Stage 1 writes only the rows the tables own: with a table built for fewer
    pairs than the buffer holds, the rows past the end keep their canary."""
    dev = require_cuda()
    rng = np.random.default_rng(13)
    T, k, E, d_h, d_e = 100, 2, 5, 256, 128
    tab = oracle.build_dispatch(_routing(rng, T, k, E), None, E, 128)
    n = T * k
    a = torch.randn((n + 40, d_h), device=dev).to(torch.float16)
    h = torch.full((n + 40, d_e), 7.0, device=dev, dtype=torch.float16)
    wg = torch.randn((E, d_e, d_h), device=dev).to(torch.float16) * 0.05
    wu = torch.randn((E, d_e, d_h), device=dev).to(torch.float16) * 0.05
    tabd = _tables_to(dev, tab)
    # the kernel sees n_rows = n: pass views of the first n rows
    binding.moe_grouped_gate_up_silu(a[:n], wg, wu, tabd, h=h[:n])
    torch.cuda.synchronize()
    assert (h[n:].float() == 7.0).all()
    assert not (h[:n].float() == 7.0).all(dim=1).any()


def _mlp_inputs(dtype, T, k, E, d_h, d_e, skew, seed, dev):
    rng = np.random.default_rng(seed)
    idx = _routing(rng, T, k, E, skew)
    td = workloads.torch_dtype(dtype)
    x = torch.randn((T, d_h), generator=torch.Generator().manual_seed(seed + 1)).to(td)
    w_gate = (torch.randn((E, d_e, d_h), generator=torch.Generator().manual_seed(seed + 2)) / d_h ** 0.5).to(td)
    w_up = (torch.randn((E, d_e, d_h), generator=torch.Generator().manual_seed(seed + 3)) / d_h ** 0.5).to(td)
    w_down = (torch.randn((E, d_h, d_e), generator=torch.Generator().manual_seed(seed + 4)) / d_e ** 0.5).to(td)
    return idx, x, w_gate.to(dev), w_up.to(dev), w_down.to(dev), rng


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T,k,E,d_h,d_e,skew", [(300, 4, 6, 512, 256, False),
                                                (200, 8, 32, 256, 192, True),
                                                (1, 1, 4, 256, 64, False),
                                                (1024, 2, 4, 512, 256, False),
                                                (64, 6, 64, 512, 256, False)])
def test_grouped_mlp_equals_two_stages(oracle, dtype, T, k, E, d_h, d_e, skew):
    """Both stages in one launch give bit for bit the h and y of the two
    separate launches (same tiles, same MMA order), and agree with the oracle.
    Covers large experts (stripe-major runs, 512 rows each), mostly-padding
    blocks (swapped MMA), a partial last N tile and a single row."""
    dev = require_cuda()
    idx, x, wg, wu, wd, rng = _mlp_inputs(dtype, T, k, E, d_h, d_e, skew, T + E, dev)
    tab = oracle.build_dispatch(idx, None, E, 128)
    a = oracle.gather_rows(bits(x), tab["sorted_token_idx"], dtype)
    tabd = _tables_to(dev, tab)
    a_d = _from_bits(a, dtype, dev)
    rw = torch.from_numpy(rng.random(T * k).astype(np.float32)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    h2 = binding.moe_grouped_gate_up_silu(a_d, wg, wu, tabd, err=err)
    y2 = binding.moe_grouped_down(h2, wd, tabd, err=err)
    yw2 = binding.moe_grouped_down(h2, wd, tabd, row_weights=rw, err=err)
    h1, y1 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, err=err)
    _, yw1 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, row_weights=rw, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bits_equal(bits(h1), bits(h2), "fused h")
    assert_bits_equal(bits(y1), bits(y2), "fused y")
    assert_bits_equal(bits(yw1), bits(yw2), "fused y with row weights")
    h_ref = oracle.grouped_gate_up_silu(a, bits(wg.cpu()), bits(wu.cpu()), tab, dtype)
    y_ref = oracle.grouped_down(bits(h1), bits(wd.cpu()), tab, dtype)
    rtol, atol = MOE_TOL[dtype]
    assert_close(bits(h1), h_ref, dtype, rtol, atol, "fused h vs oracle")
    assert_close(bits(y1), y_ref, dtype, rtol, atol, "fused y vs oracle (from the kernel's h)")


def test_grouped_mlp_repeated_calls_share_counters(oracle):
    """The per-block counters are cleared by every call: ten calls on one
    counter buffer give the same bits and no error."""
    dev = require_cuda()
    idx, x, wg, wu, wd, _ = _mlp_inputs("bf16", 300, 4, 6, 512, 256, False, 21, dev)
    tab = oracle.build_dispatch(idx, None, 6, 128)
    tabd = _tables_to(dev, tab)
    a_d = _from_bits(oracle.gather_rows(bits(x), tab["sorted_token_idx"], "bf16"), "bf16", dev)
    ready = torch.full((tabd["group_idx_for_bx"].numel() + 1,), 12345, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    _, y0 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, ready=ready, err=err)
    ys = [binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, ready=ready, err=err)[1] for _ in range(10)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for y in ys:
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


def test_grouped_mlp_beyond_the_schedule_table(oracle):
    """More M blocks than the in-kernel schedule orders (1024): tiles run in
    natural block order, padding blocks skipped; sampled rows vs the oracle
    and the fused launch bit-equal to the two separate ones."""
    dev = require_cuda()
    T, k, E, d_h, d_e = 4096, 8, 1024, 256, 64  # 256 + 1024 = 1280 M blocks
    idx, x, wg, wu, wd, rng = _mlp_inputs("f16", T, k, E, d_h, d_e, False, 31, dev)
    tab = oracle.build_dispatch(idx, None, E, 128)
    assert len(tab["group_idx_for_bx"]) > 1024
    tabd = _tables_to(dev, tab)
    a = oracle.gather_rows(bits(x), tab["sorted_token_idx"], "f16")
    a_d = _from_bits(a, "f16", dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    h2 = binding.moe_grouped_gate_up_silu(a_d, wg, wu, tabd, err=err)
    y2 = binding.moe_grouped_down(h2, wd, tabd, err=err)
    h1, y1 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bits_equal(bits(h1), bits(h2), "fused h")
    assert_bits_equal(bits(y1), bits(y2), "fused y")
    sizes, offs = tab["group_sizes"], tab["group_offsets"]
    row_expert = np.repeat(np.arange(E, dtype=np.int32), sizes)
    rows = rng.choice(T * k, size=96, replace=False)
    h_ref = oracle.rows_gate_up_silu(a[rows], row_expert[rows], bits(wg.cpu()), bits(wu.cpu()), "f16")
    y_ref = oracle.rows_down(bits(h1)[rows], row_expert[rows], bits(wd.cpu()), "f16")
    rtol, atol = MOE_TOL["f16"]
    assert_close(bits(h1)[rows], h_ref, "f16", rtol, atol, "sampled h")
    assert_close(bits(y1)[rows], y_ref, "f16", rtol, atol, "sampled y")
    assert offs[-1] + sizes[-1] == T * k


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T,k,E,d_h,d_e,skew", [(64, 6, 64, 512, 256, False),
                                                (33, 4, 8, 256, 192, True),
                                                (1, 1, 4, 256, 64, False),
                                                (64, 8, 16, 256, 128, True),
                                                (300, 8, 16, 256, 128, True),
                                                (517, 2, 4, 512, 192, False)])
def test_grouped_mlp_gathering_form_equals_gathered_rows(oracle, dtype, T, k, E, d_h, d_e, skew):
    """Stage 1 fetching its rows from x by sorted_token_idx (four-row TMA
    gathers, one per producer lane) gives the bits of the pre-gathered rows;
    covers ragged row counts (np rounded up to 16 over a small block's rows),
    a single token, full 128-row tiles and ragged last blocks of experts with
    hundreds of rows, and empty experts."""
    dev = require_cuda()
    idx, x, wg, wu, wd, _ = _mlp_inputs(dtype, T, k, E, d_h, d_e, skew, 40 + T + E, dev)
    tab = oracle.build_dispatch(idx, None, E, 128)
    if T > 64:
        assert int(np.max(tab["group_sizes"])) > 128  # full tiles and more than one block per expert
    tabd = _tables_to(dev, tab)
    a_d = _from_bits(oracle.gather_rows(bits(x), tab["sorted_token_idx"], dtype), dtype, dev)
    x_d = x.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    h1, y1 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, err=err)
    h2, y2 = binding.moe_grouped_mlp(None, wg, wu, wd, tabd, err=err, x=x_d,
                                     sorted_token_idx=tabd["sorted_token_idx"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bits_equal(bits(h2), bits(h1), "gathered h")
    assert_bits_equal(bits(y2), bits(y1), "gathered y")


@pytest.mark.parametrize("grid", [1, 7, 76, 304])
@pytest.mark.parametrize("case", ["decode", "prefill-1024x32"])
def test_expert_mlp_progress_does_not_need_a_resident_grid(oracle, monkeypatch, case, grid):
    """The persistent expert MLP takes every tile, its first included, from a
    shared counter, so a stage-2 tile never waits on a stage-1 tile that no
    running CTA holds.  Run on 1, 7 or 76 CTAs, and on 304 CTAs (twice the
    SMs: the second half can only start once CTAs of the first half have
    exited), the forward completes with no timed-out wait and gives the same
    bits as the launch with one CTA per SM (tiles are computed whole by one
    CTA, in a fixed order, so the grid cannot change a result).  Cases: the
    decode forward (few-token launch, rows gathered inside) and a 1024-token
    prefill-shaped forward over 32 experts (full 128-row tiles, large experts'
    stripe runs); the decode output is also checked against the oracle."""
    import dataclasses
    dev = require_cuda()
    if case == "decode":
        cfg = workloads.MOE_CONFIGS["decode"]
    else:
        cfg = dataclasses.replace(workloads.MOE_CONFIGS["prefill"], batch=1, seq=1024, n_experts=32)
    d = workloads.make_moe_inputs(cfg, device=dev)

    def run():
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        out = binding.moe_forward(d["x"], d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"],
                                  cfg.top_k, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error flag {int(err.item())}"
        return bits(out)

    monkeypatch.delenv("MOE_MLP_GRID", raising=False)
    want = run()
    monkeypatch.setenv("MOE_MLP_GRID", str(grid))
    got = run()
    assert_bits_equal(got, want, f"{case}, {grid} CTAs vs one per SM")
    if case == "decode":
        nb = {n: (bits(v) if v is not None else None) for n, v in d.items()}
        ref = oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                                 cfg.top_k, cfg.dtype)
        assert_close(got, ref["out"], cfg.dtype, *MOE_TOL[cfg.dtype], "decode out")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d_h,d_e", [(512, 256), (1024, 512)])
def test_expert_mlp_on_sm_pairs_matches_one_sm_form_and_oracle(oracle, monkeypatch, dtype, d_h, d_e):
    """The many-row expert MLP runs on pairs of SMs (tcgen05 cta_group::2):
    experts with more than 64 rows in 256-row units (one or two per pair of
    M blocks, the last one ragged), smaller experts swapped (their rows the
    MMA's N, split between the two SMs).  Expert sizes chosen to hit every
    boundary: 1, 15, 16, 17, 63, 64 rows (swapped), 65, 128, 255, 256, 257,
    511, 512, 700 rows (units of 256), an empty expert.  The pair launch gives
    the bits of the one-SM launch (and of its gathering form, rows read from
    the tokens by index), and h and y agree with the oracle."""
    dev = require_cuda()
    sizes = [1, 15, 0, 16, 17, 63, 64, 65, 128, 255, 256, 257, 511, 512, 700]
    E = len(sizes)
    idx = np.repeat(np.arange(E, dtype=np.int32), sizes)
    rng = np.random.default_rng(d_h + d_e)
    idx = idx[rng.permutation(idx.size)].reshape(-1, 1)  # one slot per token, tokens shuffled
    T = idx.shape[0]
    td = workloads.torch_dtype(dtype)
    g = torch.Generator().manual_seed(d_e)
    x = torch.randn((T, d_h), generator=g).to(td)
    wg = (torch.randn((E, d_e, d_h), generator=g) / d_h ** 0.5).to(td).to(dev)
    wu = (torch.randn((E, d_e, d_h), generator=g) / d_h ** 0.5).to(td).to(dev)
    wd = (torch.randn((E, d_h, d_e), generator=g) / d_e ** 0.5).to(td).to(dev)
    tab = oracle.build_dispatch(idx, None, E, 128)
    assert list(tab["group_sizes"]) == sizes
    a = oracle.gather_rows(bits(x), tab["sorted_token_idx"], dtype)
    tabd = _tables_to(dev, tab)
    a_d = _from_bits(a, dtype, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    monkeypatch.setenv("MOE_MLP_PAIRS", "0")
    h1, y1 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, err=err)
    torch.cuda.synchronize()
    monkeypatch.delenv("MOE_MLP_PAIRS")
    h2, y2 = binding.moe_grouped_mlp(a_d, wg, wu, wd, tabd, err=err)
    # the gathering form (rows read from x by index; the one-SM kernel's)
    h3, y3 = binding.moe_grouped_mlp(None, wg, wu, wd, tabd, err=err, x=x.to(dev),
                                     sorted_token_idx=tabd["sorted_token_idx"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bits_equal(bits(h2), bits(h1), "pair h vs one-SM h")
    assert_bits_equal(bits(y2), bits(y1), "pair y vs one-SM y")
    assert_bits_equal(bits(h3), bits(h1), "gathering-form h vs one-SM h")
    assert_bits_equal(bits(y3), bits(y1), "gathering-form y vs one-SM y")
    h_ref = oracle.grouped_gate_up_silu(a, bits(wg.cpu()), bits(wu.cpu()), tab, dtype)
    y_ref = oracle.grouped_down(h_ref, bits(wd.cpu()), tab, dtype)
    rtol, atol = MOE_TOL[dtype]
    assert_close(bits(h2), h_ref, dtype, rtol, atol, "pair h vs oracle")
    assert_close(bits(y2), y_ref, dtype, rtol, atol, "pair y vs oracle")
