"""The int4-weight expert MLP (weight-only W4A16) on the GPU vs the oracle.

Weights are drawn as int4 integers, packed as the pages print the format
(skeletons.py w4a8_dequant_gemm: element j in byte j/2, nibble j%2 from the
low end, two's complement) and repacked on the device by
moe_pack_int4_weights; the oracle reads the pages' format directly."""
import numpy as np
import pytest
import torch

from gpu_helpers import MOE_TOL, assert_bits_equal, assert_close, bits, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def _pack_pages(q: np.ndarray) -> np.ndarray:
    """The pages' int4 layout: element 2i in the low nibble of byte i."""
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    u = u.reshape(*q.shape[:-1], q.shape[-1] // 2, 2)
    return (u[..., 0] | (u[..., 1] << 4)).astype(np.uint8)


def _routing(rng, T, k, E, skew=False):
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


def _tables_to(dev, tab):
    return {n: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for n, v in tab.items()}


@pytest.mark.parametrize("N,R", [(40, 128), (300, 256), (128, 128)])
def test_pack_int4_weights_layout(N, R):
    """The header's layout: [E][ceil(N/R)][K/64][R rows][32 bytes]; inside each
    4-byte word element 2m in nibble m and 2m+1 in nibble m+4, as value + 8;
    rows past N hold zeros (nibbles 8)."""
    dev = require_cuda()
    rng = np.random.default_rng(N + R)
    E, K = 3, 128
    q = rng.integers(-8, 8, (E, N, K)).astype(np.int8)
    got = binding.moe_pack_int4_weights(torch.from_numpy(_pack_pages(q)).to(dev), R).cpu().numpy()
    NT, S = -(-N // R), K // 64
    qp = np.zeros((E, NT * R, K), np.int64)  # padded rows are value 0
    qp[:, :N] = q
    words = (qp.reshape(E, NT, R, S, 8, 8) + 8).transpose(0, 1, 3, 2, 4, 5)  # E, NT, S, R, word, element
    want = np.zeros(words.shape[:-1], np.uint32)
    for e in range(8):
        slot = e // 2 if e % 2 == 0 else 4 + e // 2
        want |= (words[..., e].astype(np.uint32) << np.uint32(4 * slot))
    assert got.size == E * NT * R * K // 2
    assert np.array_equal(got.view(np.uint32), want.reshape(-1))


def _experts(dev, qg, qu, qd, sg, su, sd):
    t = lambda a: None if a is None else torch.from_numpy(a).to(dev)
    return binding.Int4Experts(t(_pack_pages(qg)), t(_pack_pages(qu)), t(_pack_pages(qd)), t(sg), t(su), t(sd))


def _w4_case(dtype, T, k, E, d_h, d_e, skew, seed, scaled):
    rng = np.random.default_rng(seed)
    idx = _routing(rng, T, k, E, skew)
    td = workloads.torch_dtype(dtype)
    x = torch.randn((T, d_h), generator=torch.Generator().manual_seed(seed)).to(td)
    qg = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qu = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qd = rng.integers(-8, 8, (E, d_h, d_e)).astype(np.int8)
    if scaled:
        sg = (rng.uniform(0.5, 1.5, (E, d_e)) / (8 * np.sqrt(d_h))).astype(np.float32)
        su = (rng.uniform(0.5, 1.5, (E, d_e)) / (8 * np.sqrt(d_h))).astype(np.float32)
        sd = (rng.uniform(0.5, 1.5, (E, d_h)) / (8 * np.sqrt(d_e))).astype(np.float32)
    else:
        sg = su = sd = None
    return rng, idx, x, qg, qu, qd, sg, su, sd


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("scaled", [True, False])
@pytest.mark.parametrize("T,k,E,d_h,d_e,skew", [(64, 6, 64, 512, 256, False),
                                                (33, 4, 8, 256, 192, True),
                                                (1, 1, 4, 256, 64, False),
                                                (64, 8, 16, 256, 128, True),
                                                (300, 2, 3, 512, 128, False),   # 200-row experts
                                                (200, 4, 8, 256, 192, True)])   # 65..128-row blocks
def test_w4_mlp_vs_oracle(oracle, dtype, scaled, T, k, E, d_h, d_e, skew):
    """Stage 1 against the oracle; stage 2 against the oracle fed the
    kernel's h (isolates stage 2).  Ragged row counts, a partial N tile
    (d_e = 192), a single token, experts with up to 64 rows, empty experts,
    experts of more than 64 rows (128-row blocks split into two 64-row
    units, and ragged last blocks), with and without per-channel scales."""
    dev = require_cuda()
    rng, idx, x, qg, qu, qd, sg, su, sd = _w4_case(dtype, T, k, E, d_h, d_e, skew, 50 + T + E, scaled)
    if not scaled:
        # keep unscaled int4 sums (|q| <= 8 over d_h, then d_e, inputs) inside the fp16 range
        x = (x.float() * (0.05 if d_h <= 256 else 0.01)).to(x.dtype)
    tab = oracle.build_dispatch(idx, None, E, 128)
    tabd = _tables_to(dev, tab)
    pg, pu, pd = _pack_pages(qg), _pack_pages(qu), _pack_pages(qd)
    ex = _experts(dev, qg, qu, qd, sg, su, sd)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    h, y = binding.moe_grouped_mlp_w4a16(x.to(dev), tabd["sorted_token_idx"], ex, tabd, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    a = oracle.gather_rows(bits(x), tab["sorted_token_idx"], dtype)
    h_ref = oracle.grouped_gate_up_silu_w4(a, pg, pu, tab, dtype, s_gate=sg, s_up=su)
    y_ref = oracle.grouped_down_w4(bits(h), pd, tab, dtype, s_down=sd)
    rtol, atol = MOE_TOL[dtype]
    assert_close(bits(h), h_ref, dtype, rtol, atol, "int4 h")
    assert_close(bits(y), y_ref, dtype, rtol, atol, "int4 y (from the kernel's h)")


def test_w4_mlp_integer_inputs_bit_exact(oracle):
    """fp16, integer operands: gate logits 42 or 43 (silu = identity in
    fp32), |h| <= 344 and |y| <= 688, so every sum is exact and h, y match
    the oracle bit for bit; power-of-two scales keep it exact."""
    dev = require_cuda()
    rng = np.random.default_rng(7)
    T, k, E, d_h, d_e = 64, 4, 8, 256, 128
    idx = _routing(rng, T, k, E)
    tab = oracle.build_dispatch(idx, None, E, 128)
    x = np.zeros((T, d_h), np.float16)
    x[:, 0] = 6
    x[:, 1:10] = rng.integers(0, 2, (T, 9))
    qg = np.zeros((E, d_e, d_h), np.int8)
    qg[:, :, 0] = 7
    qg[:, :, 1] = rng.integers(0, 2, (E, d_e))
    qu = np.zeros((E, d_e, d_h), np.int8)
    qu[:, :, 2:10] = rng.integers(-1, 2, (E, d_e, 8))
    qd = np.zeros((E, d_h, d_e), np.int8)
    qd[:, :, 3:5] = rng.integers(-1, 2, (E, d_h, 2))
    su = rng.choice([0.5, 1.0, 2.0], (E, d_e)).astype(np.float32)
    sd = rng.choice([0.25, 1.0, 2.0], (E, d_h)).astype(np.float32)
    tabd = _tables_to(dev, tab)
    pg, pu, pd = _pack_pages(qg), _pack_pages(qu), _pack_pages(qd)
    ex = _experts(dev, qg, qu, qd, None, su, sd)
    h, y = binding.moe_grouped_mlp_w4a16(torch.from_numpy(x).to(dev), tabd["sorted_token_idx"], ex, tabd)
    torch.cuda.synchronize()
    a = oracle.gather_rows(x.view(np.uint16), tab["sorted_token_idx"], "f16")
    h_ref = oracle.grouped_gate_up_silu_w4(a, pg, pu, tab, "f16", s_up=su)
    y_ref = oracle.grouped_down_w4(h_ref, pd, tab, "f16", s_down=sd)
    assert_bits_equal(bits(h), h_ref, "integer int4 h")
    assert_bits_equal(bits(y), y_ref, "integer int4 y")


def test_w4_forward_decode_size_vs_oracle(oracle):
    """The whole forward with int4 experts at the decode size (T=64, d_hidden
    2048, d_expert 768, 64 experts, top-6, fp16): routing tables bit-exact,
    the output within the MoE tolerance of the oracle's composition."""
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["decode"]
    T, d_h, d_e, E, k = cfg.T, cfg.d_hidden, cfg.d_expert, cfg.n_experts, cfg.top_k
    d = workloads.make_moe_inputs(cfg, device=dev, seed=cfg.seed, with_experts=False)
    rng = np.random.default_rng(8)
    qg = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qu = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qd = rng.integers(-8, 8, (E, d_h, d_e)).astype(np.int8)
    sg = (np.full((E, d_e), 1.0) / (8 * np.sqrt(d_h))).astype(np.float32)
    su = sg.copy()
    sd = (np.full((E, d_h), 1.0) / (8 * np.sqrt(d_e))).astype(np.float32)
    pg, pu, pd = _pack_pages(qg), _pack_pages(qu), _pack_pages(qd)
    ex = _experts(dev, qg, qu, qd, sg, su, sd)
    ws = torch.empty(binding.forward_workspace_bytes(T, d_h, d_e, E, k, d["x"].dtype), dtype=torch.uint8,
                     device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = binding.moe_forward_w4a16(d["x"], d["wg"], d["bias"], ex, k, ws=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    v = binding.forward_workspace_views(ws, T, d_h, d_e, E, k, d["x"].dtype)
    xb, wgb = bits(d["x"]), bits(d["wg"])
    idx, w = oracle.gate_topk(xb, wgb, None, k, "f16")
    assert np.array_equal(v["topk_idx"].cpu().numpy(), idx)
    tab = oracle.build_dispatch(idx, w, E, 128)
    for name in ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx",
                 "sorted_token_idx"):
        assert_bits_equal(v[name].cpu().numpy().reshape(-1), tab[name].reshape(-1), name)
    a = oracle.gather_rows(xb, tab["sorted_token_idx"], "f16")
    h_ref = oracle.grouped_gate_up_silu_w4(a, pg, pu, tab, "f16", s_gate=sg, s_up=su)
    y_ref = oracle.grouped_down_w4(h_ref, pd, tab, "f16", s_down=sd)
    out_ref, _ = oracle.reduce_fused(y_ref, tab["token_topk_to_pos"].reshape(T, k), w, "f16", "f16")
    assert_close(bits(out), out_ref, "f16", *MOE_TOL["f16"], "int4 forward out")


@pytest.mark.parametrize("T,d_h,d_e,E,k", [(300, 256, 128, 8, 2), (1030, 512, 256, 16, 4)])
def test_w4_forward_beyond_64_tokens_vs_oracle(oracle, T, d_h, d_e, E, k):
    """The int4 forward past the decode sizes: experts of 75..260 rows, so
    full 128-row blocks split into two 64-row units and ragged last blocks;
    at T = 1030 the gate takes its tensor-core path.  Routing and tables
    bit-exact, the output within the MoE tolerance of the oracle."""
    dev = require_cuda()
    cfg = workloads.MoEConfig("w4-big", 1, T, d_h, d_e, E, k, "f16", 60 + T)
    d = workloads.make_moe_inputs(cfg, device=dev, with_experts=False)
    rng = np.random.default_rng(T)
    qg = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qu = rng.integers(-8, 8, (E, d_e, d_h)).astype(np.int8)
    qd = rng.integers(-8, 8, (E, d_h, d_e)).astype(np.int8)
    sg = (rng.uniform(0.5, 1.5, (E, d_e)) / (8 * np.sqrt(d_h))).astype(np.float32)
    su = (rng.uniform(0.5, 1.5, (E, d_e)) / (8 * np.sqrt(d_h))).astype(np.float32)
    sd = (rng.uniform(0.5, 1.5, (E, d_h)) / (8 * np.sqrt(d_e))).astype(np.float32)
    pg, pu, pd = _pack_pages(qg), _pack_pages(qu), _pack_pages(qd)
    ex = _experts(dev, qg, qu, qd, sg, su, sd)
    ws = torch.empty(binding.forward_workspace_bytes(T, d_h, d_e, E, k, d["x"].dtype), dtype=torch.uint8,
                     device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = binding.moe_forward_w4a16(d["x"], d["wg"], d["bias"], ex, k, ws=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    v = binding.forward_workspace_views(ws, T, d_h, d_e, E, k, d["x"].dtype)
    xb, wgb = bits(d["x"]), bits(d["wg"])
    idx, w = oracle.gate_topk(xb, wgb, None, k, "f16")
    assert np.array_equal(v["topk_idx"].cpu().numpy(), idx)
    tab = oracle.build_dispatch(idx, w, E, 128)
    assert tab["group_sizes"].max() > 64
    for name in ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx",
                 "sorted_token_idx"):
        assert_bits_equal(v[name].cpu().numpy().reshape(-1), tab[name].reshape(-1), name)
    a = oracle.gather_rows(xb, tab["sorted_token_idx"], "f16")
    h_ref = oracle.grouped_gate_up_silu_w4(a, pg, pu, tab, "f16", s_gate=sg, s_up=su)
    assert_close(bits(v["h"]), h_ref, "f16", *MOE_TOL["f16"], "int4 h")
    y_ref = oracle.grouped_down_w4(bits(v["h"]), pd, tab, "f16", s_down=sd)
    assert_close(bits(v["y"]), y_ref, "f16", *MOE_TOL["f16"], "int4 y (from the kernel's h)")
    y_full = oracle.grouped_down_w4(h_ref, pd, tab, "f16", s_down=sd)
    out_ref, _ = oracle.reduce_fused(y_full, tab["token_topk_to_pos"].reshape(T, k), w, "f16", "f16")
    assert_close(bits(out), out_ref, "f16", *MOE_TOL["f16"], "int4 forward out")


def test_w4_argument_errors():
    dev = require_cuda()
    from oracle import oracle
    rng = np.random.default_rng(9)
    T, k, E = 65, 2, 4
    tab = _tables_to(dev, oracle.build_dispatch(_routing(rng, T, k, E), None, E, 128))
    x = torch.zeros((T, 256), dtype=torch.float16, device=dev)
    z = np.zeros((E, 64, 256), np.int8)
    ex = _experts(dev, z, z, np.zeros((E, 256, 64), np.int8), None, None, None)
    with pytest.raises(binding.MoEError):  # a dtype the int4 kernel does not run
        binding.moe_grouped_mlp_w4a16(x.float(), tab["sorted_token_idx"], ex, tab)
    with pytest.raises(ValueError):  # wrong scale shape
        binding.Int4Experts(*[torch.zeros((E, 64, 128), dtype=torch.uint8, device=dev)] * 2,
                            torch.zeros((E, 256, 32), dtype=torch.uint8, device=dev),
                            s_gate=torch.ones((E, 32), device=dev))
    with pytest.raises(ValueError):  # K not a multiple of 64
        binding.moe_pack_int4_weights(torch.zeros((E, 64, 40), dtype=torch.uint8, device=dev), 128)
