"""Writes past the end (or before the start) of an output or a workspace.

Every output and workspace each entry point writes is placed between two
4 KiB guard bands of a byte pattern; after the call the bands must hold the
pattern still.  The shapes are ragged (tokens, experts, rows per expert and
columns that are not multiples of the kernels' tiles) so the edge masks of
the gate, the dispatch, the gather, both GEMM stages (swapped and full
tiles), the combine (both kernels) and the forward are the ones exercised.
No index here is out of range for the buffers themselves: the check is that
no kernel writes outside them."""
import numpy as np
import pytest
import torch

from gpu_helpers import require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side; keeps the view 256-byte aligned
PATTERN = 0xA5


class Guards:
    """Buffers placed between two guard bands of PATTERN bytes."""

    def __init__(self, dev):
        self.dev = dev
        self.items = []

    def empty(self, shape, dtype, name):
        shape = tuple(int(s) for s in shape)
        nbytes = torch.empty((), dtype=dtype).element_size()
        for s in shape:
            nbytes *= s
        assert nbytes > 0, name
        raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=self.dev)
        self.items.append((name, raw, nbytes))
        return raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def zeros(self, shape, dtype, name):
        t = self.empty(shape, dtype, name)
        t.zero_()
        return t

    def check(self):
        torch.cuda.synchronize()
        for name, raw, nbytes in self.items:
            head = int((raw[:GUARD] != PATTERN).sum())
            tail = int((raw[GUARD + nbytes:] != PATTERN).sum())
            assert head == 0 and tail == 0, (
                f"{name}: {head} guard bytes before and {tail} after the buffer were overwritten")


def _dispatch_out(G, T, k, E):
    mb = binding.num_m_blocks(T, k, E)
    i32 = torch.int32
    return dict(group_sizes=G.empty((E,), i32, "group_sizes"),
                group_offsets=G.empty((E,), i32, "group_offsets"),
                group_padded_offsets=G.empty((E,), i32, "group_padded_offsets"),
                group_idx_for_bx=G.empty((mb,), i32, "group_idx_for_bx"),
                sorted_token_idx=G.empty((T * k,), i32, "sorted_token_idx"),
                sorted_row_weight=G.empty((T * k,), torch.float32, "sorted_row_weight"),
                token_topk_to_pos=G.empty((T, k), i32, "token_topk_to_pos"))


@pytest.mark.parametrize("T,d_h,E,k,dtype", [(601, 512, 100, 4, "f16"),   # 16 x 16 CTAs, ragged
                                             (37, 512, 40, 3, "bf16"),    # top-k fused, E <= 64
                                             (5, 256, 72, 8, "f16"),      # one-warp CTAs
                                             (700, 768, 64, 6, "bf16"),   # 4 tokens per fused CTA
                                             (1100, 512, 100, 4, "f16")])  # tensor-core gate, ragged
def test_routing_dispatch_gather_stay_inside(T, d_h, E, k, dtype):
    dev = require_cuda()
    G = Guards(dev)
    td = workloads.torch_dtype(dtype)
    g = torch.Generator(device=dev).manual_seed(T * 7 + E)
    x = torch.randn((T, d_h), generator=g, device=dev).to(td)
    wg = (torch.randn((E, d_h), generator=g, device=dev) / d_h ** 0.5).to(td)
    idx = G.empty((T, k), torch.int32, "topk_idx")
    w = G.empty((T, k), torch.float32, "topk_w")
    ws = G.empty((int(binding.lib().moe_gate_topk_workspace_bytes(T, E)),), torch.uint8, "gate workspace")
    binding.moe_gate_topk(x, wg, None, k, topk_idx=idx, topk_w=w, ws=ws)
    need = int(binding.lib().moe_build_dispatch_workspace_bytes(T, k, E))
    dws = G.empty((max(need, 16),), torch.uint8, "dispatch workspace")
    tab = binding.moe_build_dispatch(idx, w, E, out=_dispatch_out(G, T, k, E), ws=dws)
    tab2 = binding.moe_build_dispatch_noalloc(idx, w, E, out=_dispatch_out(G, T, k, E))
    a = G.empty((T * k, d_h), td, "gathered rows")
    binding.moe_gather_rows(x, tab["sorted_token_idx"], out=a)
    a2 = G.empty((T * k, d_h), td, "rows gathered in token order")
    binding.moe_gather_rows_by_token(x, tab["token_topk_to_pos"], T * k, out=a2)
    G.check()
    for name in tab:
        assert torch.equal(tab[name], tab2[name]), name
    assert torch.equal(a, a2)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T,E,k,d_h,d_e", [(150, 3, 2, 256, 192),   # full (non-swapped) tiles, partial N
                                           (61, 5, 3, 512, 128),    # swapped tiles only
                                           (97, 9, 4, 256, 320),
                                           (300, 6, 3, 512, 256),   # SM-pair kernel: 256-row units
                                           (90, 24, 2, 1024, 512)])  # SM-pair kernel: mostly swapped units
def test_expert_gemms_stay_inside(dtype, T, E, k, d_h, d_e):
    dev = require_cuda()
    cfg = workloads.MoEConfig("guard", 1, T, d_h, d_e, E, k, dtype, 21 + T)
    d = workloads.make_moe_inputs(cfg, device=dev)
    td = workloads.torch_dtype(dtype)
    idx, w = binding.moe_gate_topk(d["x"], d["wg"], None, k)
    tab = binding.moe_build_dispatch(idx, w, E)
    a = binding.moe_gather_rows(d["x"], tab["sorted_token_idx"])
    Tk = T * k
    mb = tab["group_idx_for_bx"].numel()
    G = Guards(dev)
    err = G.zeros((1,), torch.int32, "err")
    h = G.empty((Tk, d_e), td, "h (gate/up)")
    binding.moe_grouped_gate_up_silu(a, d["w_gate"], d["w_up"], tab, h=h, err=err)
    y = G.empty((Tk, d_h), td, "y (down)")
    binding.moe_grouped_down(h, d["w_down"], tab, row_weights=tab["sorted_row_weight"], y=y, err=err)
    h2 = G.empty((Tk, d_e), td, "h (expert MLP)")
    y2 = G.empty((Tk, d_h), td, "y (expert MLP)")
    ready = G.empty((mb + 1,), torch.int32, "ready counters")
    binding.moe_grouped_mlp(a, d["w_gate"], d["w_up"], d["w_down"], tab, h=h2, y=y2, ready=ready, err=err)
    h3 = G.empty((Tk, d_e), td, "h (expert MLP, gathering)")
    y3 = G.empty((Tk, d_h), td, "y (expert MLP, gathering)")
    ready3 = G.empty((mb + 1,), torch.int32, "ready counters (gathering)")
    binding.moe_grouped_mlp(None, d["w_gate"], d["w_up"], d["w_down"], tab, h=h3, y=y3, ready=ready3,
                            err=err, x=d["x"], sorted_token_idx=tab["sorted_token_idx"])
    G.check()
    assert int(err.item()) == 0
    assert torch.equal(h2, h3) and torch.equal(y2, y3)


@pytest.mark.parametrize("T,K,H,in_dt,out_dt", [(33, 8, 768, "bf16", "bf16"), (7, 40, 256, "f16", "f16"),
                                                (19, 3, 512, "f32", "bf16"), (1, 8, 256, "f32", "f32")])
def test_combine_stays_inside(T, K, H, in_dt, out_dt):
    dev = require_cuda()
    r = workloads.make_reduce_inputs(T, K, H, in_dt, 5, device=dev, scales=True)
    G = Guards(dev)
    err = G.zeros((1,), torch.int32, "err")
    out = G.empty((T, H), workloads.torch_dtype(out_dt), "combine out")
    binding.moe_reduce_fused(r["x"], r["pos"], r["w"], out=out, err=err)
    out8 = G.empty((T, H), torch.float8_e4m3fn, "scaled combine e4m3 out")
    binding.moe_reduce_fused_scaled(r["x"], r["pos"], r["w"], x_sf=r["x_sf"], sf=r["sf"], out=out8, err=err)
    G.check()
    assert int(err.item()) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T,E,k,d_h,d_e", [(150, 3, 2, 256, 192), (61, 5, 3, 512, 128), (65, 8, 2, 256, 128),
                                           (1100, 20, 4, 512, 256)])  # tensor-core gate, SM-pair expert MLP
def test_forward_stays_inside_its_workspace(dtype, T, E, k, d_h, d_e):
    dev = require_cuda()
    cfg = workloads.MoEConfig("guard", 1, T, d_h, d_e, E, k, dtype, 40 + T)
    d = workloads.make_moe_inputs(cfg, device=dev)
    td = workloads.torch_dtype(dtype)
    G = Guards(dev)
    ws = G.empty((binding.forward_workspace_bytes(T, d_h, d_e, E, k, td),), torch.uint8, "forward workspace")
    out = G.empty((T, d_h), td, "forward out")
    err = G.zeros((1,), torch.int32, "err")
    binding.moe_forward(d["x"], d["wg"], None, d["w_gate"], d["w_up"], d["w_down"], k, ws=ws, out=out, err=err)
    G.check()
    assert int(err.item()) == 0
    ref = binding.moe_forward(d["x"], d["wg"], None, d["w_gate"], d["w_up"], d["w_down"], k)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_int4_forward_and_copy_stay_inside():
    dev = require_cuda()
    T, k, E, d_h, d_e = 33, 4, 8, 256, 192
    rng = np.random.default_rng(3)

    def u8(shape):
        return torch.from_numpy(rng.integers(0, 256, shape, dtype=np.uint8)).to(dev)

    def scale(shape, fan_in):
        return torch.from_numpy((rng.uniform(0.5, 1.5, shape) / (8 * np.sqrt(fan_in))).astype(np.float32)).to(dev)

    ex = binding.Int4Experts(u8((E, d_e, d_h // 2)), u8((E, d_e, d_h // 2)), u8((E, d_h, d_e // 2)),
                             scale((E, d_e), d_h), scale((E, d_e), d_h), scale((E, d_h), d_e))
    g = torch.Generator(device=dev).manual_seed(9)
    x = torch.randn((T, d_h), generator=g, device=dev).to(torch.float16)
    wg = (torch.randn((E, d_h), generator=g, device=dev) / d_h ** 0.5).to(torch.float16)
    G = Guards(dev)
    ws = G.empty((binding.forward_workspace_bytes(T, d_h, d_e, E, k, torch.float16),), torch.uint8,
                 "int4 forward workspace")
    out = G.empty((T, d_h), torch.float16, "int4 forward out")
    err = G.zeros((1,), torch.int32, "err")
    binding.moe_forward_w4a16(x, wg, None, ex, k, ws=ws, out=out, err=err)
    src = torch.arange(4096 + 48, dtype=torch.int32, device=dev).to(torch.uint8)
    dst = G.empty((4096 + 48,), torch.uint8, "copy dst")
    binding.moe_copy(src, dst)
    G.check()
    assert int(err.item()) == 0
    assert torch.equal(dst, src)


@pytest.mark.parametrize("M,N,K", [(5, 300, 1984), (1, 3584, 18944), (64, 255, 320)])
def test_w4a8_stays_inside(oracle, M, N, K):
    """The W4A8 GEMM (stored and K-split atomic forms) and its grouped form:
    output and workspace between guard bands."""
    dev = require_cuda()
    d = workloads.make_w4a8_inputs(M, N, K, seed=8)
    bp = binding.moe_pack_int4_weights(d["b"].to(dev), 256)
    G = Guards(dev)
    err = G.zeros((1,), torch.int32, "err")
    ct = G.empty((N, M), torch.int32, "w4a8 Ct")
    ws = G.empty((binding.lib().moe_gemm_w4a8_workspace_bytes(M, K),), torch.uint8, "w4a8 workspace")
    binding.moe_gemm_w4a8(d["a"].to(dev), bp, N, out=ct, ws=ws, err=err)
    E = 3
    rng = np.random.default_rng(M + N)
    idx = np.stack([rng.permutation(E)[:2] for _ in range(M)]).astype(np.int32)
    tab = oracle.build_dispatch(idx, None, E, 128)
    tabd = {n: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for n, v in tab.items()}
    dg = workloads.make_w4a8_inputs(M, N, K, seed=9, E=E)
    bpg = binding.moe_pack_int4_weights(dg["b"].to(dev), 256)
    n_rows, mb = 2 * M, tab["group_idx_for_bx"].size
    c = G.empty((n_rows, N), torch.int32, "grouped w4a8 C")
    wsg = G.empty((binding.lib().moe_grouped_gemm_w4a8_workspace_bytes(n_rows, K, mb),), torch.uint8,
                  "grouped w4a8 workspace")
    binding.moe_grouped_gemm_w4a8(dg["a"].to(dev), tabd["sorted_token_idx"], bpg, tabd, N, E, out=c, ws=wsg,
                                  err=err)
    G.check()
    assert int(err.item()) == 0
    assert np.array_equal(ct.cpu().numpy(), oracle.gemm_w4a8(d["a"].numpy(), d["b"][0].numpy()))
    rows = dg["a"].numpy()[tab["sorted_token_idx"]]
    assert np.array_equal(c.cpu().numpy(), oracle.grouped_gemm_w4a8(rows, dg["b"].numpy(), tab))


@pytest.mark.parametrize("T,k,E", [(300, 4, 20),    # one-CTA dispatch
                                   (5000, 8, 64)])  # histogram / scan / scatter kernels
def test_dispatch_drops_ids_outside_the_experts(oracle, T, k, E):
    """A pair whose expert id lies outside [0, E) is dropped: counted nowhere,
    given no row, its token_topk_to_pos entry left as it was.  The valid
    pairs get the tables the oracle gives when the dropped ones are sent to
    one extra expert E instead (whose rows come after every other expert's),
    and nothing is written outside the outputs."""
    dev = require_cuda()
    rng = np.random.default_rng(T + E)
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    bad = rng.random((T, k)) < 0.05
    idx[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -1, E + 3).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    G = Guards(dev)
    out = _dispatch_out(G, T, k, E)
    out["token_topk_to_pos"].fill_(-7)
    need = int(binding.lib().moe_build_dispatch_workspace_bytes(T, k, E))
    dws = G.empty((max(need, 16),), torch.uint8, "dispatch workspace")
    binding.moe_build_dispatch(torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev), E, out=out, ws=dws)
    G.check()
    ref = oracle.build_dispatch(np.where(bad, E, idx).astype(np.int32), w, E + 1)
    got = {n: t.cpu().numpy() for n, t in out.items()}
    n_valid = int((~bad).sum())
    for name in ("group_sizes", "group_offsets", "group_padded_offsets"):
        assert np.array_equal(got[name], ref[name][:E]), name
    mb = got["group_idx_for_bx"].size
    assert np.array_equal(got["group_idx_for_bx"], np.minimum(ref["group_idx_for_bx"][:mb], E - 1))
    assert np.array_equal(got["sorted_token_idx"][:n_valid], ref["sorted_token_idx"][:n_valid])
    assert np.array_equal(got["sorted_row_weight"][:n_valid].view(np.uint32),
                          ref["sorted_row_weight"][:n_valid].view(np.uint32))
    pos = got["token_topk_to_pos"]
    assert np.array_equal(pos[~bad], ref["token_topk_to_pos"][~bad])
    assert (pos[bad] == -7).all()
