"""The whole routed forward (moe_forward) vs the oracle on the three MoE
workloads.  The small workloads are compared on every output; the prefill
workload (T=4096, d_hidden 7168, d_expert 2048, 256 experts, top-8, bf16) at
full size and in the benchmark's launch configuration on its routing and
tables (all, bit for bit), on every h / y row of three experts (the largest,
a mid-sized one, a small one) and on 256 output tokens that the oracle
computes one by one by the dense per-token brute force."""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_helpers import (MOE_TOL, assert_bits_equal, assert_close, bits, check_gate_logits,
                         gate_uses_tensor_cores, require_cuda)
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

TABLES = ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx",
          "sorted_token_idx", "token_topk_to_pos")


def _run_forward(d, cfg, T=None):
    dev = d["x"].device
    T = d["x"].shape[0] if T is None else T
    ws = torch.empty(binding.forward_workspace_bytes(T, cfg.d_hidden, cfg.d_expert, cfg.n_experts,
                                                     cfg.top_k, d["x"].dtype), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = binding.moe_forward(d["x"], d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"],
                              cfg.top_k, ws=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    views = binding.forward_workspace_views(ws, T, cfg.d_hidden, cfg.d_expert, cfg.n_experts,
                                            cfg.top_k, d["x"].dtype)
    return out, views


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_forward_small_workloads(oracle, name):
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS[name]
    d = workloads.make_moe_inputs(cfg, device=dev)
    out, views = _run_forward(d, cfg)
    nb = {n: (bits(v) if v is not None else None) for n, v in d.items()}
    ref = oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                             cfg.top_k, cfg.dtype)
    assert_bits_equal(views["topk_idx"].cpu().numpy(), ref["topk_idx"], "topk_idx")
    for n in TABLES:
        assert_bits_equal(views[n].cpu().numpy().reshape(ref[n].shape), ref[n], n)
    rtol, atol = MOE_TOL[cfg.dtype]
    assert np.allclose(views["topk_w"].cpu().numpy(), ref["topk_w"], rtol=1e-5, atol=1e-7)
    assert_close(bits(views["h"]), ref["h"], cfg.dtype, rtol, atol, "h")
    assert_close(bits(views["y"]), ref["y"], cfg.dtype, rtol, atol, "y")
    assert_close(bits(out), ref["out"], cfg.dtype, rtol, atol, "out")


def test_forward_repeat_is_stateless():
    """Two calls on the same input give the same bits (nothing carries over
    from call to call)."""
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["tiny"]
    d = workloads.make_moe_inputs(cfg, device=dev)
    o1, _ = _run_forward(d, cfg)
    o1 = o1.clone()
    o2, _ = _run_forward(d, cfg)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("T", [1, 5, 200])
def test_forward_token_counts(oracle, T):
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["tiny"]
    d = workloads.make_moe_inputs(cfg, device=dev, T=T)
    out, views = _run_forward(d, cfg)
    nb = {n: (bits(v) if v is not None else None) for n, v in d.items()}
    ref = oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                             cfg.top_k, cfg.dtype)
    for n in TABLES:
        assert_bits_equal(views[n].cpu().numpy().reshape(ref[n].shape), ref[n], n)
    assert_close(bits(out), ref["out"], cfg.dtype, *MOE_TOL[cfg.dtype], "out")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("T,E,k,d_e", [(64, 8, 2, 128), (65, 8, 2, 128), (40, 1, 1, 128), (300, 1, 1, 64),
                                        (33, 8, 8, 128), (130, 4, 4, 192)])
def test_forward_boundary_and_degenerate_shapes(oracle, dtype, T, E, k, d_e):
    """T = 64 and 65 (the largest launch that gathers its rows inside the
    expert MLP, and the smallest that runs the gather kernel first); a single
    expert (every token's only slot on expert 0: 40 rows in one ragged block,
    or 300 rows in two full blocks and a ragged one, each followed by the
    trailing block the tables add, with weight exactly 1); every
    token on every expert (k = E); a d_expert with a partial last stage-1 tile
    (192); fp16 and bf16.  Routing and tables bit for bit, the output within
    the dtype's tolerance."""
    dev = require_cuda()
    cfg = dataclasses.replace(workloads.MOE_CONFIGS["tiny"], batch=1, seq=T, n_experts=E, top_k=k,
                              d_expert=d_e, dtype=dtype)
    d = workloads.make_moe_inputs(cfg, device=dev)
    out, views = _run_forward(d, cfg)
    nb = {n: (bits(v) if v is not None else None) for n, v in d.items()}
    ref = oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                             cfg.top_k, cfg.dtype)
    assert_bits_equal(views["topk_idx"].cpu().numpy(), ref["topk_idx"], "topk_idx")
    for n in TABLES:
        assert_bits_equal(views[n].cpu().numpy().reshape(ref[n].shape), ref[n], n)
    if k == E:
        assert (ref["group_sizes"] == T).all()
    if E == 1:
        assert np.array_equal(views["topk_w"].cpu().numpy(), np.ones((T, 1), np.float32))
    rtol, atol = MOE_TOL[cfg.dtype]
    assert_close(bits(views["y"]), ref["y"], cfg.dtype, rtol, atol, "y")
    assert_close(bits(out), ref["out"], cfg.dtype, rtol, atol, "out")


def test_forward_with_no_tokens_is_a_no_op():
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["tiny"]
    d = workloads.make_moe_inputs(cfg, device=dev, T=1)
    x0 = d["x"][:0]
    out = binding.moe_forward(x0, d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, cfg.d_hidden)


@pytest.mark.parametrize("host_io", [False, True])
def test_forward_graph_replay_matches_eager(host_io):
    """moe_forward captured into a CUDA graph (binding.ForwardGraph) and
    replayed on new tokens gives the same bits as eager calls."""
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["decode"]
    d = workloads.make_moe_inputs(cfg, device=dev)
    fg = binding.ForwardGraph(d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k,
                              cfg.T, host_io=host_io)
    for seed in (1, 2):
        x = workloads.make_tokens(cfg, cfg.T, device=dev, seed=seed)
        if host_io:
            fg.x_host.copy_(x.cpu())
        else:
            fg.x.copy_(x)
        torch.cuda.synchronize()
        fg.replay()
        torch.cuda.synchronize()
        got = fg.out_host if host_io else fg.out
        want = binding.moe_forward(x, d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu().view(torch.int16), want.cpu().view(torch.int16))
        assert int(fg.err.item()) == 0


def test_forward_output_into_pinned_host_memory():
    """moe_forward with `out` a pinned host tensor: the combine stores the
    result straight into host memory, the same bits as a device `out`."""
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["decode"]
    d = workloads.make_moe_inputs(cfg, device=dev)
    want = binding.moe_forward(d["x"], d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k)
    host = torch.full((cfg.T, cfg.d_hidden), float("nan"), dtype=want.dtype).pin_memory()
    got = binding.moe_forward(d["x"], d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k,
                              out=host)
    torch.cuda.synchronize()
    assert got is host
    assert torch.equal(host.view(torch.int16), want.cpu().view(torch.int16))
    with pytest.raises(ValueError):
        binding.moe_forward(d["x"], d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k,
                            out=torch.empty((cfg.T, cfg.d_hidden), dtype=want.dtype))  # pageable


@pytest.mark.parametrize("nbytes", [16, 4096, 262144, (1 << 22) + 48])
def test_copy_kernel_host_and_device(nbytes):
    """moe_copy moves bytes pinned host -> device, device -> pinned host and
    device -> device, bit for bit, including a size that is not a whole
    number of passes of the grid."""
    dev = require_cuda()
    n = nbytes // 2
    src_h = torch.randint(-32768, 32767, (n,), dtype=torch.int16).pin_memory()
    d1 = torch.empty(n, dtype=torch.int16, device=dev)
    binding.moe_copy(src_h, d1)
    d2 = torch.empty(n, dtype=torch.int16, device=dev)
    binding.moe_copy(d1, d2)
    back = torch.empty(n, dtype=torch.int16).pin_memory()
    binding.moe_copy(d2, back)
    torch.cuda.synchronize()
    assert torch.equal(back, src_h)
    assert torch.equal(d1.cpu(), src_h)


def _compact(w, experts):
    """The listed experts' slices of a stacked weight, on the host."""
    idx = torch.as_tensor(experts, dtype=torch.long, device=w.device)
    return bits(w.index_select(0, idx))


@pytest.mark.slow
def test_forward_prefill_full_size(oracle):
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["prefill"]
    d = workloads.make_moe_inputs(cfg, device=dev)
    out, views = _run_forward(d, cfg)
    k = cfg.top_k
    # routing: all tokens, bit for bit (the logits as check_gate_logits says)
    ref_logits = oracle.gate_logits(bits(d["x"]), bits(d["wg"]), d["bias"].cpu().numpy(), cfg.dtype)
    ref_idx, ref_w = oracle.topk_softmax(ref_logits, k)
    assert_bits_equal(views["topk_idx"].cpu().numpy(), ref_idx, "topk_idx")
    check_gate_logits(views["logits"].cpu().numpy(), ref_logits, ref_idx, bits(d["x"]), bits(d["wg"]),
                      d["bias"].cpu().numpy(), cfg.dtype,
                      gate_uses_tensor_cores(cfg.T, cfg.d_hidden, cfg.n_experts))
    assert np.allclose(views["topk_w"].cpu().numpy(), ref_w, rtol=1e-5, atol=1e-7)
    tab = oracle.build_dispatch(ref_idx, ref_w, cfg.n_experts, 128)
    for n in TABLES:
        assert_bits_equal(views[n].cpu().numpy().reshape(tab[n].shape), tab[n], n)
    sizes = tab["group_sizes"]
    assert sizes.max() > 1000 and (sizes == 0).any(), "the Zipf bias should skew the loads"

    # every h and y row of three experts: the largest (> 1000 rows: many full
    # 128-row tiles, walked stripe by stripe, and a ragged last block), a
    # mid-sized one (several blocks and a ragged tail) and a small one whose
    # single block runs as a swapped tile (<= 64 rows)
    offs = tab["group_offsets"]
    big = int(np.argmax(sizes))
    mids = [int(e) for e in np.argsort(sizes) if 200 <= sizes[e] <= 900 and sizes[e] % 128 != 0]
    smalls = [int(e) for e in np.argsort(sizes) if 16 < sizes[e] <= 64]
    assert mids and smalls, "the Zipf routing should give mid-sized and small experts"
    experts = [big, mids[len(mids) // 2], smalls[-1]]
    rows = np.concatenate([np.arange(offs[e], offs[e] + sizes[e]) for e in experts]).astype(np.int64)
    re = np.concatenate([np.full(sizes[e], i, np.int32) for i, e in enumerate(experts)])
    x_h = bits(d["x"])
    a_rows = x_h[tab["sorted_token_idx"][rows]]
    h_ref = oracle.rows_gate_up_silu(a_rows, re, _compact(d["w_gate"], experts),
                                     _compact(d["w_up"], experts), cfg.dtype)
    y_ref = oracle.rows_down(h_ref, re, _compact(d["w_down"], experts), cfg.dtype)
    rtol, atol = MOE_TOL[cfg.dtype]
    rows_t = torch.from_numpy(rows).to(dev)
    assert_close(bits(views["h"].index_select(0, rows_t)), h_ref, cfg.dtype, rtol, atol,
                 f"h rows of experts {experts} ({[int(sizes[e]) for e in experts]} rows)")
    assert_close(bits(views["y"].index_select(0, rows_t)), y_ref, cfg.dtype, rtol, atol,
                 f"y rows of experts {experts}")

    # 256 output tokens (the first, the last and a seeded sample), each
    # computed by the dense per-token brute force from its own top-k; the
    # host holds at most 64 experts' weights at a time
    rng = np.random.default_rng(2)
    tokens = np.unique(np.concatenate([[0, cfg.T - 1],
                                       rng.choice(np.arange(1, cfg.T - 1), 254, replace=False)]))
    assert tokens.size == 256
    got_all = bits(out.index_select(0, torch.from_numpy(tokens.astype(np.int64)).to(dev)))
    for group in _token_groups(tokens, ref_idx, 64):
        used = np.unique(ref_idx[group])
        remap = np.zeros(cfg.n_experts, np.int32)
        remap[used] = np.arange(used.size, dtype=np.int32)
        want = oracle.moe_tokens_dense(x_h, _compact(d["w_gate"], used), _compact(d["w_up"], used),
                                       _compact(d["w_down"], used), remap[ref_idx], ref_w,
                                       group.astype(np.int32), cfg.dtype)
        got = got_all[np.searchsorted(tokens, group)]
        assert_close(got, want, cfg.dtype, rtol, atol, f"output tokens {group[:4]}...")


def _token_groups(tokens, topk_idx, max_experts):
    """Split tokens into groups whose routed experts number at most
    max_experts together (greedy, in token order)."""
    groups, cur, cur_set = [], [], set()
    for t in tokens:
        e = set(int(v) for v in topk_idx[t])
        if cur and len(cur_set | e) > max_experts:
            groups.append(np.array(cur))
            cur, cur_set = [], set()
        cur.append(int(t))
        cur_set |= e
    if cur:
        groups.append(np.array(cur))
    return groups


def test_forward_pipeline_matches_single_forwards():
    """binding.ForwardPipeline (copies in and out overlapping neighbouring
    batches' forwards) returns, for every batch, the bits of one moe_forward
    call on the same tokens; five batches cycle both buffer parities."""
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["tiny"]
    d = workloads.make_moe_inputs(cfg, device=dev)
    T, d_h, k = cfg.T, cfg.d_hidden, cfg.top_k
    pl = binding.ForwardPipeline(d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], k, T)
    xs = [workloads.make_tokens(cfg, T, device="cpu", seed=50 + i).pin_memory() for i in range(5)]
    outs = [torch.empty((T, d_h), dtype=xs[0].dtype).pin_memory() for _ in range(5)]
    evs = [pl.submit(xs[i], outs[i]) for i in range(5)]
    evs[-1].synchronize()
    pl.synchronize()
    assert int(pl.err.item()) == 0
    for i in range(5):
        ref = binding.moe_forward(xs[i].to(dev), d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], k)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref.cpu()), i
    with pytest.raises(ValueError):
        pl.submit(xs[0].to(dev), outs[0])  # tokens must be pinned host memory
