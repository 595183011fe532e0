"""Bounded waits on the GPU, tested without a fault: moe_wait_flag on a flag
that nothing sets runs out, reports MOE_ERR_TIMEOUT through the error word
and returns, and the same CUDA context then runs a forward that matches the
oracle; a flag in pinned host memory set by the host releases the work queued
behind the wait."""
import time

import numpy as np
import pytest
import torch

from gpu_helpers import MOE_TOL, assert_bits_equal, assert_close, bits, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6


def test_wait_on_a_flag_nothing_sets_times_out_and_the_context_stays_usable(oracle):
    dev = require_cuda()
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_.record()
    binding.moe_wait_flag(flag, 1, 0.05, err)
    e_.record()
    torch.cuda.synchronize()
    assert int(err.item()) == MOE_ERR_TIMEOUT
    assert s_.elapsed_time(e_) >= 45.0  # ms: it waited about its limit, then gave up
    # the context still runs the forward, bit-exact routing and tables
    cfg = workloads.MOE_CONFIGS["tiny"]
    d = workloads.make_moe_inputs(cfg, device=dev)
    err2 = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(binding.forward_workspace_bytes(cfg.T, cfg.d_hidden, cfg.d_expert, cfg.n_experts,
                                                     cfg.top_k, d["x"].dtype), dtype=torch.uint8, device=dev)
    out = binding.moe_forward(d["x"], d["wg"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], cfg.top_k,
                              ws=ws, err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    nb = {n: (bits(v) if v is not None else None) for n, v in d.items()}
    ref = oracle.moe_forward(nb["x"], nb["wg"], nb["bias"], nb["w_gate"], nb["w_up"], nb["w_down"],
                             cfg.top_k, cfg.dtype)
    views = binding.forward_workspace_views(ws, cfg.T, cfg.d_hidden, cfg.d_expert, cfg.n_experts, cfg.top_k,
                                            d["x"].dtype)
    assert_bits_equal(views["topk_idx"].cpu().numpy(), ref["topk_idx"], "topk_idx")
    assert_close(bits(out), ref["out"], cfg.dtype, *MOE_TOL[cfg.dtype], "out after a timed-out wait")


def test_host_doorbell_in_pinned_memory_releases_queued_work():
    dev = require_cuda()
    flag = torch.zeros(1, dtype=torch.int32).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    src = torch.arange(4096, dtype=torch.int32, device=dev)
    dst = torch.zeros(4096, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    binding.moe_wait_flag(flag, 1, 5.0, err, device=dev)
    binding.moe_copy(src, dst)
    time.sleep(0.05)
    assert not torch.cuda.current_stream(dev).query()  # still held by the wait
    flag[0] = 1
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(dst, src)


def test_flag_already_set_passes_at_once():
    dev = require_cuda()
    flag = torch.full((1,), 7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.moe_wait_flag(flag, 5, 2.0, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
