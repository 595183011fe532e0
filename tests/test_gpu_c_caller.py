"""The C-ABI from a plain C program: tests/c/forward_from_c.c (no Python, no
PyTorch in that process) runs moe_forward on the tiny workload; its output
must equal, bit for bit, the same call made through the Python binding, and
match the oracle within the fp16 tolerance."""
import os
import subprocess

import numpy as np
import pytest
import torch

import c_caller
from gpu_helpers import MOE_TOL, assert_bits_equal, assert_close, bits, require_cuda
from mixture_experts_routed_gate_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [64, 37])
def test_forward_from_a_c_program(oracle, tmp_path, T):
    dev = require_cuda()
    cfg = workloads.MOE_CONFIGS["tiny"]
    d = workloads.make_moe_inputs(cfg, device=dev, T=T)
    for name in ("x", "wg", "w_gate", "w_up", "w_down"):
        bits(d[name]).tofile(os.path.join(tmp_path, f"{name}.bin"))
    exe = c_caller.build(str(tmp_path))
    code = 1 if cfg.dtype == "bf16" else 0
    r = subprocess.run([exe, str(tmp_path), str(T), str(cfg.d_hidden), str(cfg.d_expert), str(cfg.n_experts),
                        str(cfg.top_k), str(code)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
    got = np.fromfile(os.path.join(tmp_path, "out.bin"), dtype="<u2").reshape(T, cfg.d_hidden)
    want = binding.moe_forward(d["x"], d["wg"], None, d["w_gate"], d["w_up"], d["w_down"], cfg.top_k)
    torch.cuda.synchronize()
    assert_bits_equal(got, bits(want), "C caller vs Python binding")
    nb = {n: (bits(v) if v is not None else None) for n, v in d.items()}
    ref = oracle.moe_forward(nb["x"], nb["wg"], None, nb["w_gate"], nb["w_up"], nb["w_down"], cfg.top_k,
                             cfg.dtype)
    assert_close(got, ref["out"], cfg.dtype, *MOE_TOL[cfg.dtype], "C caller vs oracle")
