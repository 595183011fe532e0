"""The algorithmic byte and FLOP counts behind the benchmark's roofline
fractions, checked against counts worked out by hand for the decode and
prefill workloads (host arithmetic only)."""
from mixture_experts_routed_gate_gb300 import roofline


def test_expert_mlp_counts_decode():
    # 64 tokens x top-6 = 384 routed rows, d_hidden 2048, d_expert 768, all 64
    # experts active, fp16: three 768 x 2048 weight matrices per expert
    # (603,979,776 B), the gathered rows read (1,572,864 B), h written and read
    # back (2 x 589,824 B), y written (1,572,864 B)
    assert roofline.expert_mlp_bytes(384, 2048, 768, 64, 2) == 608_305_152
    # 2 FLOPs per MAC: 384 rows x (2 x 768 + 768) x 2048 MACs
    assert roofline.expert_mlp_flops(384, 2048, 768) == 3_623_878_656


def test_expert_mlp_counts_prefill_per_active_expert():
    # every active expert adds its three 2048 x 7168 bf16 matrices: 88,080,384 B
    a = roofline.expert_mlp_bytes(32768, 7168, 2048, 190, 2)
    b = roofline.expert_mlp_bytes(32768, 7168, 2048, 191, 2)
    assert b - a == 3 * 2048 * 7168 * 2 == 88_080_384
    # activations: A 469.8 MB read, h 134.2 MB written + read, y 469.8 MB written
    assert roofline.expert_mlp_bytes(32768, 7168, 2048, 0, 2) == 32768 * (7168 + 2 * 2048 + 7168) * 2
    # 2.886 TFLOP for the two stages
    assert roofline.expert_mlp_flops(32768, 7168, 2048) == 2 * 32768 * 3 * 7168 * 2048


def test_stage_counts_add_up():
    for n, d_h, d_e, act, e in [(384, 2048, 768, 64, 2), (128, 256, 128, 8, 2), (1, 256, 64, 1, 4)]:
        assert roofline.expert_mlp_bytes(n, d_h, d_e, act, e) == \
            roofline.gate_up_bytes(n, d_h, d_e, act, e) + roofline.down_bytes(n, d_h, d_e, act, e)
        assert roofline.expert_mlp_flops(n, d_h, d_e) == \
            roofline.gate_up_flops(n, d_h, d_e) + roofline.down_flops(n, d_h, d_e)


def test_combine_counts():
    # 4096 tokens x 8 slots, 10% padding (3277 slots) never read, H 7168, bf16
    n_valid = 4096 * 8 - 3277
    assert roofline.reduce_bytes(n_valid, 4096, 8, 7168, 2, 2) == \
        n_valid * 7168 * 2 + 4096 * 7168 * 2 + 4096 * 8 * 8
    assert roofline.reduce_bytes(n_valid, 4096, 8, 7168, 2, 2, weighted=False) == \
        n_valid * 7168 * 2 + 4096 * 7168 * 2 + 4096 * 8 * 4
    assert roofline.reduce_flops(4096, 8, 7168) == 2 * 4096 * 8 * 7168


def test_forward_counts():
    # decode: gate 16.8 MFLOP + expert MLP + combine 2 x 64 x 6 x 2048
    f = roofline.moe_forward_flops(64, 6, 2048, 768, 64)
    assert f == 2 * 64 * 64 * 2048 + 3_623_878_656 + 2 * 64 * 6 * 2048
    assert roofline.moe_forward_bytes_min(64, 2048, 768, 64, 64, 2) == \
        3 * 64 * 768 * 2048 * 2 + 64 * 2048 * 2 + 2 * 64 * 2048 * 2


def test_kernels_per_step_follow_the_launch_structure():
    """The launch count the bench line claims: prefill (T=4096, 256 experts,
    top-8) runs the tensor-core logits and the selection, the histogram and
    the scan-and-scatter dispatch, the gather, the expert MLP and the combine
    (7); decode (T=64, 64 experts) the fused CUDA-core gate, the one-CTA
    dispatch, the gathering expert MLP and the combine (4)."""
    import dataclasses
    import bench
    from mixture_experts_routed_gate_gb300 import workloads
    assert bench.kernels_per_step(workloads.MOE_CONFIGS["prefill"]) == 7
    assert bench.kernels_per_step(workloads.MOE_CONFIGS["decode"]) == 4
    # below the tensor-core gate's token count with more than 64 experts: gate + top-k
    mid = dataclasses.replace(workloads.MOE_CONFIGS["prefill"], batch=1, seq=512)
    assert bench.kernels_per_step(mid) == 2 + 1 + 1 + 2
