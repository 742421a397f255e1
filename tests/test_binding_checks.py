"""The Python binding refuses tensors smaller than the shape implies before any
pointer reaches the library (a shorter tensor would let a kernel read or write
past it).  The element-count check precedes the device check, so it runs here
on CPU tensors without a GPU."""
import pytest
import torch

import sparse_mixture_experts_46_b300 as moe

S = moe.make_shape(T=16, dim=128, hidden=256, n_experts=8, top_k=2)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def test_router_rejects_short_inputs_and_outputs():
    with pytest.raises(ValueError, match="x holds 2032 elements; the shape needs 2048"):
        moe.moe_router_topk(S, bf16(2032), bf16(128, 8), i32(16, 2), f32(16, 2), i32(8))
    with pytest.raises(ValueError, match="ids holds"):
        moe.moe_router_topk(S, bf16(16, 128), bf16(128, 8), i32(15, 2), f32(16, 2), i32(8))
    with pytest.raises(ValueError, match="counts holds"):
        moe.moe_router_topk(S, bf16(16, 128), bf16(128, 8), i32(16, 2), f32(16, 2), i32(7))


def test_grouping_ffn_and_combine_reject_short_buffers():
    ws = torch.zeros(1, dtype=torch.uint8)
    with pytest.raises(ValueError, match="offsets holds 8 elements; the shape needs 9"):
        moe.moe_permute(S, bf16(16, 128), i32(32), i32(8), i32(32), i32(32), bf16(32, 128), ws)
    with pytest.raises(ValueError, match="h holds"):
        moe.moe_expert_ffn_grouped(S, bf16(32, 128), i32(9), bf16(8, 256, 128),
                                   bf16(8, 256, 128), bf16(8, 128, 256), bf16(31, 256),
                                   bf16(32, 128), ws)
    with pytest.raises(ValueError, match="w2 holds"):
        moe.moe_expert_ffn_grouped(S, bf16(32, 128), i32(9), bf16(8, 256, 128),
                                   bf16(8, 256, 128), bf16(7, 128, 256), bf16(32, 256),
                                   bf16(32, 128), ws)
    with pytest.raises(ValueError, match="residual holds"):
        moe.moe_combine(S, bf16(32, 128), i32(32), f32(32), bf16(16, 128), residual=bf16(8, 128))


def test_layer_backward_and_statistics_reject_short_buffers():
    ws = torch.zeros(1, dtype=torch.uint8)
    with pytest.raises(ValueError, match="gates holds"):
        moe.moe_layer_forward(S, bf16(16, 128), bf16(128, 8), bf16(8, 256, 128),
                              bf16(8, 256, 128), bf16(8, 128, 256), bf16(16, 128), ws,
                              gates=f32(16))
    B = moe.make_shape(T=16, dim=256, hidden=256, n_experts=8, top_k=2)
    w = bf16(8, 256, 256)
    with pytest.raises(ValueError, match="dw3 holds"):
        moe.moe_layer_backward(B, bf16(16, 256), bf16(256, 8), w, w, w, bf16(16, 256),
                               bf16(16, 256), f32(256, 8), f32(8, 256, 256), f32(8, 255, 256),
                               f32(8, 256, 256), ws)
    with pytest.raises(ValueError, match="repeats holds 1 elements; the shape needs 2"):
        moe.moe_routing_stats(S, i32(16, 2), i32(2 * 8), i32(1))


def test_full_size_cpu_tensors_pass_the_count_check_and_stop_at_the_device_check():
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        moe.moe_router_topk(S, bf16(16, 128), bf16(128, 8), i32(16, 2), f32(16, 2), i32(8))


def test_statistics_reject_short_slot_counts():
    with pytest.raises(ValueError, match="slot_counts holds 15 elements; the shape needs 16"):
        moe.moe_routing_stats(S, i32(16, 2), i32(15), i32(2))
