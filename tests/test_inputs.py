"""The seeded input generator: reproducible bits, the stated distributions, BHSD layout."""
import numpy as np
import torch

from exact_attention_17_gb300 import inputs


def test_bits_independent_of_thread_count():
    a = inputs.draw_bf16((3, inputs.CHUNK // 2 + 5), seed=9, tensor_id=1, threads=1)
    b = inputs.draw_bf16((3, inputs.CHUNK // 2 + 5), seed=9, tensor_id=1, threads=5)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_seed_and_tensor_id_change_the_draw():
    a = inputs.draw_bf16((64,), seed=1, tensor_id=0)
    assert not torch.equal(a, inputs.draw_bf16((64,), seed=2, tensor_id=0))
    assert not torch.equal(a, inputs.draw_bf16((64,), seed=1, tensor_id=1))


def test_distributions():
    x = inputs.draw_bf16((1 << 20,), seed=3, tensor_id=0, dist="normal", std=2.0).float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 2.0) < 0.01
    u = inputs.draw_bf16((1 << 20,), seed=3, tensor_id=2, dist="uniform").float()
    assert u.min().item() >= -1.0 and u.max().item() <= 1.0
    assert abs(u.mean().item()) < 0.01 and abs(u.var().item() - 1 / 3) < 0.01


def test_workload_table_shapes():
    w = inputs.workload("b2_h8_n1000_d64")
    Q, K, V = inputs.workload_inputs(w)
    assert Q.shape == (2, 8, 1000, 64) and K.shape == V.shape == (2, 8, 1000, 64)
    assert Q.dtype == torch.bfloat16 and Q.is_contiguous()
    assert w.scale == float(np.float32(0.125))
    assert inputs.WORKLOADS[2].causal and inputs.WORKLOADS[2].flops == 4 * 4 * 16 * 4096 * 4096 * 128 / 2
    bits = inputs.bf16_bits(Q)
    assert bits.dtype == np.uint16 and bits.shape == tuple(Q.shape)
