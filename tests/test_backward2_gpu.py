"""Parity of the two-tile backward kernel (two 64-row query tiles in flight,
head dimension 128) against the fp64 oracle's gradients.

FA2_BACKWARD_KERNEL=two_tile selects it; the bounds are those of
tests/test_backward_gpu.py (the rounding of P and dS is the same), and the
results are also compared with the one-tile kernel on the same inputs.
"""
import numpy as np
import pytest
import torch

import exact_attention_17_gb300 as fa2
from exact_attention_17_gb300 import inputs
from test_backward_gpu import check, gpu_pass, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture
def two_tile(monkeypatch):
    monkeypatch.setenv("FA2_BACKWARD_KERNEL", "two_tile")


CASES = [
    (1, 2, 64, 64, False),
    (1, 2, 128, 128, True),
    (2, 1, 256, 256, True),
    (1, 1, 300, 300, True),
    (1, 2, 64, 1000, False),
    (1, 1, 1, 1, False),
    (1, 1, 65, 65, True),
    (1, 1, 127, 129, True),
    (1, 1, 128, 384, True),    # keys past 127 are seen by no query: zero dK, dV
    (1, 3, 513, 129, False),
    (2, 2, 640, 640, True),
    (1, 1, 1000, 1000, False),
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal", CASES)
def test_two_tile_backward_matches_oracle(oracle_mod, two_tile, B, H, Nq, Nk, causal):
    d = 128
    seed = 500 + Nq + 7 * Nk + int(causal)
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed)
    dO = inputs.draw_bf16((B, H, Nq, d), seed, 3)
    got = gpu_pass(Q, K, V, dO, causal, scale_for(d))
    check(oracle_mod, Q, K, V, dO, causal, scale_for(d), got)
    if causal and Nk > Nq:
        for g in got[1:]:
            assert np.all(g[:, :, Nq:] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_two_tile_backward_fp16(oracle_mod, two_tile, causal):
    B, H, Nq, Nk, d = 1, 2, 700, 500, 128
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, 611, qk_std=1.5, dtype=torch.float16)
    dO = inputs.draw_bf16((B, H, Nq, d), 611, 3, dtype=torch.float16)
    got = gpu_pass(Q, K, V, dO, causal, scale_for(d))
    check(oracle_mod, Q, K, V, dO, causal, scale_for(d), got, dtype="fp16")


def test_two_tile_backward_repeated_calls_and_agreement(oracle_mod, monkeypatch):
    """dQ is accumulated: repeated calls must start from zero each time; dK
    and dV need no atomics and repeat bit for bit; the one-tile kernel gives
    the same gradients up to rounding."""
    B, H, Nq, Nk, d = 1, 2, 384, 256, 128
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, 612)
    dO = inputs.draw_bf16((B, H, Nq, d), 612, 3)
    monkeypatch.setenv("FA2_BACKWARD_KERNEL", "two_tile")
    a = gpu_pass(Q, K, V, dO, True, scale_for(d))
    b = gpu_pass(Q, K, V, dO, True, scale_for(d))
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    check(oracle_mod, Q, K, V, dO, True, scale_for(d), b)
    monkeypatch.setenv("FA2_BACKWARD_KERNEL", "one_tile")
    c = gpu_pass(Q, K, V, dO, True, scale_for(d))
    for x, y in zip(a, c):
        assert np.max(np.abs(x - y)) <= 2e-3 * max(np.max(np.abs(y)), 1e-30)


@pytest.mark.parametrize("name,heads", [("b4_h16_n4096_d128_causal", None),
                                        ("b1_h32_n16384_d128_causal", [0, 9, 18, 31])])
def test_two_tile_backward_full_size(oracle_mod, two_tile, name, heads):
    w = inputs.workload(name)
    Q, K, V = inputs.workload_inputs(w)
    dO = inputs.draw_bf16((w.B, w.H, w.Nq, w.d), w.seed, 3)
    got = gpu_pass(Q, K, V, dO, w.causal, w.scale)
    check(oracle_mod, Q, K, V, dO, w.causal, w.scale, got, heads=heads)
    for g in got:
        assert np.all(np.isfinite(g))
