"""Parity of the tensor-core backward pass against the fp64 oracle.

The GPU's forward pass produces O and LSE; the backward pass then gives dQ,
dK and dV for a seeded upstream gradient dO.  The oracle computes the exact
gradients of the attention definition from the same inputs, together with
per-element magnitudes M (see oracle/attn_ref.c; pinned to their
definitions in tests/test_oracle_backward.py).

Bound for bf16 inputs.  The kernel rounds P (for dV) and dS (for dQ, dK) to
bf16, whose unit roundoff is u = 2^-8 (8-bit significand, round to nearest
even), and takes D_i = dO_i . O_i from the forward's O, whose weights carry
the same rounding, so D_i is off by at most u A_i.  To first order every
element is then within u M of the exact gradient.  The remaining error comes
from fp32 arithmetic: the recomputed scores (d products summed in fp32),
the forward's LSE, ex2.approx, the fp32 sums of dP, D and the dQ
reductions; each moves an element by well under 2^-13 M.  The test allows
(2^-8 + 2^-10) M + 1e-6.

Bound for fp16 inputs.  u = 2^-11, but P and dS values below fp16's normal
range (2^-14) are rounded with an absolute error of up to 2^-25 instead of a
relative one, which M does not cover; the test allows 2^-7 M + 1e-6 there.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_17_gb300 as fa2
from exact_attention_17_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
REL = {"bf16": 2.0 ** -8 + 2.0 ** -10, "fp16": 2.0 ** -7}
ABS = 1e-6


def scale_for(d):
    return float(np.float32(1.0 / math.sqrt(d)))


def gpu_pass(Q, K, V, dO, causal, scale):
    q, k, v, do = (t.to(DEV) for t in (Q, K, V, dO))
    o, lse = fa2.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa2.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None, reset=True) == fa2.FA2_OK
    return [t.cpu().double().numpy() for t in (dq, dk, dv)]


def check(oracle_mod, Q, K, V, dO, causal, scale, got, heads=None, dtype="bf16"):
    """got: (dQ, dK, dV) as [B,H,N,d]; compares the listed flat heads (all by default)."""
    B, H = Q.shape[:2]
    ref = oracle_mod.attention_backward(inputs.bf16_bits(Q), inputs.bf16_bits(K), inputs.bf16_bits(V),
                                        inputs.bf16_bits(dO), causal, scale, heads=heads,
                                        dtype=dtype, magnitudes=True)
    hl = list(range(B * H)) if heads is None else list(heads)
    for name, g, r, m in zip(("dQ", "dK", "dV"), got, ref[:3], ref[3:]):
        g = g.reshape(B * H, *g.shape[2:])[hl]
        err = np.abs(g - r)
        bound = REL[dtype] * m + ABS
        worst = np.max(err - bound)
        ratio = float(np.max(err / (m + ABS / REL[dtype])))
        assert worst <= 0, (f"{name}: error exceeds the bound by {worst:.3e} (max err {err.max():.3e}, "
                            f"max err / M {ratio:.3e})")
        # the bound is not vacuous: the result tracks the exact gradient closely
        # overall (with the elementwise ABS as a floor, for gradients that are
        # exactly zero, e.g. dQ with a single key)
        assert np.linalg.norm(g - r) <= max(1e-2 * np.linalg.norm(r), ABS * np.sqrt(r.size)), name


SMALL = [
    (1, 2, 128, 128, 64, False),
    (1, 2, 200, 300, 64, False),
    (2, 1, 256, 256, 128, True),
    (1, 1, 300, 300, 128, True),
    (1, 2, 64, 1000, 128, False),
    (1, 1, 500, 130, 64, True),
    (1, 1, 1, 1, 64, False),
    (1, 1, 128, 384, 128, True),    # keys past 127 are seen by no query: zero dK, dV
    (1, 3, 513, 129, 128, False),
    (2, 2, 640, 640, 64, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SMALL)
def test_backward_matches_oracle(oracle_mod, B, H, Nq, Nk, d, causal):
    seed = 100 + Nq + 7 * Nk + d + int(causal)
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed)
    dO = inputs.draw_bf16((B, H, Nq, d), seed, 3)
    scale = scale_for(d)
    got = gpu_pass(Q, K, V, dO, causal, scale)
    check(oracle_mod, Q, K, V, dO, causal, scale, got)
    if causal and Nk > Nq:
        # keys that no query sees
        for g in got[1:]:
            assert np.all(g[:, :, Nq:] == 0)


def test_no_query_rows_gives_zero_key_gradients():
    k = torch.randn(1, 2, 300, 64, device=DEV).bfloat16()
    dk = torch.full((1, 2, 300, 64), 7.0, device=DEV)
    dv = torch.full((1, 2, 300, 64), 7.0, device=DEV)
    rc = fa2.fa2_backward(None, k.data_ptr(), k.data_ptr(), None, None, None, None, dk.data_ptr(),
                          dv.data_ptr(), 1, 2, 0, 300, 64, 1, 0.125, None, 0, None)
    torch.cuda.synchronize()
    assert rc == fa2.FA2_OK
    assert torch.all(dk == 0) and torch.all(dv == 0)


def test_repeated_calls_reset_the_dq_accumulator(oracle_mod):
    B, H, Nq, Nk, d = 1, 2, 384, 256, 128
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, 77)
    dO = inputs.draw_bf16((B, H, Nq, d), 77, 3)
    q, k, v, do = (t.to(DEV) for t in (Q, K, V, dO))
    o, lse = fa2.forward(q, k, v)
    outs = [fa2.backward(q, k, v, o, lse, do) for _ in range(2)]
    dq = torch.empty_like(outs[0][0]).fill_(123.0)
    dk = torch.empty_like(outs[0][1]).fill_(123.0)
    dv = torch.empty_like(outs[0][2]).fill_(123.0)
    fa2.backward(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    got = [t.cpu().double().numpy() for t in (dq, dk, dv)]
    check(oracle_mod, Q, K, V, dO, False, scale_for(d), got)
    # dK and dV need no atomics: bitwise repeatable
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])


@pytest.mark.parametrize("name,heads", [("b4_h16_n4096_d128_causal", None),
                                        ("b1_h32_n16384_d128_causal", [0, 5, 9, 14, 18, 23, 27, 31])])
def test_backward_full_size(oracle_mod, name, heads):
    """The full workloads, every head on the GPU; against the oracle every head
    of the 4096-length workload and eight of the 32 heads of the 16384-length
    one (about 5 s of oracle time per head there)."""
    w = inputs.workload(name)
    Q, K, V = inputs.workload_inputs(w)
    dO = inputs.draw_bf16((w.B, w.H, w.Nq, w.d), w.seed, 3)
    got = gpu_pass(Q, K, V, dO, w.causal, w.scale)
    check(oracle_mod, Q, K, V, dO, w.causal, w.scale, got, heads=heads)
    for g in got:
        assert np.all(np.isfinite(g))


FP16 = [
    (1, 2, 128, 128, 64, False),
    (1, 2, 200, 300, 128, True),
    (2, 1, 513, 129, 128, False),
    (1, 1, 640, 640, 64, True),
    (1, 2, 1000, 1000, 128, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", FP16)
def test_backward_fp16_matches_oracle(oracle_mod, B, H, Nq, Nk, d, causal):
    """fp16 Q, K, V and dO (fa2_backward_typed): P and dS are rounded to fp16
    (2^-11 relative per term, or 2^-25 absolute below fp16's normal range)."""
    seed = 300 + Nq + 3 * Nk + d + int(causal)
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed, qk_std=1.5, dtype=torch.float16)
    dO = inputs.draw_bf16((B, H, Nq, d), seed, 3, dtype=torch.float16)
    scale = scale_for(d)
    got = gpu_pass(Q, K, V, dO, causal, scale)
    check(oracle_mod, Q, K, V, dO, causal, scale, got, dtype="fp16")
