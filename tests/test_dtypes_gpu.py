"""GPU parity for the other element types: fp16 Q/K/V and O stored in the
input dtype (the "Triton内核实战" wrapper returns O in the input dtype).

Compared with the fp64 oracle reading the same 16-bit patterns, within the
same tolerances as the bf16 path."""
import math

import numpy as np
import pytest
import torch

import exact_attention_17_gb300 as fa2
import oracle
from exact_attention_17_gb300 import build as libbuild
from exact_attention_17_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-2


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    libbuild.build()
    oracle.build()
    fa2.fa2_device_status(None, reset=True)
    yield torch.device("cuda:0")
    assert fa2.fa2_device_status(None, reset=True) == fa2.FA2_OK


CASES = [(1, 2, 1, 1), (1, 3, 130, 70), (2, 2, 257, 1000), (1, 2, 1000, 1000), (1, 1, 513, 129),
         (1, 4, 2048, 2048)]


@pytest.mark.parametrize("in_name,out_name", [("fp16", "fp32"), ("fp16", "same"), ("bf16", "same")])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk", CASES)
def test_element_types(dev, in_name, out_name, d, causal, B, H, Nq, Nk):
    in_dtype = torch.float16 if in_name == "fp16" else torch.bfloat16
    out_dtype = torch.float32 if out_name == "fp32" else in_dtype
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed=Nq * 31 + Nk + d, qk_std=1.5, dtype=in_dtype)
    scale = float(np.float32(1 / math.sqrt(d)))
    O, L = fa2.forward(Q.to(dev), K.to(dev), V.to(dev), causal=causal, scale=scale, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert O.dtype == out_dtype and fa2.fa2_device_status(None) == fa2.FA2_OK
    Or, Lr = oracle.attention(*(inputs.bf16_bits(t) for t in (Q, K, V)), causal, scale, dtype=in_name)
    O = O.float().cpu().double().numpy()
    L = L.cpu().double().numpy()
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    eo, el = float(np.max(np.abs(O - Or))), float(np.max(np.abs(L - Lr)))
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


def test_fp16_is_more_accurate_than_bf16_on_the_same_values(dev):
    """Values exact in both types: fp16's P rounding (11 significant bits)
    should not be worse than bf16's (8 bits)."""
    B, H, Nq, Nk, d = 1, 4, 512, 2048, 128
    Qb, Kb, Vb = inputs.make_qkv(B, H, Nq, Nk, d, seed=5)
    # bf16 values of magnitude in [2^-14, 2^15] are exact in fp16: zero out the rest
    Qb, Kb, Vb = (torch.where(t.float().abs() < 2.0 ** -14, torch.zeros_like(t), t) for t in (Qb, Kb, Vb))
    Qh, Kh, Vh = Qb.half(), Kb.half(), Vb.half()
    assert torch.equal(Qh.bfloat16(), Qb) and torch.equal(Vh.bfloat16(), Vb)
    Or, Lr = oracle.attention(*(inputs.bf16_bits(t) for t in (Qb, Kb, Vb)), False, 0.0883883461356163)
    Ob, _ = fa2.forward(Qb.to(dev), Kb.to(dev), Vb.to(dev), scale=0.0883883461356163)
    Oh, _ = fa2.forward(Qh.to(dev), Kh.to(dev), Vh.to(dev), scale=0.0883883461356163)
    torch.cuda.synchronize()
    eb = float(np.max(np.abs(Ob.cpu().double().numpy() - Or)))
    eh = float(np.max(np.abs(Oh.cpu().double().numpy() - Or)))
    assert eh <= eb


def test_dtype_errors(dev):
    B, H, N, d = 1, 1, 64, 64
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device=dev)
    o = torch.empty(B, H, N, d, device=dev)
    l = torch.empty(B, H, N, device=dev)
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, N, N, d, 0, 0.125)
    assert fa2.fa2_forward_typed(*args, fa2.FA2_DTYPE_FP32, fa2.FA2_DTYPE_FP32, None) == fa2.FA2_ERR_DTYPE
    assert fa2.fa2_forward_typed(*args, fa2.FA2_DTYPE_BF16, fa2.FA2_DTYPE_FP16, None) == fa2.FA2_ERR_DTYPE
    assert fa2.fa2_forward_typed(*args, 7, fa2.FA2_DTYPE_FP32, None) == fa2.FA2_ERR_DTYPE
    assert fa2.fa2_forward_typed(*args, fa2.FA2_DTYPE_BF16, fa2.FA2_DTYPE_FP32, None) == fa2.FA2_OK
    torch.cuda.synchronize()
