"""The forward pass from host buffers (fa2_forward_host).

The head groups are copied in, computed and copied out on the library's
three streams; the result must equal fa2_forward's on the same inputs (each
row's arithmetic is the same), and match the fp64 oracle at the contract's
tolerances, for any number of groups, with pinned or pageable host memory.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_17_gb300 as fa2
import oracle
from exact_attention_17_gb300 import build as libbuild
from exact_attention_17_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    libbuild.build()
    oracle.build()
    fa2.fa2_device_status(None, reset=True)
    yield
    assert fa2.fa2_device_status(None, reset=True) == fa2.FA2_OK


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [(2, 5, 300, 700, 128, False), (1, 7, 513, 513, 128, True),
                                                (1, 3, 129, 129, 64, True), (2, 2, 1000, 1000, 256, False)])
@pytest.mark.parametrize("chunks", [1, 3, 8, 16])
def test_host_buffers_match_the_device_entry_point(B, H, Nq, Nk, d, causal, chunks):
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed=40 + Nq + chunks)
    scale = float(np.float32(1 / math.sqrt(d)))
    stream = torch.cuda.Stream()
    Qp, Kp, Vp = Q.pin_memory(), K.pin_memory(), V.pin_memory()
    Oh, Lh = fa2.forward_host(Qp, Kp, Vp, causal=causal, scale=scale, chunks=chunks, stream=stream)
    stream.synchronize()
    assert fa2.fa2_device_status(None) == fa2.FA2_OK
    Od, Ld = fa2.forward(Q.to(DEV), K.to(DEV), V.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert float((Oh - Od.cpu()).abs().max()) <= 1e-6
    assert float((Lh - Ld.cpu()).abs().max()) <= 1e-6
    Or, Lr = oracle.attention(inputs.bf16_bits(Q), inputs.bf16_bits(K), inputs.bf16_bits(V), causal, scale)
    assert float(np.max(np.abs(Oh.double().numpy() - Or))) <= 2e-2
    assert float(np.max(np.abs(Lh.double().numpy() - Lr))) <= 1e-2


def test_pageable_host_memory_and_stream_order():
    """Pageable buffers give the same result; the call is ordered after work
    already queued on the stream and before work queued after it."""
    B, H, Nq, Nk, d = 1, 4, 384, 640, 128
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed=77)
    stream = torch.cuda.Stream()
    qd, kd, vd = (torch.empty_like(t, device=DEV) for t in (Q, K, V))
    od = torch.empty(B, H, Nq, d, device=DEV)
    ld = torch.empty(B, H, Nq, device=DEV)
    with torch.cuda.stream(stream):
        od.fill_(float("nan"))   # queued before the call: must not land after it
    Oh = torch.empty(B, H, Nq, d)
    Lh = torch.empty(B, H, Nq)
    fa2.forward_host(Q, K, V, out=Oh, lse=Lh, device_buffers=(qd, kd, vd, od, ld), chunks=4, stream=stream)
    with torch.cuda.stream(stream):
        o2 = od.clone()          # queued after the call: sees the computed O
    stream.synchronize()
    Od, Ld = fa2.forward(Q.to(DEV), K.to(DEV), V.to(DEV))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(Oh).all())
    assert float((Oh - Od.cpu()).abs().max()) <= 1e-6 and float((Lh - Ld.cpu()).abs().max()) <= 1e-6
    assert torch.equal(o2, od)
