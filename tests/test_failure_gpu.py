"""Failure detection on the GPU without a fault.

Every wait of the pipeline kernels is bounded: a wait that runs out sets the
library's device status word, the kernel stops and returns, and the host
reads the status.  Here a wait runs out on purpose, on a barrier that
nothing completes (fa2_check_wait_timeout), and the test checks that the
status is reported, that it took about the requested time, and that the
context still computes correct results afterwards.
"""
import math
import time

import numpy as np
import pytest
import torch

import exact_attention_17_gb300 as fa2
import oracle
from exact_attention_17_gb300 import build as libbuild
from exact_attention_17_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    libbuild.build()
    oracle.build()
    fa2.fa2_device_status(None, reset=True)
    yield torch.device("cuda:0")
    fa2.fa2_device_status(None, reset=True)


def test_bounded_wait_reports_a_timeout_and_the_context_survives(dev):
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None, reset=True) == fa2.FA2_OK
    limit_ns = 20_000_000
    t0 = time.monotonic()
    assert fa2.fa2_check_wait_timeout(limit_ns) == fa2.FA2_OK
    assert fa2.fa2_device_status(None, reset=True) == fa2.FA2_ERR_TIMEOUT
    elapsed = time.monotonic() - t0
    assert limit_ns * 1e-9 * 0.9 <= elapsed < 10.0
    assert fa2.fa2_device_status(None) == fa2.FA2_OK      # the reset cleared it

    # the same context keeps computing correct results
    Q, K, V = inputs.make_qkv(1, 2, 300, 400, 128, seed=11)
    scale = float(np.float32(1 / math.sqrt(128)))
    O, L = fa2.forward(Q.to(dev), K.to(dev), V.to(dev), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None) == fa2.FA2_OK
    Or, Lr = oracle.attention(*(inputs.bf16_bits(t) for t in (Q, K, V)), True, scale)
    assert float(np.max(np.abs(O.cpu().double().numpy() - Or))) <= 2e-2
    assert float(np.max(np.abs(L.cpu().double().numpy() - Lr))) <= 1e-2
