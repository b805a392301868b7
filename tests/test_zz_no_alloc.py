"""The split-KV entry point that allocates nothing (fa2_forward_splitkv_static).

Some callers cannot allocate device memory where they call attention -- a
plugin inside a framework that owns all device memory and gives it no
allocator, or a server that reserves its memory at start-up and forbids
allocation while serving -- so they cannot pass fa2_forward_splitkv a
workspace.  This entry point keeps the partial results in the library's own
32 MiB device array instead.  The test calls it through the C ABI and checks
it against the workspace entry point on consecutive calls with different
problems.  Both run the same kernels with the same split plan and no
atomics, so their results must be bitwise equal; the shared array keeps the
previous call's contents, and a call before each checked one leaves very
different partial results there (V scaled by 64 over more rows), so that a
read of stale partials would show.  One result is also checked against the
fp64 oracle, and a problem too large for the array is refused before
anything runs.

This file is collected last so that a failure here comes after every other
test has run; it also passes on its own in a fresh process.
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


def call_static(Q, K, V, causal, splits):
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    scale = float(np.float32(1 / math.sqrt(d)))
    O = torch.full((B, H, Nq, d), float("nan"), device=Q.device)
    L = torch.full((B, H, Nq), float("nan"), device=Q.device)
    rc = fa2.fa2_forward_splitkv_static(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                        L.data_ptr(), B, H, Nq, Nk, d, causal, scale, splits, None)
    assert rc == fa2.FA2_OK, fa2.fa2_status_string(rc)
    return O, L


def poison(dev, B, H, Nq, Nk, d, causal, splits, seed):
    """A call over more rows with V scaled by 64: its partial results, left in
    the shared array, differ from any checked call's everywhere."""
    Q, K, V = (t.to(dev) for t in inputs.make_qkv(B, H + 1, Nq, Nk, d, seed=seed + 1000))
    call_static(Q, K, (V.float() * 64).bfloat16(), causal, splits)


def run_both(dev, B, H, Nq, Nk, d, causal, splits, seed, with_oracle=False):
    Qh, Kh, Vh = inputs.make_qkv(B, H, Nq, Nk, d, seed=seed)
    Q, K, V = Qh.to(dev), Kh.to(dev), Vh.to(dev)
    scale = float(np.float32(1 / math.sqrt(d)))
    poison(dev, B, H, Nq, Nk, d, causal, splits, seed)
    Os, Ls = call_static(Q, K, V, causal, splits)
    need = fa2.fa2_splitkv_workspace_bytes(B, H, Nq, d, splits)
    assert need <= 32 << 20
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    Ow = torch.empty_like(Os)
    Lw = torch.empty_like(Ls)
    rc = fa2.fa2_forward_splitkv(Q.data_ptr(), K.data_ptr(), V.data_ptr(), Ow.data_ptr(), Lw.data_ptr(),
                                 B, H, Nq, Nk, d, causal, scale, splits, ws.data_ptr(), need, None)
    assert rc == fa2.FA2_OK, fa2.fa2_status_string(rc)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None) == fa2.FA2_OK
    assert bool(torch.isfinite(Os).all()) and bool(torch.isfinite(Ls).all())
    # same kernels, same split plan, no atomics: bitwise equal
    assert torch.equal(Os, Ow), float((Os - Ow).abs().max())
    assert torch.equal(Ls, Lw), float((Ls - Lw).abs().max())
    if with_oracle:
        Or, Lr = oracle.attention(inputs.bf16_bits(Qh), inputs.bf16_bits(Kh), inputs.bf16_bits(Vh),
                                  causal, scale)
        eo = float(np.max(np.abs(Os.cpu().double().numpy() - Or)))
        el = float(np.max(np.abs(Ls.cpu().double().numpy() - Lr)))
        assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


def test_static_scratch_matches_workspace_entry_point_on_consecutive_calls(dev):
    decode = (2, 8, 1, 8192, 128, False, 8)
    causal_ragged = (1, 4, 300, 3000, 64, True, 4)
    run_both(dev, *decode, seed=101, with_oracle=True)
    run_both(dev, *causal_ragged, seed=102, with_oracle=True)
    run_both(dev, *decode, seed=103)


def test_static_scratch_refuses_problems_larger_than_its_buffer(dev):
    B, H, Nq, Nk, d = 16, 32, 128, 8192, 128      # 4 ranges need about 135 MB of partials
    assert fa2.fa2_splitkv_workspace_bytes(B, H, Nq, d, 4) > 32 << 20
    q = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, H, Nk, d, dtype=torch.bfloat16, device=dev)
    o = torch.full((B, H, Nq, d), float("nan"), device=dev)
    l = torch.full((B, H, Nq), float("nan"), device=dev)
    rc = fa2.fa2_forward_splitkv_static(q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), l.data_ptr(),
                                        B, H, Nq, Nk, d, 0, 0.1, 4, None)
    assert rc == fa2.FA2_ERR_SCRATCH
    assert "32 MiB" in fa2.fa2_status_string(rc)
    torch.cuda.synchronize()
    assert bool(torch.isnan(o).all()) and bool(torch.isnan(l).all())
