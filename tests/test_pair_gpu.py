"""GPU parity of the two-SM forward kernel (a CTA pair per 512 query rows).

The kernel is selected with FA2_FORWARD_KERNEL=pair, which runs it for every
head-dimension-128 problem, including the small and ragged ones the
default choice would give to the one-CTA kernel, so that the pair's edge
cases (a pair sub-tile whose peer rows lie past Nq, causal diagonals inside
a 256-row pair sub-tile, key tails) are all exercised.  Results are compared
with the fp64 oracle at the contract's tolerances on every row, and with
the one-CTA kernel on the same inputs.
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


@pytest.fixture
def pair(monkeypatch):
    monkeypatch.setenv("FA2_FORWARD_KERNEL", "pair")


def run(dev, Q, K, V, causal, scale, **kw):
    O, L = fa2.forward(Q.to(dev), K.to(dev), V.to(dev), causal=causal, scale=scale, **kw)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None, reset=True) == fa2.FA2_OK
    return O, L


def bits(*ts):
    return [inputs.bf16_bits(t) for t in ts]


def check(O, L, Or, Lr, what):
    O = O.detach().cpu().double().numpy()
    L = L.detach().cpu().double().numpy()
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L)), what
    eo = float(np.max(np.abs(O - Or))) if O.size else 0.0
    el = float(np.max(np.abs(L - Lr))) if L.size else 0.0
    assert eo <= TOL_O and el <= TOL_LSE, f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


EDGE = [(1, 1), (2, 2), (127, 127), (128, 128), (129, 129), (255, 255), (256, 256), (257, 257),
        (383, 383), (511, 511), (512, 512), (513, 513), (640, 640), (1000, 1000), (1023, 1023),
        (1025, 1025), (100, 700), (700, 100), (129, 1), (5, 257), (513, 129), (300, 1500)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", EDGE)
def test_pair_edge_sizes(dev, pair, nq, nk, causal):
    B, H = (1, 3) if nq * nk < 300000 else (1, 1)
    Q, K, V = inputs.make_qkv(B, H, nq, nk, 128, seed=nq * 31 + nk)
    scale = float(np.float32(1 / math.sqrt(128)))
    O, L = run(dev, Q, K, V, causal, scale)
    Or, Lr = oracle.attention(*bits(Q, K, V), causal, scale)
    check(O, L, Or, Lr, f"pair Nq={nq} Nk={nk} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_pair_fp16_inputs_and_outputs(dev, pair, causal):
    B, H, Nq, Nk = 1, 2, 1100, 900
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, 128, seed=91, dtype=torch.float16)
    scale = float(np.float32(1 / math.sqrt(128)))
    bq, bk, bv = (inputs.bf16_bits(t) for t in (Q, K, V))
    Or, Lr = oracle.attention(bq, bk, bv, causal, scale, dtype="fp16")
    for out_dtype in (torch.float32, torch.float16):
        O, L = run(dev, Q, K, V, causal, scale, out_dtype=out_dtype)
        # (fp16 O adds a rounding of at most 2^-11 |O|, far inside the tolerance)
        Od = O.float().cpu().double().numpy()
        assert float(np.max(np.abs(Od - Or))) <= TOL_O
        assert float(np.max(np.abs(L.cpu().double().numpy() - Lr))) <= TOL_LSE


@pytest.mark.parametrize("causal", [False, True])
def test_pair_split_kv(dev, pair, causal):
    B, H, Nq, Nk = 1, 2, 600, 2000
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, 128, seed=92)
    scale = float(np.float32(1 / math.sqrt(128)))
    Or, Lr = oracle.attention(*bits(Q, K, V), causal, scale)
    for splits in (2, 3, 16):
        O, L = run(dev, Q, K, V, causal, scale, num_splits=splits)
        check(O, L, Or, Lr, f"pair split {splits} causal={causal}")


def test_pair_peaky_scores_and_rising_maximum(dev, pair):
    """std-4 inputs at scale 0.3 move the running maximum often (O rescaled in TMEM)."""
    Q, K, V = inputs.make_qkv(2, 2, 700, 900, 128, seed=93, qk_std=4.0)
    for causal in (False, True):
        O, L = run(dev, Q, K, V, causal, 0.3)
        Or, Lr = oracle.attention(*bits(Q, K, V), causal, 0.3)
        check(O, L, Or, Lr, f"pair peaky causal={causal}")


@pytest.mark.parametrize("idx", [2, 3])
def test_pair_long_causal_workloads_every_row(dev, pair, idx):
    w = inputs.WORKLOADS[idx]
    Q, K, V = inputs.workload_inputs(w)
    O, L = run(dev, Q, K, V, w.causal, w.scale)
    O, L = O.cpu(), L.cpu()
    Or, Lr = oracle.attention(*bits(Q, K, V), w.causal, w.scale)
    check(O, L, Or, Lr, "pair " + w.name)


def test_pair_agrees_with_the_one_cta_kernel(dev, monkeypatch):
    """Both kernels on the same non-causal 16384-length heads: the same
    arithmetic per row, so the results agree far inside the tolerance."""
    w = inputs.workload("b1_h32_n16384_d128")
    Q, K, V = inputs.make_qkv(1, 4, w.Nq, w.Nk, w.d, w.seed, v_dist=w.v_dist)
    monkeypatch.setenv("FA2_FORWARD_KERNEL", "pair")
    Op, Lp = run(dev, Q, K, V, False, w.scale)
    monkeypatch.setenv("FA2_FORWARD_KERNEL", "single")
    Os, Ls = run(dev, Q, K, V, False, w.scale)
    assert float((Op - Os).abs().max()) <= 2e-3
    assert float((Lp - Ls).abs().max()) <= 1e-4
    rows = np.random.default_rng(5).integers(0, 4 * w.Nq, size=64)
    Or, Lr = oracle.attention_rows(*bits(Q, K, V), False, w.scale, rows)
    check(Op.reshape(-1, w.d)[torch.as_tensor(rows, device=dev)], Lp.reshape(-1)[torch.as_tensor(rows, device=dev)],
          Or, Lr, "pair non-causal 16384 sampled rows")
