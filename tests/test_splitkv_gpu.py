"""GPU parity of the split-KV forward and of the merge entry point.

Split-KV ("Flash Attention 全解析(上)" section 4) must give the attention of
the whole key range: compared with the fp64 oracle on the same bf16 inputs,
within the same tolerances as the single-pass forward.  The merge entry
point is compared with the oracle's float64 merge of the same partial
results.
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


def bits(*ts):
    return [inputs.bf16_bits(t) for t in ts]


def check(O, L, Or, Lr, what):
    O = O.detach().cpu().double().numpy()
    L = L.detach().cpu().double().numpy()
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L)), what
    eo, el = float(np.max(np.abs(O - Or))), float(np.max(np.abs(L - Lr)))
    assert eo <= TOL_O and el <= TOL_LSE, f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


CASES = [  # B, H, Nq, Nk, d, causal, splits
    (2, 4, 1, 8192, 128, False, 8),       # decode: one query row
    (4, 2, 17, 3000, 64, False, 5),       # ragged keys, ragged split sizes
    (1, 3, 700, 700, 128, True, 4),       # causal: early rows have empty ranges
    (1, 2, 1000, 1000, 64, True, 3),
    (2, 2, 300, 5000, 128, False, 64),    # more splits requested than useful
    (1, 1, 128, 129, 128, False, 2),      # second range is a single key
    (1, 2, 256, 100, 64, True, 4),        # one key tile: falls back to one pass
    (2, 2, 3, 5000, 256, False, 6),       # head dimension 256, decode-like
    (1, 2, 700, 900, 256, True, 3),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", CASES)
def test_splitkv_matches_oracle(dev, B, H, Nq, Nk, d, causal, splits):
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed=Nq + Nk + splits)
    scale = float(np.float32(1 / math.sqrt(d)))
    O, L = fa2.forward(Q.to(dev), K.to(dev), V.to(dev), causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None) == fa2.FA2_OK
    Or, Lr = oracle.attention(*bits(Q, K, V), causal, scale)
    check(O, L, Or, Lr, f"split-KV {(B, H, Nq, Nk, d, causal, splits)}")


@pytest.mark.parametrize("splits", [2, 4])
def test_splitkv_cross_length_workload(dev, splits):
    """The short-query / long-key workload at full size, sampled rows."""
    w = inputs.workload("b16_h32_nq128_nk8192_d128")
    Q, K, V = inputs.workload_inputs(w)
    O, L = fa2.forward(Q.to(dev), K.to(dev), V.to(dev), causal=w.causal, scale=w.scale, num_splits=splits)
    torch.cuda.synchronize()
    rng = np.random.default_rng(splits)
    rows = np.unique(np.concatenate([[0, w.Nq - 1, w.B * w.H * w.Nq - 1],
                                     rng.integers(0, w.B * w.H * w.Nq, 200)]))
    Or, Lr = oracle.attention_rows(*bits(Q, K, V), w.causal, w.scale, rows)
    idx = torch.as_tensor(rows, device=dev)
    check(O.reshape(-1, w.d)[idx], L.reshape(-1)[idx], Or, Lr, f"cross-length, {splits} splits")


def test_splitkv_equals_single_pass_closely(dev):
    Q, K, V = inputs.make_qkv(2, 4, 256, 4096, 128, seed=21)
    Q, K, V = Q.to(dev), K.to(dev), V.to(dev)
    O1, L1 = fa2.forward(Q, K, V, scale=0.0883883461356163)
    O4, L4 = fa2.forward(Q, K, V, scale=0.0883883461356163, num_splits=4)
    torch.cuda.synchronize()
    assert float((O1 - O4).abs().max()) < 5e-3 and float((L1 - L4).abs().max()) < 1e-4


def test_merge_matches_oracle_merge(dev):
    rng = np.random.default_rng(31)
    P, R, d = 5, 1000, 128
    O_parts = rng.standard_normal((P, R, d)).astype(np.float32)
    L_parts = (rng.standard_normal((P, R)) * 4).astype(np.float32)
    L_parts[1, :300] = -np.inf                      # empty parts for some rows
    L_parts[:, 7] = -np.inf                         # a row with no key at all
    O, L = fa2.merge(torch.from_numpy(O_parts).to(dev), torch.from_numpy(L_parts).to(dev))
    torch.cuda.synchronize()
    Or, Lr = oracle.merge(O_parts, L_parts)
    O, L = O.cpu().double().numpy(), L.cpu().double().numpy()
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isfinite(L), fin)
    assert np.max(np.abs(L[fin] - Lr[fin])) < 1e-5
    assert np.max(np.abs(O - Or)) < 1e-5
    assert np.all(O[7] == 0)


def test_merge_of_gpu_results_over_key_ranges(dev):
    """Ring-attention merge of forward results over three key ranges."""
    B, H, Nq, Nk, d = 1, 4, 300, 1200, 64
    Q, K, V = inputs.make_qkv(B, H, Nq, Nk, d, seed=41)
    cuts = [0, 256, 640, Nk]
    parts = [fa2.forward(Q.to(dev), K[:, :, a:b].contiguous().to(dev), V[:, :, a:b].contiguous().to(dev), scale=0.125)
             for a, b in zip(cuts[:-1], cuts[1:])]
    O, L = fa2.merge(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]))
    torch.cuda.synchronize()
    Or, Lr = oracle.attention(*bits(Q, K, V), False, 0.125)
    check(O, L, Or, Lr, "merged key ranges")


def test_splitkv_workspace_errors(dev):
    B, H, Nq, Nk, d = 1, 2, 64, 2048, 128
    q = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, H, Nk, d, dtype=torch.bfloat16, device=dev)
    o = torch.empty(B, H, Nq, d, device=dev)
    l = torch.empty(B, H, Nq, device=dev)
    need = fa2.fa2_splitkv_workspace_bytes(B, H, Nq, d, 4)
    assert need >= 4 * B * H * Nq * (d + 1) * 4
    ws = torch.empty(need + 512, dtype=torch.uint8, device=dev)
    args = (q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, Nq, Nk, d, 0, 0.1, 4)
    assert fa2.fa2_forward_splitkv(*args, None, need, None) == fa2.FA2_ERR_NULL
    assert fa2.fa2_forward_splitkv(*args, ws.data_ptr() + 16, need, None) == fa2.FA2_ERR_ALIGN
    assert fa2.fa2_forward_splitkv(*args, ws.data_ptr(), need - 1, None) == fa2.FA2_ERR_MEMORY
    bad = args[:-1] + (0,)
    assert fa2.fa2_forward_splitkv(*bad, ws.data_ptr(), need, None) == fa2.FA2_ERR_SHAPE
    assert fa2.fa2_forward_splitkv(*args, ws.data_ptr(), need, None) == fa2.FA2_OK
    torch.cuda.synchronize()


# Causal key ranges one key tile long on grids large enough for two query
# sub-tiles per CTA: ranges that only a CTA's second sub-tile reaches (its
# first has no kept key there) and ranges past both, on the kernel form whose
# issuing warp waits on named barriers.
@pytest.mark.parametrize("d", [64, 128])
def test_splitkv_two_subtile_grid_with_ranges_only_the_second_subtile_reaches(dev, d):
    B, H, N, splits = 1, 4, 4096, 32
    assert (N + 255) // 256 * B * H * splits >= 2 * torch.cuda.get_device_properties(0).multi_processor_count
    Q, K, V = inputs.make_qkv(B, H, N, N, d, seed=97 + d)
    scale = float(np.float32(1 / math.sqrt(d)))
    O, L = fa2.forward(Q.to(dev), K.to(dev), V.to(dev), causal=True, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(None) == fa2.FA2_OK
    Or, Lr = oracle.attention(*bits(Q, K, V), True, scale)
    check(O, L, Or, Lr, f"split-KV two-sub-tile grid d={d}")
