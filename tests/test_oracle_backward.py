"""Pins for the oracle's backward pass, independent of the oracle's own code.

The pages name the backward pass but print no formulas, so the oracle writes
out the chain rule of the attention definition.  These checks tie it to
things it does not compute itself: torch's float64 autograd of its own
attention routine (an independent library), central differences of torch's
float64 forward (which use no gradient code at all), closed forms and the
mathematics' invariants.  The last tests plant mistakes in copies of the
oracle source and check that the pins catch each one.
"""
import os
import shutil

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from test_oracle import from_bits, rand_bits, to_bits


def causal_keep(Nq, Nk):
    return torch.ones(Nq, Nk, dtype=torch.bool).tril()


def torch_grads(Qb, Kb, Vb, dOb, causal, scale):
    """float64 autograd of torch's attention (top-left causal mask given explicitly)."""
    q, k, v = (torch.from_numpy(from_bits(x)).requires_grad_(True) for x in (Qb, Kb, Vb))
    g = torch.from_numpy(from_bits(dOb))
    sc = float(np.float64(np.float32(scale)))
    mask = causal_keep(q.shape[2], k.shape[2]) if causal else None
    O = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=sc)
    O.backward(g)
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def flat(a):
    return a.reshape(-1, *a.shape[2:])


def check_against_autograd(orc):
    rng = np.random.default_rng(21)
    for (B, H, Nq, Nk, d, causal) in [(1, 2, 5, 7, 8, False), (2, 1, 9, 9, 16, True),
                                      (1, 1, 12, 5, 4, True), (1, 1, 4, 11, 8, True)]:
        Q, K, V, G = (rand_bits(rng, sh) for sh in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d), (B, H, Nq, d)))
        dQ, dK, dV = orc.attention_backward(Q, K, V, G, causal, 0.35)
        tq, tk, tv = torch_grads(Q, K, V, G, causal, 0.35)
        assert np.max(np.abs(dQ - flat(tq))) < 1e-12
        assert np.max(np.abs(dK - flat(tk))) < 1e-12
        assert np.max(np.abs(dV - flat(tv))) < 1e-12


def check_against_central_differences(orc):
    """The gradient of f = sum(O * dO) by central differences of torch's float64
    forward (no gradient code involved)."""
    rng = np.random.default_rng(22)
    B, H, Nq, Nk, d = 1, 1, 4, 6, 3
    for causal in (False, True):
        Q, K, V, G = (rand_bits(rng, sh) for sh in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d), (B, H, Nq, d)))
        dQ, dK, dV = orc.attention_backward(Q, K, V, G, causal, 0.5)
        base = [torch.from_numpy(from_bits(x)) for x in (Q, K, V)]
        g = torch.from_numpy(from_bits(G))
        mask = causal_keep(Nq, Nk) if causal else None

        def f(ts):
            return float((F.scaled_dot_product_attention(*ts, attn_mask=mask, scale=0.5) * g).sum())

        h = 1e-5
        for which, grad in ((0, dQ), (1, dK), (2, dV)):
            shape = base[which].shape
            for idx in np.ndindex(*shape[2:]):
                plus = [t.clone() for t in base]
                minus = [t.clone() for t in base]
                plus[which][(0, 0) + idx] += h
                minus[which][(0, 0) + idx] -= h
                fd = (f(plus) - f(minus)) / (2 * h)
                assert abs(fd - grad[(0,) + idx]) < 1e-7, (which, idx, fd, grad[(0,) + idx])


def check_closed_forms(orc):
    rng = np.random.default_rng(23)
    B, H, Nq, Nk, d = 1, 2, 6, 5, 8
    Q, V, G = rand_bits(rng, (B, H, Nq, d)), rand_bits(rng, (B, H, Nk, d)), rand_bits(rng, (B, H, Nq, d))
    g = from_bits(G)
    # K = 0: uniform weights, dQ = scale * sum_j ds_ij k_j = 0; dV_j = sum_i dO_i / Nk
    K0 = to_bits(np.zeros((B, H, Nk, d)))
    dQ, dK, dV = orc.attention_backward(Q, K0, V, G, False, 0.4)
    assert np.all(dQ == 0)
    assert np.allclose(dV, flat(g).sum(axis=1, keepdims=True) / Nk, atol=1e-14, rtol=0)
    # one key: p = 1, ds = 0 -> dQ = dK = 0, dV_0 = sum_i dO_i
    K1, V1 = rand_bits(rng, (B, H, 1, d)), rand_bits(rng, (B, H, 1, d))
    dQ, dK, dV = orc.attention_backward(Q, K1, V1, G, False, 0.4)
    assert np.max(np.abs(dQ)) < 1e-14 and np.max(np.abs(dK)) < 1e-14
    assert np.allclose(dV[:, 0], flat(g).sum(axis=1), atol=1e-14, rtol=0)
    # every V row equal: O is that row for every weighting, so ds = 0
    Vc = np.broadcast_to(from_bits(V)[:, :, :1], (B, H, Nk, d))
    K = rand_bits(rng, (B, H, Nk, d))
    for causal in (False, True):
        dQ, dK, dV = orc.attention_backward(Q, K, to_bits(Vc), G, causal, 0.4)
        assert np.max(np.abs(dQ)) < 1e-12 and np.max(np.abs(dK)) < 1e-12
    # causal row 0 keeps key 0 only: its weight is 1 whatever the scores
    dQ, dK, dV = orc.attention_backward(Q, K, V, G, True, 0.4)
    assert np.max(np.abs(dQ[:, 0])) < 1e-13


def check_invariants(orc):
    rng = np.random.default_rng(24)
    B, H, Nq, Nk, d = 1, 2, 7, 9, 8
    Q, K, V, G = (rand_bits(rng, sh) for sh in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d), (B, H, Nq, d)))
    g = flat(from_bits(G))
    for causal in (False, True):
        dQ, dK, dV, mQ, mK, mV = orc.attention_backward(Q, K, V, G, causal, 0.3, magnitudes=True)
        # softmax weights of each row sum to 1: sum_j dV_j = sum_i dO_i
        assert np.allclose(dV.sum(axis=1), g.sum(axis=1), atol=1e-12, rtol=0)
        # the rows of ds sum to 0: sum_j dK_j = scale sum_i (sum_j ds_ij) q_i = 0
        assert np.max(np.abs(dK.sum(axis=1))) < 1e-12
        # each element is bounded by the sum of its terms' magnitudes
        for a, m in ((dQ, mQ), (dK, mK), (dV, mV)):
            assert np.all(np.abs(a) <= m + 1e-15)
    # a joint permutation of the keys permutes dK and dV and leaves dQ (non-causal)
    perm = rng.permutation(Nk)
    dQ, dK, dV = orc.attention_backward(Q, K, V, G, False, 0.3)
    pQ, pK, pV = orc.attention_backward(Q, np.ascontiguousarray(K[:, :, perm]),
                                        np.ascontiguousarray(V[:, :, perm]), G, False, 0.3)
    assert np.allclose(pQ, dQ, atol=1e-13, rtol=0)
    assert np.allclose(pK, dK[:, perm], atol=1e-13, rtol=0)
    assert np.allclose(pV, dV[:, perm], atol=1e-13, rtol=0)
    # selected heads equal the matching slices of the all-heads result
    sQ, sK, sV = orc.attention_backward(Q, K, V, G, True, 0.3, heads=[1])
    aQ, aK, aV = orc.attention_backward(Q, K, V, G, True, 0.3)
    assert np.array_equal(sQ[0], aQ[1]) and np.array_equal(sK[0], aK[1]) and np.array_equal(sV[0], aV[1])


def check_fp16(orc):
    rng = np.random.default_rng(25)
    sh = (1, 1, 6, 8)
    Q, K, V, G = (rng.standard_normal(sh).astype(np.float16) for _ in range(4))
    dQ, dK, dV = orc.attention_backward(Q.view(np.uint16), K.view(np.uint16), V.view(np.uint16),
                                        G.view(np.uint16), True, 0.5, dtype="fp16")
    q, k, v = (torch.from_numpy(x.astype(np.float64)).requires_grad_(True) for x in (Q, K, V))
    O = F.scaled_dot_product_attention(q, k, v, attn_mask=causal_keep(6, 6), scale=0.5)
    O.backward(torch.from_numpy(G.astype(np.float64)))
    assert np.max(np.abs(dQ - flat(q.grad.numpy()))) < 1e-12
    assert np.max(np.abs(dK - flat(k.grad.numpy()))) < 1e-12
    assert np.max(np.abs(dV - flat(v.grad.numpy()))) < 1e-12


def magnitudes_from_definition(Qb, Kb, Vb, dOb, causal, scale):
    """The magnitudes M_dQ, M_dK, M_dV recomputed from their definitions in
    torch float64, sharing nothing with the oracle's C code: the weights p
    come from torch's softmax, ds = dL/ds from torch's autograd through that
    softmax (L = sum(O * dO)), and A_i = sum_j p_ij sum_c |dO_ic| |v_jc|.
        M_dV = p^T |dO|
        M_dQ = scale (|ds| + p A) |K|
        M_dK = scale (|ds| + p A)^T |Q|"""
    q, k, v, g = (torch.from_numpy(from_bits(x)) for x in (Qb, Kb, Vb, dOb))
    sc = float(np.float64(np.float32(scale)))
    s = (sc * q @ k.transpose(-1, -2)).requires_grad_(True)
    if causal:
        s_masked = s.masked_fill(~causal_keep(q.shape[2], k.shape[2]), float("-inf"))
    else:
        s_masked = s
    p = torch.softmax(s_masked, dim=-1)
    (p @ v * g).sum().backward()
    ds = s.grad.abs()
    p = p.detach()
    A = (p * (g.abs() @ v.abs().transpose(-1, -2))).sum(-1, keepdim=True)
    w = ds + p * A
    mq = sc * w @ k.abs()
    mk = sc * w.transpose(-1, -2) @ q.abs()
    mv = p.transpose(-1, -2) @ g.abs()
    return flat(mq.numpy()), flat(mk.numpy()), flat(mv.numpy())


def check_magnitudes(orc):
    """The per-element magnitudes that set the GPU tests' gradient bound equal
    their definitions (an independent recomputation), so that a magnitude
    that is too large -- which would loosen the GPU bound silently -- fails
    here."""
    rng = np.random.default_rng(26)
    for (B, H, Nq, Nk, d, causal, scale) in [(1, 2, 6, 9, 8, False, 0.35), (2, 1, 9, 9, 16, True, 0.3),
                                             (1, 1, 12, 5, 4, True, 0.6), (1, 1, 4, 11, 8, True, 0.25)]:
        Q, K, V, G = (rand_bits(rng, sh) for sh in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d), (B, H, Nq, d)))
        _, _, _, mQ, mK, mV = orc.attention_backward(Q, K, V, G, causal, scale, magnitudes=True)
        rq, rk, rv = magnitudes_from_definition(Q, K, V, G, causal, scale)
        for got, ref in ((mQ, rq), (mK, rk), (mV, rv)):
            assert got.shape == ref.shape
            assert np.all(np.abs(got - ref) <= 1e-12 * np.maximum(np.abs(ref), 1e-300) + 1e-300)


CHECKS = (check_against_autograd, check_against_central_differences, check_closed_forms,
          check_invariants, check_fp16, check_magnitudes)


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_backward_pin(oracle_mod, check):
    check(oracle_mod._default())


def test_bad_arguments(oracle_mod):
    orc = oracle_mod._default()
    z = np.zeros((1, 1, 2, 4), dtype=np.uint16)
    with pytest.raises(ValueError):
        orc.attention_backward(z, np.zeros((1, 1, 0, 4), dtype=np.uint16),
                               np.zeros((1, 1, 0, 4), dtype=np.uint16), z, False, 1.0)
    with pytest.raises(ValueError):
        orc.attention_backward(z, z, z, z, False, 1.0, heads=[3])


def all_backward_pins(orc):
    for check in CHECKS:
        try:
            check(orc)
        except AssertionError:
            return False, check.__name__
    return True, None


# Planted mistakes in the backward half of the oracle source: each must fail a pin.
MUTANTS = {
    "dropped_row_term": ("const double ds = exp(s[j] - lse) * (dp[j] - D);",
                         "const double ds = exp(s[j] - lse) * (dp[j]);"),
    "row_term_without_weights": ("D += exp(s[j] - lse) * dp[j];", "D += dp[j];"),
    "dK_without_scale": ("dk[c] += J->scale * ds * qc;", "dk[c] += ds * qc;"),
    "dV_from_ds": ("dv[c] += p * gc;", "dv[c] += ds * gc;"),
    "causal_key_off_by_one": ("if (j >= kept_keys(J, i))", "if (j > kept_keys(J, i))"),
    "dQ_from_q": ("const double kc = widen(kb[j * d + c], J->dtype);",
                  "const double kc = widen(q[c], J->dtype);"),
    "dp_from_k": ("gv += widen(gb[i * d + c], J->dtype) * widen(v[c], J->dtype);",
                  "gv += widen(gb[i * d + c], J->dtype) * widen(k[c], J->dtype);"),
    "weights_without_scale": ("const double p = exp(J->scale * acc - J->LSE[i]);",
                              "const double p = exp(acc - J->LSE[i]);"),
    "row_term_in_key_pass": ("const double ds = p * (gv - J->Dr[i]);", "const double ds = p * gv;"),
    # mistakes that only inflate the magnitudes M (and so would loosen the GPU bound)
    "magnitude_A_doubled": ("A += exp(s[j] - lse) * da[j];", "A += 2.0 * exp(s[j] - lse) * da[j];"),
    "magnitude_ds_doubled_in_query_pass": ("const double w = fabs(ds) + exp(s[j] - lse) * A;",
                                           "const double w = 2.0 * fabs(ds) + exp(s[j] - lse) * A;"),
    "magnitude_A_doubled_in_key_pass": ("const double w = fabs(ds) + p * J->Ar[i];",
                                        "const double w = fabs(ds) + 2.0 * p * J->Ar[i];"),
    "magnitude_dQ_without_scale": ("mq[c] += J->scale * w * fabs(kc);", "mq[c] += w * fabs(kc);"),
    "magnitude_dK_without_scale": ("mk[c] += J->scale * w * fabs(qc);", "mk[c] += w * fabs(qc);"),
    "magnitude_dV_without_weights": ("mv[c] += p * fabs(gc);", "mv[c] += fabs(gc);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_pins_catch_planted_mistake(oracle_mod, tmp_path, name):
    src = os.path.join(os.path.dirname(oracle_mod.__file__), "attn_ref.c")
    text = open(src).read()
    old, new = MUTANTS[name]
    assert text.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    path = tmp_path / "mutant.c"
    path.write_text(text.replace(old, new))
    lib = oracle_mod.compile_source(str(path), str(tmp_path / f"mutant_{name}.so"))
    ok, _ = all_backward_pins(oracle_mod.Oracle(lib))
    assert not ok, f"planted mistake {name} passed every backward pin"


def test_backward_pins_pass_on_unmodified_copy(oracle_mod, tmp_path):
    src = os.path.join(os.path.dirname(oracle_mod.__file__), "attn_ref.c")
    shutil.copy(src, tmp_path / "copy.c")
    lib = oracle_mod.compile_source(str(tmp_path / "copy.c"), str(tmp_path / "copy.so"))
    ok, failed = all_backward_pins(oracle_mod.Oracle(lib))
    assert ok, failed
