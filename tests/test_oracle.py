"""Pins for the fp64 oracle, independent of the oracle's own code.

Each check ties the oracle to something it does not compute itself: the
numbers the pages print for their worked example, an independent library
routine (torch's float64 CPU attention and logsumexp), closed forms, the
mathematics' invariants, high-precision brute force, and a tiled
online-softmax restatement of the method.  The last test plants mistakes in
copies of the oracle's C source and checks that these pins catch each one.
"""
import decimal
import math
import os
import re
import shutil

import numpy as np
import pytest
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_online_softmax.txt")


def to_bits(a) -> np.ndarray:
    """float array -> bf16 bit patterns (RNE); values in the tests are chosen exact in bf16."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bits(rng, shape, std=1.0):
    return to_bits(rng.standard_normal(shape) * std)


def read_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = [x.strip() for x in line.split("=", 1)]
                vals[k] = v
    return vals


def torch_reference(Qb, Kb, Vb, causal, scale):
    """Library routine in float64: torch SDPA for O, torch.logsumexp for LSE."""
    q, k, v = (torch.from_numpy(from_bits(x)) for x in (Qb, Kb, Vb))
    Nq, Nk = q.shape[2], k.shape[2]
    sc = torch.tensor(np.float64(np.float32(scale)), dtype=torch.float64)
    O = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=float(sc))
    s = (q @ k.transpose(-1, -2)) * sc
    if causal:
        keep = torch.ones(Nq, Nk, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, float("-inf"))
    return O.numpy(), torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------- worked example

def worked_example_inputs(scores):
    """d = n: q = e_0, k_j = scores[j] e_0, V = identity, scale 1 -> weights = softmax(scores)."""
    n = len(scores)
    Q = np.zeros((1, 1, 1, n)); Q[0, 0, 0, 0] = 1.0
    K = np.zeros((1, 1, n, n)); K[0, 0, :, 0] = scores
    V = np.eye(n).reshape(1, 1, n, n)
    return to_bits(Q), to_bits(K), to_bits(V)


def check_worked_example(orc):
    g = read_golden()
    scores = [float(x) for x in g["scores"].split()]
    bc = int(g["block_size"])
    places = int(g["printed_decimals"])
    tol = 0.5 * 10 ** -places + 1e-12
    # block 1 alone: running max and sum after the first block
    Q, K, V = worked_example_inputs(scores[:bc])
    O1, L1 = orc.attention(Q, K, V, False, 1.0)
    m1 = max(scores[:bc])
    assert m1 == float(g["m_after_block1"])
    assert abs(math.exp(L1[0, 0, 0] - m1) - float(g["l_after_block1"])) <= tol
    # both blocks: the one-shot sum equals the page's blockwise value
    Q, K, V = worked_example_inputs(scores)
    O, L = orc.attention(Q, K, V, False, 1.0)
    m2 = max(scores)
    assert m2 == float(g["m_after_block2"])
    assert abs(math.exp(L[0, 0, 0] - m2) - float(g["l_after_block2"])) <= tol
    # with V = I the output row is the softmax of the scores (library routine)
    ref = torch.softmax(torch.tensor(scores, dtype=torch.float64), 0).numpy()
    assert np.allclose(O[0, 0, 0], ref, rtol=0, atol=1e-14)
    assert abs(O[0, 0, 0].sum() - 1.0) < 1e-14


def test_worked_example(oracle_mod):
    check_worked_example(oracle_mod)


def test_worked_example_blockwise_recurrence(oracle_mod):
    """The page's blockwise update (l2 = l1 e^(m1-m2) + sum of the new block) gives the oracle's l."""
    g = read_golden()
    scores = [float(x) for x in g["scores"].split()]
    Q, K, V = worked_example_inputs(scores[:2])
    _, L1 = oracle_mod.attention(Q, K, V, False, 1.0)
    Q, K, V = worked_example_inputs(scores)
    _, L = oracle_mod.attention(Q, K, V, False, 1.0)
    m1, m2 = 3.0, 5.0
    l1 = math.exp(L1[0, 0, 0] - m1)
    l2 = l1 * math.exp(m1 - m2) + math.exp(2.0 - m2) + math.exp(5.0 - m2)
    assert abs(l2 - math.exp(L[0, 0, 0] - m2)) < 1e-14


# ---------------------------------------------------------------- library routine

SHAPES = [
    (1, 1, 1, 1, 1), (1, 1, 5, 7, 4), (2, 3, 9, 9, 16), (1, 2, 17, 5, 8),
    (1, 1, 33, 64, 64), (2, 1, 64, 33, 64), (1, 1, 20, 20, 128), (1, 2, 19, 23, 256),
]


def check_against_torch(orc, seed=0, shapes=SHAPES, tol=1e-12):
    rng = np.random.default_rng(seed)
    for (B, H, Nq, Nk, d) in shapes:
        for causal in (False, True):
            Q, K, V = rand_bits(rng, (B, H, Nq, d)), rand_bits(rng, (B, H, Nk, d)), rand_bits(rng, (B, H, Nk, d))
            scale = float(np.float32(1 / math.sqrt(d)))
            O, L = orc.attention(Q, K, V, causal, scale)
            Ot, Lt = torch_reference(Q, K, V, causal, scale)
            assert np.max(np.abs(O - Ot)) < tol, (B, H, Nq, Nk, d, causal)
            assert np.max(np.abs(L - Lt)) < tol, (B, H, Nq, Nk, d, causal)


def test_against_torch_float64(oracle_mod):
    check_against_torch(oracle_mod)


def test_rows_api_matches_full(oracle_mod):
    rng = np.random.default_rng(3)
    B, H, Nq, Nk, d = 2, 3, 37, 29, 16
    Q, K, V = rand_bits(rng, (B, H, Nq, d)), rand_bits(rng, (B, H, Nk, d)), rand_bits(rng, (B, H, Nk, d))
    for causal in (False, True):
        O, L = oracle_mod.attention(Q, K, V, causal, 0.25)
        rows = rng.permutation(B * H * Nq)[:50]
        Or, Lr = oracle_mod.attention_rows(Q, K, V, causal, 0.25, rows)
        assert np.array_equal(Or, O.reshape(-1, d)[rows])
        assert np.array_equal(Lr, L.reshape(-1)[rows])


def test_thread_count_does_not_change_bits(oracle_mod):
    rng = np.random.default_rng(4)
    Q, K, V = rand_bits(rng, (1, 4, 50, 32)), rand_bits(rng, (1, 4, 70, 32)), rand_bits(rng, (1, 4, 70, 32))
    a = oracle_mod.attention(Q, K, V, True, 0.2, nthreads=1)
    b = oracle_mod.attention(Q, K, V, True, 0.2, nthreads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_arguments(oracle_mod):
    Q = to_bits(np.zeros((1, 1, 2, 4)))
    K = to_bits(np.zeros((1, 1, 0, 4)))
    with pytest.raises(ValueError):
        oracle_mod.attention(Q, K, K, False, 1.0)       # Nk = 0: softmax over nothing
    K = to_bits(np.zeros((1, 1, 3, 4)))
    with pytest.raises(ValueError):
        oracle_mod.attention_rows(Q, K, K, False, 1.0, [2])  # row id out of range


# ---------------------------------------------------------------- brute force

def test_brute_force_high_precision(oracle_mod):
    """40-digit decimal evaluation of the definition on a tiny case."""
    decimal.getcontext().prec = 40
    D = decimal.Decimal
    rng = np.random.default_rng(5)
    B, H, Nq, Nk, d = 1, 1, 3, 5, 3
    Q, K, V = rand_bits(rng, (B, H, Nq, d)), rand_bits(rng, (B, H, Nk, d)), rand_bits(rng, (B, H, Nk, d))
    scale = float(np.float32(0.7))
    q, k, v = from_bits(Q)[0, 0], from_bits(K)[0, 0], from_bits(V)[0, 0]
    for causal in (False, True):
        O, L = oracle_mod.attention(Q, K, V, causal, scale)
        for i in range(Nq):
            keep = range(Nk) if not causal else range(min(i + 1, Nk))
            s = [D(scale) * sum(D(q[i, c]) * D(k[j, c]) for c in range(d)) for j in keep]
            z = sum(x.exp() for x in s)
            assert abs(float(z.ln()) - L[0, 0, i]) < 1e-13
            for c in range(d):
                o = sum(s_j.exp() / z * D(v[j, c]) for s_j, j in zip(s, keep))
                assert abs(float(o) - O[0, 0, i, c]) < 1e-13


# ---------------------------------------------------------------- closed forms

def check_closed_forms(orc):
    rng = np.random.default_rng(6)
    # K = 0: every kept key has score 0 -> uniform weights, LSE = ln |J_i|
    for (Nq, Nk, causal) in [(8, 8, False), (8, 8, True), (5, 9, True), (9, 5, True)]:
        d = 8
        Q, V = rand_bits(rng, (1, 2, Nq, d)), rand_bits(rng, (1, 2, Nk, d))
        K = to_bits(np.zeros((1, 2, Nk, d)))
        O, L = orc.attention(Q, K, V, causal, 0.5)
        v = from_bits(V)
        for i in range(Nq):
            n = min(i + 1, Nk) if causal else Nk
            assert np.allclose(O[:, :, i], v[:, :, :n].mean(axis=2), atol=1e-14, rtol=0)
            assert np.allclose(L[:, :, i], math.log(n), atol=1e-14, rtol=0)
    # one key: weight 1, LSE = the score itself
    Q, K, V = rand_bits(rng, (2, 1, 6, 4)), rand_bits(rng, (2, 1, 1, 4)), rand_bits(rng, (2, 1, 1, 4))
    for causal in (False, True):
        O, L = orc.attention(Q, K, V, causal, 0.5)
        q, k, v = from_bits(Q), from_bits(K), from_bits(V)
        assert np.array_equal(O, np.broadcast_to(v, O.shape))
        s = 0.5 * np.einsum("bhid,bhjd->bhi", q, k)
        assert np.allclose(L, s, atol=1e-14, rtol=0)
    # causal row 0 keeps only key 0
    Q, K, V = rand_bits(rng, (1, 3, 4, 16)), rand_bits(rng, (1, 3, 4, 16)), rand_bits(rng, (1, 3, 4, 16))
    O, L = orc.attention(Q, K, V, True, 0.25)
    q, k, v = from_bits(Q), from_bits(K), from_bits(V)
    assert np.array_equal(O[:, :, 0], v[:, :, 0])
    assert np.allclose(L[:, :, 0], 0.25 * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-14, rtol=0)
    # a dominant key (score 64 above the rest) takes all the weight
    d, Nk = 4, 6
    Q = np.zeros((1, 1, 1, d)); Q[..., 0] = 1.0
    K = np.zeros((1, 1, Nk, d)); K[..., 3, 0] = 64.0
    V = rng.integers(-4, 5, size=(1, 1, Nk, d)).astype(np.float64)
    O, L = orc.attention(to_bits(Q), to_bits(K), to_bits(V), False, 1.0)
    assert np.allclose(O[0, 0, 0], V[0, 0, 3], atol=1e-25, rtol=1e-15)
    assert abs(L[0, 0, 0] - 64.0) < 1e-25 + 1e-15 * 64


def test_closed_forms(oracle_mod):
    check_closed_forms(oracle_mod)


# ---------------------------------------------------------------- invariants

def check_invariants(orc):
    rng = np.random.default_rng(7)
    B, H, Nq, Nk, d = 1, 2, 24, 40, 16
    Q, K, V = rand_bits(rng, (B, H, Nq, d), 2.0), rand_bits(rng, (B, H, Nk, d), 2.0), rand_bits(rng, (B, H, Nk, d))
    q, k, v = from_bits(Q), from_bits(K), from_bits(V)
    scale = 0.25
    for causal in (False, True):
        O, L = orc.attention(Q, K, V, causal, scale)
        s = scale * np.einsum("bhid,bhjd->bhij", q, k)
        for i in range(Nq):
            n = min(i + 1, Nk) if causal else Nk
            vi = v[:, :, :n]
            # rows of O are convex combinations of the kept V rows
            assert np.all(O[:, :, i] >= vi.min(axis=2) - 1e-12)
            assert np.all(O[:, :, i] <= vi.max(axis=2) + 1e-12)
            # max s <= LSE <= max s + ln n
            smax = s[:, :, i, :n].max(axis=-1)
            assert np.all(L[:, :, i] >= smax - 1e-12)
            assert np.all(L[:, :, i] <= smax + math.log(n) + 1e-12)
    # weights sum to one: V = 1 gives O = 1
    ones = to_bits(np.ones((B, H, Nk, d)))
    for causal in (False, True):
        O, _ = orc.attention(Q, K, ones, causal, scale)
        assert np.allclose(O, 1.0, atol=1e-14, rtol=0)
    # jointly permuting K and V rows does not change a non-causal result
    perm = rng.permutation(Nk)
    O1, L1 = orc.attention(Q, K, V, False, scale)
    O2, L2 = orc.attention(Q, np.ascontiguousarray(K[:, :, perm]), np.ascontiguousarray(V[:, :, perm]), False, scale)
    assert np.allclose(O1, O2, atol=1e-13, rtol=0) and np.allclose(L1, L2, atol=1e-13, rtol=0)
    # permuting only V (not K) does change it
    O3, _ = orc.attention(Q, K, np.ascontiguousarray(V[:, :, perm]), False, scale)
    assert not np.allclose(O1, O3, atol=1e-6)


def test_invariants(oracle_mod):
    check_invariants(oracle_mod)


def check_lse_merge(orc):
    """Ring-attention merge of two key halves ("FlashAttention 怎么做?", 多卡 question):
    L = log(e^L1 + e^L2), O = e^(L1-L) O1 + e^(L2-L) O2 equals the full result."""
    rng = np.random.default_rng(8)
    B, H, Nq, Nk, d = 2, 2, 19, 50, 32
    Q, K, V = rand_bits(rng, (B, H, Nq, d), 2.0), rand_bits(rng, (B, H, Nk, d), 2.0), rand_bits(rng, (B, H, Nk, d))
    O, L = orc.attention(Q, K, V, False, 0.3)
    h = 21
    O1, L1 = orc.attention(Q, np.ascontiguousarray(K[:, :, :h]), np.ascontiguousarray(V[:, :, :h]), False, 0.3)
    O2, L2 = orc.attention(Q, np.ascontiguousarray(K[:, :, h:]), np.ascontiguousarray(V[:, :, h:]), False, 0.3)
    Lm = np.logaddexp(L1, L2)
    Om = np.exp(L1 - Lm)[..., None] * O1 + np.exp(L2 - Lm)[..., None] * O2
    assert np.allclose(L, Lm, atol=1e-12, rtol=0)
    assert np.allclose(O, Om, atol=1e-12, rtol=0)


def test_lse_merge_identity(oracle_mod):
    check_lse_merge(oracle_mod)


# ---------------------------------------------------------------- tiled restatement

def tiled_forward(q, k, v, scale, causal, bc):
    """Online softmax over key blocks of size bc, written from the update rules
    in "FlashAttention 怎么做?" (推导 / 关键公式): m' = max(m, rowmax S),
    P = e^(S - m'), l' = e^(m - m') l + rowsum P, O' = e^(m - m') O + P V,
    then O / l and L = m + log l once at the end.  Masked keys score -inf."""
    Nq, d = q.shape
    Nk = k.shape[0]
    m = np.full(Nq, -np.inf)
    l = np.zeros(Nq)
    O = np.zeros((Nq, d))
    rows = np.arange(Nq)[:, None]
    for j0 in range(0, Nk, bc):
        kj, vj = k[j0:j0 + bc], v[j0:j0 + bc]
        S = scale * (q @ kj.T)
        if causal:
            cols = np.arange(j0, j0 + kj.shape[0])[None, :]
            S = np.where(cols > rows, -np.inf, S)
        m_new = np.maximum(m, S.max(axis=1))
        P = np.exp(S - m_new[:, None])
        a = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        l = a * l + P.sum(axis=1)
        O = a[:, None] * O + P @ vj
        m = m_new
    return O / l[:, None], m + np.log(l)


def test_tiled_online_softmax_matches_oracle(oracle_mod):
    """The self-check of the NumPy listing's page (seed 0, (100, 32), Bc = 16,
    a ragged last block), plus causal and cross-length cases."""
    rng = np.random.default_rng(0)
    cases = [(100, 100, 32, False, 16), (100, 100, 32, True, 16), (37, 100, 32, True, 16),
             (100, 37, 64, True, 8), (1, 300, 16, False, 128), (130, 130, 8, True, 64)]
    for Nq, Nk, d, causal, bc in cases:
        Q, K, V = rand_bits(rng, (1, 1, Nq, d)), rand_bits(rng, (1, 1, Nk, d)), rand_bits(rng, (1, 1, Nk, d))
        scale = float(np.float32(1 / math.sqrt(d)))
        O, L = oracle_mod.attention(Q, K, V, causal, scale)
        Ot, Lt = tiled_forward(from_bits(Q)[0, 0], from_bits(K)[0, 0], from_bits(V)[0, 0],
                               np.float64(np.float32(scale)), causal, bc)
        assert np.allclose(O[0, 0], Ot, atol=1e-12, rtol=0)
        assert np.allclose(L[0, 0], Lt, atol=1e-12, rtol=0)


# ---------------------------------------------------------------- planted mistakes

MUTANTS = {
    "max_wrong_direction": ("if (s[j] > m)", "if (s[j] < m)"),
    "scale_dropped": ("s[j] = J->scale * acc;", "s[j] = acc;"),
    "causal_off_by_one_short": ("n = i + 1;", "n = (i > 0 ? i : 1);"),
    "causal_off_by_one_long": ("if (J->causal && i + 1 < n)\n        n = i + 1;",
                               "if (J->causal && i + 2 < n)\n        n = i + 2;"),
    "causal_ignored": ("if (J->causal && i + 1 < n)", "if (0 && i + 1 < n)"),
    "normaliser_sign": ("l += exp(s[j] - m);", "l += exp(m - s[j]);"),
    "normaliser_dropped": ("exp(s[j] - m) / l;", "exp(s[j] - m);"),
    "lse_max_dropped": ("*lse = m + log(l);", "*lse = log(l);"),
    "lse_log_dropped": ("*lse = m + log(l);", "*lse = m;"),
    "v_rows_reversed": ("vb[j * d + c]", "vb[(n - 1 - j) * d + c]"),
    "q_transposed": ("widen(q[c], J->dtype)", "widen(q[d - 1 - c], J->dtype)"),
    "fp16_exponent_bias": ("exponent - 25", "exponent - 24"),
    "fp16_subnormal_scale": ("ldexp((double)fraction, -24)", "ldexp((double)fraction, -25)"),
    "fp16_implicit_bit": ("(fraction | 0x400)", "(fraction)"),
    "k_from_query_block": ("const uint16_t *kb = J->K + bh * J->Nk * d;",
                           "const uint16_t *kb = J->K + (bh > 0 ? bh - 1 : 0) * J->Nk * d;"),
    "widening_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
}


def check_fp16_widening(orc):
    """Every finite binary16 pattern widens to the value torch's float16 -> float64
    conversion gives (a library routine), and fp16 attention matches torch."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    finite = np.isfinite(ref)
    got = np.array([orc.widen(int(b), "fp16") for b in bits[finite]])
    assert np.array_equal(got, ref[finite])
    rng = np.random.default_rng(14)
    for causal in (False, True):
        q, k, v = (rng.standard_normal(sh).astype(np.float16) for sh in ((1, 2, 9, 16), (1, 2, 12, 16), (1, 2, 12, 16)))
        O, L = orc.attention(q.view(np.uint16), k.view(np.uint16), v.view(np.uint16), causal, 0.25, dtype="fp16")
        qt, kt, vt = (torch.from_numpy(x.astype(np.float64)) for x in (q, k, v))
        Ot = F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=0.25).numpy()
        assert np.max(np.abs(O - Ot)) < 1e-12


def test_fp16_widening_and_attention(oracle_mod):
    check_fp16_widening(oracle_mod)


def all_pins(orc):
    for check in (check_worked_example, check_against_torch, check_closed_forms,
                  check_invariants, check_lse_merge, check_fp16_widening):
        try:
            check(orc)
        except AssertionError:
            return False, check.__name__
    return True, None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(oracle_mod, tmp_path, name):
    src = os.path.join(os.path.dirname(oracle_mod.__file__), "attn_ref.c")
    text = open(src).read()
    old, new = MUTANTS[name]
    assert text.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    mutated = text.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle_mod.compile_source(str(path), str(tmp_path / f"mutant_{name}.so"))
    ok, _ = all_pins(oracle_mod.Oracle(lib))
    assert not ok, f"planted mistake {name} passed every pin"


def test_pins_pass_on_unmodified_copy(oracle_mod, tmp_path):
    src = os.path.join(os.path.dirname(oracle_mod.__file__), "attn_ref.c")
    shutil.copy(src, tmp_path / "copy.c")
    lib = oracle_mod.compile_source(str(tmp_path / "copy.c"), str(tmp_path / "copy.so"))
    ok, failed = all_pins(oracle_mod.Oracle(lib))
    assert ok, failed


# ---------------------------------------------------------------- merge of partial results

def test_merge_of_key_partitions_equals_full(oracle_mod):
    """Merging the oracle's results over a partition of the keys (any number
    of parts, uneven, one part empty under the causal mask) gives the oracle's
    result over all keys."""
    rng = np.random.default_rng(12)
    B, H, Nq, Nk, d = 1, 2, 30, 70, 16
    Q, K, V = rand_bits(rng, (B, H, Nq, d), 2.0), rand_bits(rng, (B, H, Nk, d), 2.0), rand_bits(rng, (B, H, Nk, d))
    cuts = [0, 7, 31, 32, 58, 70]
    O, L = oracle_mod.attention(Q, K, V, False, 0.3)
    parts = [oracle_mod.attention(Q, np.ascontiguousarray(K[:, :, a:b]), np.ascontiguousarray(V[:, :, a:b]), False, 0.3)
             for a, b in zip(cuts[:-1], cuts[1:])]
    Om, Lm = oracle_mod.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(Om, O, atol=1e-12, rtol=0) and np.allclose(Lm, L, atol=1e-12, rtol=0)


def test_merge_closed_forms(oracle_mod):
    rng = np.random.default_rng(13)
    O1 = rng.standard_normal((5, 8))
    L1 = rng.standard_normal(5)
    # one part: identity
    O, L = oracle_mod.merge(O1[None], L1[None])
    assert np.allclose(O, O1) and np.allclose(L, L1)
    # two equal parts: same O, LSE + log 2
    O, L = oracle_mod.merge(np.stack([O1, O1]), np.stack([L1, L1]))
    assert np.allclose(O, O1, atol=1e-15) and np.allclose(L, L1 + math.log(2), atol=1e-15)
    # an empty part (-inf) contributes nothing; all parts empty -> O = 0, LSE = -inf
    Linf = np.full(5, -np.inf)
    O, L = oracle_mod.merge(np.stack([O1, rng.standard_normal((5, 8))]), np.stack([L1, Linf]))
    assert np.allclose(O, O1) and np.allclose(L, L1)
    O, L = oracle_mod.merge(np.stack([O1, O1]), np.stack([Linf, Linf]))
    assert np.all(O == 0) and np.all(np.isneginf(L))
    # weights follow the pages' two-part formula e^(L1-L), e^(L2-L)
    O2, L2 = rng.standard_normal((5, 8)), rng.standard_normal(5)
    O, L = oracle_mod.merge(np.stack([O1, O2]), np.stack([L1, L2]))
    Lr = np.log(np.exp(L1) + np.exp(L2))
    assert np.allclose(L, Lr, atol=1e-14)
    assert np.allclose(O, np.exp(L1 - Lr)[:, None] * O1 + np.exp(L2 - Lr)[:, None] * O2, atol=1e-14)
