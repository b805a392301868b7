"""Model of the forward kernels' choice of the softmax exponent offset.

The online softmax of "FlashAttention-2 算法架构升级" §三 (and the update
equations of "FlashAttention 怎么做?online softmax 怎么更新?", 关键公式)
rescales the running sum and output whenever the row max grows.  The
one-CTA forward kernel keeps an offset m per row (log2 units) that moves only
when a tile's scores exceed it by more than 8, so every term P = 2^(t - m)
stays <= 2^8, and it takes the row max of a tile only when it may have to
move: once m is finite it computes the exponentials with m as it stands, and
only when their row sum exceeds 2^8 (which every move implies, since the sum
is at least its largest term) takes the max, decides, and redoes them.

This file restates both orders (max first, and exponentials first) in
float32 numpy with one row at a time, and checks on seeded rows -- Gaussian
scores, rising maxima, one dominant key, masked keys and rows whose first
tiles are fully masked -- that

* the two orders choose the same offsets and produce the same P and sums;
* no term ever exceeds 2^8;
* O / l and the LSE equal the exact softmax (float64) to float32 rounding.

Planted mistakes (a bound of 2^16 on the sum, no max-first step while the
offset is still -inf, exponentials not redone after a move) must each fail
one of these checks.
"""
import numpy as np
import pytest

LOG2E = np.float32(1.4426950408889634)
RESCALE_LOG2 = np.float32(8.0)
BOUND = np.float32(256.0)
TILE = 128


def _exps(s, sl2, m):
    off = np.float32(0.0) if m == -np.inf else m
    with np.errstate(over="ignore"):
        t = (s * sl2 - off).astype(np.float32)
        p = np.exp2(t).astype(np.float32)
    return p, np.float32(p.sum(dtype=np.float32))


def _decide(s, sl2, m, first):
    mx = np.float32(s.max())
    m_cand = np.float32(max(m, np.float32(mx * sl2)))
    move = first or (m_cand > m + RESCALE_LOG2)
    m_new = m_cand if move else m
    if not move:
        alpha = np.float32(1.0)
    elif m == -np.inf:
        alpha = np.float32(0.0)
    else:
        alpha = np.float32(np.exp2(np.float32(m - m_new)))
    return m_new, alpha


def run_row(tiles, sl2, order, bound=BOUND, max_first_at_inf=True, redo=True):
    """One row over its key tiles; returns (weights per key, l, m, offsets, P tiles)."""
    m = np.float32(-np.inf)
    l = np.float32(0.0)
    acc = np.zeros(0, np.float64)     # running output weights per key (stands for O)
    offsets, ptiles = [], []
    for j, s in enumerate(tiles):
        if order == "max_first" or (max_first_at_inf and m == -np.inf):
            m_new, alpha = _decide(s, sl2, m, j == 0)
            p, rs = _exps(s, sl2, m_new)
        else:
            m_new, alpha = m, np.float32(1.0)
            p, rs = _exps(s, sl2, m_new)
            if not rs <= bound:
                m_new, alpha = _decide(s, sl2, m, j == 0)
                if redo:
                    p, rs = _exps(s, sl2, m_new)
        l = np.float32(l * alpha + rs)
        acc = np.concatenate([acc * float(alpha), p.astype(np.float64)])
        m = m_new
        offsets.append(float(m))
        ptiles.append(p)
    return acc, l, m, offsets, ptiles


def _rows(seed):
    """(name, tiles, scale) cases: scores of one row split into 128-key tiles."""
    rng = np.random.default_rng(seed)
    n = 6
    f = np.float32
    cases = [("gaussian", rng.standard_normal((n, TILE)).astype(f), f(0.088))]
    rising = rng.standard_normal((n, TILE)).astype(f) + (np.arange(n, dtype=f) * 40)[:, None]
    cases.append(("rising", rising, f(0.5)))
    # growth of about 8.7 (log2) per tile: just past the bound of 2^8
    slow = rng.standard_normal((n, TILE)).astype(f) + (np.arange(n, dtype=f) * 12)[:, None]
    cases.append(("rising_slow", slow, f(0.5)))
    peaky = rng.standard_normal((n, TILE)).astype(f)
    peaky[3, 17] = 300.0
    cases.append(("peaky", peaky, f(0.2)))
    masked = rng.standard_normal((n, TILE)).astype(f) * 4
    masked[:, rng.random(TILE) < 0.3] = -np.inf
    masked[-1, 40:] = -np.inf
    cases.append(("masked", masked, f(0.3)))
    prefix = rng.standard_normal((n, TILE)).astype(f) * 3
    prefix[:2] = -np.inf                      # the row's first tiles hold no kept key
    cases.append(("masked_prefix", prefix, f(0.25)))
    falling = rng.standard_normal((n, TILE)).astype(f) - (np.arange(n, dtype=f) * 30)[:, None]
    cases.append(("falling", falling, f(0.5)))
    return cases


def _check_row(tiles, scale, **kw):
    sl2 = np.float32(scale * LOG2E)
    acc, l, m, offsets, ptiles = run_row(tiles, sl2, "exps_first", **kw)
    ref_acc, ref_l, ref_m, ref_offsets, ref_p = run_row(tiles, sl2, "max_first")
    assert offsets == ref_offsets, f"offsets differ: {offsets} vs {ref_offsets}"
    for p, q in zip(ptiles, ref_p):
        np.testing.assert_array_equal(p, q)
    assert l == ref_l
    assert max(float(p.max()) for p in ptiles) <= 2.0 ** 8, "a term exceeds 2^8"
    # O / l and LSE against the exact softmax of the whole row
    z = tiles.reshape(-1).astype(np.float64) * float(scale)
    zmax = z.max()
    w = np.exp(z - zmax)
    np.testing.assert_allclose(acc / float(l), w / w.sum(), rtol=0, atol=2e-6)
    lse = (float(m) + np.log2(float(l))) * np.log(2.0)
    assert abs(lse - (zmax + np.log(w.sum()))) < 1e-4 * max(1.0, abs(lse))


@pytest.mark.parametrize("seed", range(6))
def test_exponentials_first_matches_max_first(seed):
    for name, tiles, scale in _rows(seed):
        _check_row(tiles, scale)


def test_rising_rows_do_move_the_offset():
    """The cases must exercise moves after the first tile, or the checks above say little."""
    moved = 0
    for seed in range(6):
        for name, tiles, scale in _rows(seed):
            sl2 = np.float32(scale * LOG2E)
            offs = run_row(tiles, sl2, "exps_first")[3]
            moved += sum(1 for a, b in zip(offs, offs[1:]) if a != b and a != -np.inf)
    assert moved >= 20


@pytest.mark.parametrize("mutant", ["loose_bound", "no_max_first_at_inf", "no_redo"])
def test_model_catches_planted_mistakes(mutant):
    kw = {"loose_bound": dict(bound=np.float32(65536.0)),
          "no_max_first_at_inf": dict(max_first_at_inf=False),
          "no_redo": dict(redo=False)}[mutant]
    caught = 0
    for seed in range(6):
        for name, tiles, scale in _rows(seed):
            try:
                _check_row(tiles, scale, **kw)
            except AssertionError:
                caught += 1
    assert caught > 0, f"{mutant} passed every row"
