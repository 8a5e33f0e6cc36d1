"""Pins for the oracle's draft-side sampler (CPU only).

The draft step draws each draft token from softmax(draft logits / T)
("論文解説: Speculative Sampling", §アルゴリズム Step 1 and the listing's drafting
loop).  The pins check the oracle against a library softmax, the interval
definition of the inverse CDF, brute-force argmax and a chi-square test, so
that a dropped temperature, an off-by-one in the CDF or a wrong tie rule fails.
"""

import numpy as np
from scipy import special, stats

import oracle


def test_draft_sample_follows_the_tempered_softmax():
    """Theorem-style pin: over many uniforms, tokens are distributed as
    softmax(l / T) (chi-square against scipy's softmax)."""
    rng = np.random.default_rng(21)
    V = 8
    l = rng.normal(size=V) * 2.0
    for T in (0.6, 1.0, 1.7):
        n = 60000
        u = rng.random(n)
        r = oracle.draft_sample(np.broadcast_to(l, (n, V)), np.full(n, T), u)
        assert not r["status"].any()
        obs = np.bincount(r["tokens"], minlength=V)
        exp = special.softmax(l / T) * n
        assert stats.chisquare(obs, exp).pvalue > 1e-3


def test_draft_sample_matches_the_interval_definition():
    """Brute force: the token k is the one with C(k-1) <= u R < C(k) over the
    library softmax, and the returned probability is that softmax value."""
    rng = np.random.default_rng(22)
    for _ in range(300):
        V = int(rng.integers(1, 12))
        l = rng.normal(size=V) * 3
        l[rng.random(V) < 0.2] = -np.inf
        if np.all(np.isinf(l)):
            l[0] = 0.0
        T = float(rng.uniform(0.2, 2.0))
        u = float(rng.random())
        r = oracle.draft_sample(l[None], np.array([T]), np.array([u]))
        p = special.softmax(l / T)
        acc, want = 0.0, None
        for x in range(V):
            if acc <= u < acc + p[x]:
                want = x
                break
            acc += p[x]
        if want is None:                      # rounding at the top end
            want = int(np.flatnonzero(p > 0)[-1])
        assert int(r["tokens"][0]) == want
        np.testing.assert_allclose(r["probs"][0], p[want], rtol=1e-12)
        assert r["cdf_lo"][0] <= u < r["cdf_hi"][0] + 1e-12


def test_draft_sample_greedy_rows_take_the_first_argmax():
    rng = np.random.default_rng(23)
    l = rng.integers(-3, 3, size=(200, 9)).astype(np.float64)
    r = oracle.draft_sample(l, np.zeros(200), rng.random(200))
    for b in range(200):
        best = 0
        for i in range(1, 9):
            if l[b, i] > l[b, best]:
                best = i
        assert int(r["tokens"][b]) == best
    assert np.all(r["probs"] == 0) and not r["status"].any()


def test_draft_sample_flags_bad_rows():
    l = np.zeros((5, 4))
    l[1, 2] = np.nan
    l[2, :] = -np.inf
    T = np.array([np.nan, 1.0, 1.0, 1e-30, 0.0])
    l[4, 1] = np.nan
    r = oracle.draft_sample(l, T, np.full(5, 0.5))
    assert list(r["status"]) == [oracle.ROW_BAD_TEMPERATURE, oracle.ROW_NONFINITE,
                                 oracle.ROW_NONFINITE, oracle.ROW_BAD_TEMPERATURE,
                                 oracle.ROW_NONFINITE]
    assert np.all(r["tokens"] == -1)
