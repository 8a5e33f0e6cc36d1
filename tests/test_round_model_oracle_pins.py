"""Pins for the oracle's model of whole rounds (CPU only).

The round model of "論文解説: Speculative Sampling" (§期待される高速化): the
tokens a round commits and the wall-clock speedup estimate.  The pins check
the law of n_accepted by enumerating every accept pattern, the expectation
against the page's closed form, the acceptance probability against the
total-variation identity, the known-overlap input pairs and the oracle's own
accept test, and the speedup estimate against a cost-counting simulation of
the decoding process.
"""

import itertools

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_48_gb300 import workloads as W


def test_accepted_count_law_by_enumerating_accept_patterns():
    rng = np.random.default_rng(31)
    for g in range(1, 9):
        a = rng.uniform(0.05, 0.99, g)
        want = np.zeros(g + 1)
        for pattern in itertools.product([0, 1], repeat=g):
            pr = np.prod([a[i] if pattern[i] else 1 - a[i] for i in range(g)])
            n = pattern.index(0) if 0 in pattern else g     # stop at the first rejection
            want[n] += pr
        np.testing.assert_allclose(oracle.accepted_count_law(a), want, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("alpha", [0.05, 0.5, 0.65, 0.72, 0.85, 0.99])
def test_expected_tokens_matches_the_pages_closed_form(alpha):
    for g in range(1, 12):
        E = oracle.expected_tokens_per_round([alpha] * g)
        np.testing.assert_allclose(E, (1 - alpha ** (g + 1)) / (1 - alpha), rtol=1e-12)


def test_expected_tokens_limits():
    for g in range(1, 10):
        assert oracle.expected_tokens_per_round([1.0] * g) == g + 1    # every draft kept
        assert oracle.expected_tokens_per_round([0.0] * g) == 1        # replacement only


def test_acceptance_probability_is_one_minus_total_variation():
    rng = np.random.default_rng(32)
    for _ in range(50):
        V = int(rng.integers(2, 300))
        lp, lq = rng.normal(size=V) * 2, rng.normal(size=V) * 2
        T = float(rng.uniform(0.3, 2.0))
        p = np.exp(lp / T - (lp / T).max())
        p /= p.sum()
        q = np.exp(lq / T - (lq / T).max())
        q /= q.sum()
        tv = 0.5 * np.abs(p - q).sum()
        np.testing.assert_allclose(oracle.acceptance_probability(lp, lq, T), 1 - tv, rtol=1e-10,
                                   atol=1e-13)
    same = rng.normal(size=64)
    np.testing.assert_allclose(oracle.acceptance_probability(same, same, 0.7), 1.0, rtol=1e-14)


@pytest.mark.parametrize("alpha", [0.2, 0.6, 0.8, 0.97, 1.0])
def test_known_overlap_pairs(alpha):
    """The generator's pairs have the overlap they were built for."""
    pr = W.make_alpha_pair(40, 3000, alpha)
    a = oracle.acceptance_probability(pr.target_logits.double().numpy(),
                                      pr.draft_logits.double().numpy(), 1.0)
    assert abs(a - alpha) < 1e-6


def test_acceptance_probability_matches_the_accept_test():
    """Monte Carlo through the oracle's own chain verifier (gamma = 1): the
    fraction of accepted drafts converges to sum min(p, q)."""
    pr = W.make_alpha_pair(41, 16, 0.7, sigma=1.0)
    lp = pr.target_logits.double().numpy()
    lq = pr.draft_logits.double().numpy()
    n = 40000
    rng = np.random.default_rng(33)
    q = np.exp(lq - lq.max())
    q /= q.sum()
    drafts = rng.choice(16, size=(n, 1), p=q)
    target = np.broadcast_to(lp, (n, 2, 16))
    draft = np.broadcast_to(lq, (n, 1, 16))
    r = oracle.verify_chain(target, draft, False, drafts, np.ones(n), rng.random((n, 2)))
    rate = r["num_accepted"].mean()
    a = oracle.acceptance_probability(lp, lq)
    assert abs(rate - a) < 5 * np.sqrt(a * (1 - a) / n)


def test_speedup_estimate_matches_a_cost_counting_simulation():
    """Decode 2e6 tokens with Bernoulli(alpha) accepts, charging gamma * c for
    each round's drafts and 1 for its target pass; plain decoding costs 1 per
    token.  The measured speedup converges to E / (1 + gamma c)."""
    rng = np.random.default_rng(34)
    for alpha, g, c in [(0.8, 4, 0.05), (0.65, 7, 0.1), (0.9, 2, 0.3)]:
        rounds = 400000
        accepts = rng.random((rounds, g)) < alpha
        n = np.where(accepts.all(axis=1), g, np.argmin(accepts, axis=1))
        tokens = (n + 1).sum()
        cost = rounds * (g * c + 1.0)
        measured = tokens / cost
        est = oracle.speedup_estimate(oracle.expected_tokens_per_round([alpha] * g), g, c)
        assert abs(measured - est) < 0.01 * est
