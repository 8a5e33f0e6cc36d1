"""The multi-round simulator on the GPU against the oracle's round model.

Every round runs the library's draft sampler and chain verifier. The
measured tokens per round, the law of n_accepted and the per-position
acceptance rates must match what the oracle predicts for the same stored
p / q pair. The oracle takes the pair's overlap from its own softmax of the
stored logits.
"""

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verification_48_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def sim():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as pkg
    pkg.lib()
    from speculative_decoding_verification_48_gb300 import simulate
    return simulate


def _oracle_alpha(seed, V, alpha):
    pr = W.make_alpha_pair(seed, V, alpha)
    return oracle.acceptance_probability(pr.target_logits.double().numpy(),
                                         pr.draft_logits.double().numpy(), 1.0)


@pytest.mark.parametrize("gamma,alpha", [(1, 0.6), (4, 0.8), (7, 0.72)])
def test_rounds_follow_the_round_model(sim, gamma, alpha):
    r = sim.simulate(gamma, alpha, sequences=2048, tokens=48, V=4096, seed=7, device=DEV)
    a = _oracle_alpha(7, 4096, alpha)
    law = oracle.accepted_count_law([a] * gamma)
    E = oracle.expected_tokens_per_round([a] * gamma)
    assert r.rounds > 10000
    assert abs(r.tokens_per_round - E) < 5 * r.tokens_per_round_se, (r.tokens_per_round, E)
    h = np.array(r.n_accepted_hist, dtype=np.float64)
    assert h.sum() == r.rounds
    assert stats.chisquare(h, law * h.sum()).pvalue > 1e-4
    reach = np.cumsum(h[::-1])[::-1]
    for i, ai in enumerate(r.accept_rate):
        se = np.sqrt(a * (1 - a) / reach[i])
        assert abs(ai - a) < 6 * se, (i, ai, a)
    np.testing.assert_allclose(r.speedup_model, r.tokens_per_round / (1 + gamma * r.c))
    assert r.us_per_round > 0
    assert r.tokens >= r.sequences * r.tokens_per_sequence


def test_identical_draft_and_target_accept_everything(sim):
    """alpha = 1 stores the same logits for p and q: u q(x) < p(x) holds
    for every u < 1, so each round commits gamma + 1 tokens."""
    r = sim.simulate(5, 1.0, sequences=256, tokens=30, V=1024, seed=3, device=DEV)
    assert r.n_accepted_hist == [0] * 5 + [r.rounds]
    assert r.tokens_per_round == 6.0
    assert r.rounds == 256 * 5                       # 30 tokens in 5 rounds of 6


def test_sweep_matches_the_model_across_gamma(sim):
    rs = sim.sweep(0.85, range(1, 9), sequences=1024, tokens=40, V=2048, seed=11, device=DEV)
    a = _oracle_alpha(11, 2048, 0.85)
    for r in rs:
        E = oracle.expected_tokens_per_round([a] * r.gamma)
        assert abs(r.tokens_per_round - E) < 5 * r.tokens_per_round_se, (r.gamma, E)
    best = max(rs, key=lambda r: r.speedup_model).gamma
    model = [oracle.speedup_estimate(oracle.expected_tokens_per_round([a] * g), g, 0.05)
             for g in range(1, 9)]
    assert abs(best - (int(np.argmax(model)) + 1)) <= 2
