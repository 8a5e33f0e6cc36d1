"""Pins for the float64 oracle: closed forms, distribution theorems, brute force
and the pages' worked examples.  CPU only.

Each test is chosen so that a plausible slip in the oracle (a dropped
temperature, a wrong residual sign, an off-by-one row, a wrong tie rule, a
wrong walk) fails it.  Reference distributions come from
``scipy.special.softmax`` (a library routine, not the oracle's own code).
"""

import json
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sample(rng, probs, n):
    """n i.i.d. draws from each row of probs [P, V] -> [n, P] (library sampler)."""
    out = np.empty((n, probs.shape[0]), np.int64)
    for i, p in enumerate(probs):
        out[:, i] = rng.choice(len(p), size=n, p=p / p.sum())
    return out


def _run_rounds(tl, dl, probs_mode, T, rounds, seed, chunk=200_000):
    """Run the oracle on `rounds` i.i.d. rounds with fixed per-position rows."""
    rng = np.random.default_rng(seed)
    g1, V = tl.shape
    g = g1 - 1
    q = dl if probs_mode else special.softmax(dl / T, axis=-1)
    toks, nacc = [], []
    done = 0
    while done < rounds:
        n = min(chunk, rounds - done)
        x = _sample(rng, q, n)
        u = rng.random((n, g1))
        r = oracle.verify_chain(np.broadcast_to(tl, (n, g1, V)),
                                np.broadcast_to(dl, (n, g, V)), probs_mode, x,
                                np.full(n, T), u)
        assert not r["status"].any()
        toks.append(r["tokens"])
        nacc.append(r["num_accepted"])
        done += n
    return np.concatenate(toks), np.concatenate(nacc)


# ---------------------------------------------------------------------------
# Building blocks
# ---------------------------------------------------------------------------

def test_inverse_cdf_matches_interval_definition():
    """k is the unique index with C(k-1) <= u R < C(k) (brute force)."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        V = int(rng.integers(1, 12))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[rng.integers(V)] = 1.0
        u = rng.random()
        k, _, _ = oracle.inverse_cdf(w[None], np.array([u]))
        R = sum(w)
        lo = 0.0
        want = None
        for x in range(V):
            hi = lo + w[x]
            if lo <= u * R < hi:
                want = x
                break
            lo = hi
        assert want is not None and int(k[0]) == want


def test_inverse_cdf_uniform_weights_is_floor():
    V = 1000
    u = np.random.default_rng(1).random(5000) * 0.999
    k, _, _ = oracle.inverse_cdf(np.ones((u.size, V)), u)
    assert np.array_equal(k, np.floor(u * V).astype(np.int64))


def test_first_argmax_tie_rules():
    rng = np.random.default_rng(2)
    for _ in range(500):
        V = int(rng.integers(1, 20))
        row = rng.integers(-3, 3, size=V).astype(np.float64)
        if rng.random() < 0.3:
            row[row == 0] = -0.0
        best = 0
        for i in range(1, V):            # brute force: strictly larger wins
            if row[i] > row[best]:
                best = i
        assert int(oracle.first_argmax(row)) == best
    assert int(oracle.first_argmax(np.array([-0.0, 0.0, -1.0]))) == 0
    assert int(oracle.first_argmax(np.array([-np.inf, -np.inf]))) == 0


def test_tempered_softmax_matches_library():
    rng = np.random.default_rng(3)
    l = rng.normal(size=(6, 50)) * 3
    for T in (0.05, 0.7, 1.0, 2.5):
        np.testing.assert_allclose(oracle.tempered_softmax(l, np.full(6, T)),
                                   special.softmax(l / T, axis=-1), rtol=1e-12, atol=1e-300)


def test_residual_invariants():
    """norm(max(0, p - q)) sums to 1, is 0 where q >= p and > 0 where p > q."""
    rng = np.random.default_rng(4)
    for _ in range(50):
        V = int(rng.integers(2, 64))
        p = special.softmax(rng.normal(size=V) * 2)
        q = special.softmax(rng.normal(size=V) * 2)
        r = oracle.residual_distribution(p, q)
        assert abs(r.sum() - 1) < 1e-12
        assert np.all(r[q >= p] == 0)
        assert np.all(r[p > q] > 0)
        # total variation identity: sum max(0, p-q) = 1 - sum min(p, q) = TV
        tv = 0.5 * np.abs(p - q).sum()
        np.testing.assert_allclose(np.maximum(0, p - q).sum(), tv, rtol=1e-12)


# ---------------------------------------------------------------------------
# Accept test: acceptance probability = sum min(p, q) = 1 - TV(p, q)
# ---------------------------------------------------------------------------

def test_acceptance_probability_exact_over_drafts():
    """E_{x~q}[min(1, p(x)/q(x))] from the oracle's per-draft acceptance
    probabilities equals sum_x min(p, q) = 1 - TV(p, q) to 1e-12."""
    rng = np.random.default_rng(6)
    V, T = 16, 0.8
    tl = rng.normal(size=(2, V)) * 2
    dl = tl[:1] + rng.normal(size=(1, V))
    p = special.softmax(tl[0] / T)
    q = special.softmax(dl[0] / T)
    x = np.arange(V)[:, None]
    r = oracle.verify_chain(np.broadcast_to(tl, (V, 2, V)), np.broadcast_to(dl, (V, 1, V)),
                            False, x, np.full(V, T), np.zeros((V, 2)))
    acc = r["diag"][:, 0, 2]
    np.testing.assert_allclose(r["diag"][:, 0, 0], p, rtol=1e-12)
    np.testing.assert_allclose(r["diag"][:, 0, 1], q, rtol=1e-12)
    want = np.minimum(p, q).sum()
    assert abs((q * acc).sum() - want) < 1e-12
    assert abs(want - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12


def test_acceptance_rate_monte_carlo():
    """Empirical acceptance of draft 1 over 10^6 rounds ~ sum min(p, q)."""
    rng = np.random.default_rng(7)
    V, T = 8, 0.7
    tl = rng.normal(size=(2, V)) * 2
    dl = tl[:1] + rng.normal(size=(1, V)) * 1.5
    p = special.softmax(tl[0] / T)
    q = special.softmax(dl[0] / T)
    alpha = np.minimum(p, q).sum()
    _, nacc = _run_rounds(tl, dl, False, T, 1_000_000, seed=8)
    n = nacc.size
    sd = np.sqrt(alpha * (1 - alpha) / n)
    assert abs(nacc.mean() - alpha) < 5 * sd


# ---------------------------------------------------------------------------
# Theorem 1: emitted tokens are distributed as p, slot by slot
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("probs_mode", [False, True])
def test_theorem1_chi_square(probs_mode):
    rng = np.random.default_rng(9 + probs_mode)
    V, g, T = 8, 3, 0.9
    tl = rng.normal(size=(g + 1, V)) * 1.5
    dl = tl[:g] + rng.normal(size=(g, V)) * 1.2
    if probs_mode:
        dl = special.softmax(dl, axis=-1)        # q given as probabilities
    rounds = 1_000_000 if not probs_mode else 400_000
    toks, nacc = _run_rounds(tl, dl, probs_mode, T, rounds, seed=11 + probs_mode)
    for i in range(g + 1):
        p_i = special.softmax(tl[i] / T)
        reached = nacc >= i
        obs = np.bincount(toks[reached, i], minlength=V)
        exp = p_i * reached.sum()
        pval = stats.chisquare(obs, exp).pvalue
        assert pval > 1e-3, (i, pval, obs, exp)


def test_rejected_slot_follows_residual():
    """Given a rejection at draft 1, the corrected token ~ norm(max(0, p - q))."""
    rng = np.random.default_rng(12)
    V, T = 8, 1.0
    tl = rng.normal(size=(2, V)) * 2
    dl = tl[:1] + rng.normal(size=(1, V)) * 2
    toks, nacc = _run_rounds(tl, dl, False, T, 600_000, seed=13)
    p = special.softmax(tl[0] / T)
    q = special.softmax(dl[0] / T)
    res = np.maximum(0, p - q)
    res /= res.sum()
    rej = nacc == 0
    obs = np.bincount(toks[rej, 0], minlength=V)
    keep = res > 0
    assert np.all(obs[~keep] == 0)
    assert stats.chisquare(obs[keep], res[keep] * rej.sum()).pvalue > 1e-3


# ---------------------------------------------------------------------------
# Tokens per round at constant acceptance alpha: (1 - a^(g+1)) / (1 - a)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("alpha", [0.6, 0.85])
def test_expected_tokens_per_round(alpha):
    """q = alpha p + (1 - alpha) s with s supported where p = 0 gives
    sum min(p, q) = alpha at every position (the constant-alpha setting of
    [SpS] §期待される高速化)."""
    rng = np.random.default_rng(int(alpha * 100))
    V, g, T = 8, 4, 1.0
    tl = np.full((g + 1, V), -np.inf)
    tl[:, :4] = rng.normal(size=(g + 1, 4))
    q = np.zeros((g, V))
    for i in range(g):
        p_i = special.softmax(tl[i])
        s = np.zeros(V)
        s[4:] = rng.random(4) + 0.1
        s /= s.sum()
        q[i] = alpha * p_i + (1 - alpha) * s
    toks, nacc = _run_rounds(tl, q, True, T, 1_000_000, seed=21)
    emitted = nacc + 1
    want = (1 - alpha ** (g + 1)) / (1 - alpha)
    assert abs(emitted.mean() - want) < 4 * emitted.std() / np.sqrt(emitted.size)
    # full law: P(n = k) = alpha^k (1 - alpha) for k < g, alpha^g for k = g
    law = np.array([alpha ** k * (1 - alpha) for k in range(g)] + [alpha ** g])
    obs = np.bincount(nacc, minlength=g + 1)
    assert stats.chisquare(obs, law * nacc.size).pvalue > 1e-3


# ---------------------------------------------------------------------------
# The pages' worked examples
# ---------------------------------------------------------------------------

def test_sps_sequence_diagram_golden():
    g = json.load(open(os.path.join(GOLDEN, "sps_sequence_diagram.json")))
    gamma, V = g["gamma"], 8
    rng = np.random.default_rng(31)
    tl = rng.normal(size=(1, gamma + 1, V))
    dl = rng.normal(size=(1, gamma, V))
    x = np.array([[1, 2, 3, 4]])
    # drafts 1, 2 pass for any u = 0 with p > 0; draft 3 has p/q < 1 and
    # u = 0.999 so it fails.
    dl[0, 2, 3] = tl[0, 2, 3] + 3.0
    u = np.array([[0.0, 0.0, 0.999, 0.5, 0.25]])
    r = oracle.verify_chain(tl, dl, False, x, np.array([1.0]), u)
    n = int(r["num_accepted"][0])
    assert n == g["accepted"]
    committed = [t for t in r["tokens"][0] if t >= 0]
    assert len(committed) == g["tokens_committed"]
    assert committed[:2] == [1, 2]
    assert committed[2] != 3          # the residual is 0 where q >= p
    assert r["diag"][0, 2, 3] > 0     # residual mass recorded at the rejection


def test_sd_intro_greedy_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "sd_intro_greedy_example.json")))
    words = sorted(set(g["draft"]) | set(g["target_choice"]))
    vocab = {w: i for i, w in enumerate(words)}
    V = 8
    gamma = len(g["draft"])
    rng = np.random.default_rng(41)
    tl = rng.normal(size=(1, gamma + 1, V))
    for i, w in enumerate(g["target_choice"]):
        tl[0, i, vocab[w]] = tl[0, i].max() + 1.0
    x = np.array([[vocab[w] for w in g["draft"]]])
    r = oracle.verify_chain_greedy(tl, x)
    inv = {i: w for w, i in vocab.items()}
    committed = [inv[int(t)] for t in r["tokens"][0] if t >= 0]
    assert committed == g["committed"]
    assert int(r["num_accepted"][0]) == g["accepted"]
    for w in g["discarded"]:
        assert vocab[w] not in r["tokens"][0][: len(committed)]
    # same through the stochastic entry with T = 0
    r2 = oracle.verify_chain(tl, np.zeros((1, gamma, V)), False, x, np.array([0.0]),
                             np.zeros((1, gamma + 1)))
    assert np.array_equal(r2["tokens"], r["tokens"])


# ---------------------------------------------------------------------------
# Token tree: walk == deepest node whose whole root path matches (brute force)
# ---------------------------------------------------------------------------

def _random_tree(rng, N, V):
    par = [-1]
    for n in range(1, N):
        par.append(int(rng.integers(0, n)))
    par = np.array(par)
    tok = np.zeros(N, np.int64)
    tok[0] = rng.integers(V)
    for n in range(N):
        ch = np.flatnonzero(par == n)
        if ch.size > V:
            return None, None
        if ch.size:
            tok[ch] = rng.choice(V, size=ch.size, replace=False)   # distinct siblings
    return par, tok


def _brute_force_tree(logits, par, tok, D):
    N = len(par)
    a = [max(range(logits.shape[1]), key=lambda x: (logits[n, x], -x)) for n in range(N)]
    best, best_depth = 0, 0
    for n in range(1, N):
        chain = []
        c = n
        while c != 0:
            chain.append(c)
            c = par[c]
        chain.reverse()
        ok = all(tok[c] == a[par[c]] for c in chain)
        if ok and len(chain) <= D and len(chain) > best_depth:
            best, best_depth = n, len(chain)
    path = []
    c = best
    while c != 0:
        path.append(c)
        c = par[c]
    path.reverse()
    return path, [int(tok[c]) for c in path] + [a[best]]


def test_tree_walk_matches_brute_force():
    rng = np.random.default_rng(51)
    n_cases = 0
    for _ in range(400):
        N = int(rng.integers(2, 13))
        V = int(rng.integers(2, 6))
        par, tok = _random_tree(rng, N, V)
        if par is None:
            continue
        logits = rng.integers(-2, 3, size=(N, V)).astype(np.float64)
        D = int(rng.integers(1, 9))
        r = oracle.verify_tree_greedy(logits[None], par[None], tok[None], D)
        path, toks = _brute_force_tree(logits, par, tok, D)
        d = int(r["num_accepted"][0])
        assert d == len(path)
        assert list(r["path"][0, :d]) == path and np.all(r["path"][0, d:] == -1)
        assert list(r["tokens"][0, :d + 1]) == toks and np.all(r["tokens"][0, d + 1:] == -1)
        n_cases += 1
    assert n_cases > 300


def test_tree_validation():
    logits = np.zeros((1, 3, 4))
    ok_par = np.array([[-1, 0, 1]])
    tok = np.array([[0, 0, 0]])
    assert oracle.verify_tree_greedy(logits, ok_par, tok, 4)["status"][0] == 0
    for bad in ([0, 0, 1], [-1, 1, 1], [-1, 0, 3], [-1, -1, 0]):
        r = oracle.verify_tree_greedy(logits, np.array([bad]), tok, 4)
        assert r["status"][0] & oracle.ROW_BAD_TREE
        assert r["num_accepted"][0] == 0 and np.all(r["tokens"][0] == -1)
    r = oracle.verify_tree_greedy(logits, ok_par, np.array([[0, 4, 0]]), 4)
    assert r["status"][0] & oracle.ROW_BAD_TOKEN


# ---------------------------------------------------------------------------
# Degenerate cases of the chain
# ---------------------------------------------------------------------------

def test_zero_probability_conventions():
    """q(x) = 0 < p(x): accept; p(x) = q(x) = 0: reject; residual mass 0 at a
    rejection falls back to p_j."""
    V = 4
    tl = np.array([[[0.0, 1.0, -np.inf, 0.5], [0.0, 0.0, 0.0, 0.0]]])
    dl = np.array([[[0.0, 1.0, -np.inf, -np.inf]]])
    r = oracle.verify_chain(tl, dl, False, np.array([[3]]), np.array([1.0]),
                            np.array([[0.999, 0.3]]))
    assert r["num_accepted"][0] == 1          # q(3) = 0 < p(3): accepted
    # identical rows and a draft with p = q = 0: rejected, R = 0 -> draw from p_0
    dl2 = tl[:, :1].copy()
    r = oracle.verify_chain(tl, dl2, False, np.array([[2]]), np.array([1.0]),
                            np.array([[0.0, 0.3]]))
    assert r["num_accepted"][0] == 0
    p0 = special.softmax(tl[0, 0])
    k = int(np.searchsorted(np.cumsum(p0), 0.3 * p0.sum(), side="right"))
    assert r["tokens"][0, 0] == k and r["diag"][0, 0, 3] == 0


def test_data_errors_flag_rows():
    rng = np.random.default_rng(61)
    B, g, V = 5, 2, 6
    tl = rng.normal(size=(B, g + 1, V))
    dl = rng.normal(size=(B, g, V))
    x = rng.integers(0, V, size=(B, g))
    T = np.array([1.0, 1.0, 0.0, np.nan, 1e-30])
    x[0, 1] = V                       # token out of range
    tl[1, 2, 3] = np.nan              # NaN in a row that is read
    tl[2, 0, 0] = np.nan              # NaN in a greedy row
    u = rng.random((B, g + 1))
    r = oracle.verify_chain(tl, dl, False, x, T, u)
    assert r["status"][0] & oracle.ROW_BAD_TOKEN
    assert r["status"][1] & oracle.ROW_NONFINITE
    assert r["status"][2] & oracle.ROW_NONFINITE
    assert r["status"][3] & oracle.ROW_BAD_TEMPERATURE
    assert r["status"][4] & oracle.ROW_BAD_TEMPERATURE
    assert np.all(r["tokens"] == -1) and np.all(r["num_accepted"] == 0)


def test_greedy_rows_ignore_draft_logits_and_uniforms():
    rng = np.random.default_rng(71)
    B, g, V = 6, 3, 9
    tl = rng.integers(-2, 2, size=(B, g + 1, V)).astype(np.float64)
    x = rng.integers(0, V, size=(B, g))
    a = [[max(range(V), key=lambda v: (tl[b, i, v], -v)) for i in range(g + 1)] for b in range(B)]
    x[0] = a[0][:g]                                   # all accepted -> bonus a_g
    r1 = oracle.verify_chain(tl, rng.normal(size=(B, g, V)), False, x, np.zeros(B),
                             rng.random((B, g + 1)))
    r2 = oracle.verify_chain(tl, rng.normal(size=(B, g, V)), False, x, -np.ones(B),
                             rng.random((B, g + 1)))
    assert np.array_equal(r1["tokens"], r2["tokens"])
    assert r1["num_accepted"][0] == g and r1["tokens"][0, g] == a[0][g]
    for b in range(B):
        j = next((i for i in range(g) if x[b, i] != a[b][i]), g)
        assert r1["num_accepted"][b] == j
        assert list(r1["tokens"][b, :j + 1]) == list(x[b, :j]) + [a[b][j]]
