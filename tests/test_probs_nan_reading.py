"""CPU pins of the reading that decides which draft data can flag a row.

Draft rows given as probabilities are used as given and read only where
the method reads them ("論文解説: Speculative Sampling", §技術的詳細 ステップ3
reads q_i(x_i) for every draft; §修正付き棄却サンプリング reads the whole row
q_j at a rejected position j to form max(0, p_j - q_j)).  A NaN elsewhere in
such a row is never read, so it cannot change the result and does not flag
the row.  Draft logit rows are different: q_i = softmax(l_i / T) is formed
over every entry of every row, so a NaN anywhere in them flags the row.
Greedy rows read no draft data at all.

Each case below differs from a clean case in one planted NaN; a checker
that flagged every NaN, or none, fails one of them.
"""

import numpy as np
from scipy import special

import oracle

B, G, V = 6, 3, 40


def _probs_case(seed=11):
    rng = np.random.default_rng(seed)
    tl = rng.normal(size=(B, G + 1, V))
    q = special.softmax(rng.normal(size=(B, G, V)), axis=-1)
    x = rng.integers(0, V, size=(B, G))
    u = rng.random((B, G + 1))
    T = np.full(B, 0.9)
    return tl, q, x, T, u


def _run(tl, q, probs, x, T, u):
    return oracle.verify_chain(tl, q, probs, x, T, u)


def test_probability_rows_flag_only_where_read():
    tl, q, x, T, u = _probs_case()
    u[0, :G] = 0.0                     # row 0 accepts every draft (bonus draw)
    u[1, 0] = 0.999999                 # row 1 rejects at 0 unless p/q > 1 there
    q[1, 0, x[1, 0]] = 0.9             # ... q(x_0) large: rejected at 0
    clean = _run(tl, q, True, x, T, u)
    assert clean["num_accepted"][0] == G and clean["num_accepted"][1] == 0
    assert not clean["status"].any()

    # row 0: NaN off the drafts in every draft row -> never read
    q0 = q.copy()
    for i in range(G):
        y = (x[0, i] + 1) % V
        q0[0, i, y] = np.nan
    r = _run(tl, q0, True, x, T, u)
    assert r["status"][0] == 0
    assert np.array_equal(r["tokens"][0], clean["tokens"][0])

    # row 0: NaN at q_i(x_i) of the last draft -> read by its accept test
    q1 = q.copy()
    q1[0, G - 1, x[0, G - 1]] = np.nan
    assert _run(tl, q1, True, x, T, u)["status"][0] == oracle.ROW_NONFINITE

    # row 1 (rejected at 0): NaN anywhere in row 0 -> read by the residual
    q2 = q.copy()
    q2[1, 0, (x[1, 0] + 7) % V] = np.nan
    assert _run(tl, q2, True, x, T, u)["status"][1] == oracle.ROW_NONFINITE

    # row 1: NaN in a later row, off its draft -> never read
    q3 = q.copy()
    q3[1, 2, (x[1, 2] + 3) % V] = np.nan
    r = _run(tl, q3, True, x, T, u)
    assert r["status"][1] == 0 and np.array_equal(r["tokens"][1], clean["tokens"][1])

    # row 1: NaN at a later draft's own q(x_i) -> read by its accept test
    q4 = q.copy()
    q4[1, 2, x[1, 2]] = np.nan
    assert _run(tl, q4, True, x, T, u)["status"][1] == oracle.ROW_NONFINITE


def test_logit_rows_flag_anywhere():
    rng = np.random.default_rng(12)
    tl = rng.normal(size=(B, G + 1, V))
    dl = tl[:, :G] + rng.normal(size=(B, G, V))
    x = rng.integers(0, V, size=(B, G))
    u = rng.random((B, G + 1))
    u[0, :G] = 0.0
    T = np.full(B, 1.1)
    T[2] = 0.0                         # a greedy row
    clean = _run(tl, dl, False, x, T, u)
    assert not clean["status"].any()
    d = dl.copy()
    d[0, 1, (x[0, 1] + 5) % V] = np.nan   # off the draft: still part of softmax(l / T)
    d[2, :, :] = np.nan                   # greedy row: draft rows unused
    r = _run(tl, d, False, x, T, u)
    assert r["status"][0] == oracle.ROW_NONFINITE
    assert r["status"][2] == 0 and np.array_equal(r["tokens"][2], clean["tokens"][2])
