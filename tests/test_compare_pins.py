"""CPU pins of the parity checker (``oracle/compare.py``).

The checker excuses a stochastic row only where the single floating-point
decision that separates the library's result from the oracle's lies within
1e-5 of its boundary (the accept test u_i * q_i(x_i) < p_i(x_i) of
"論文解説: Speculative Sampling" §技術的詳細 ステップ3, or the inverse-CDF
draw of §修正付き棄却サンプリング).  These tests plant mistakes in copies of
the oracle's own outputs — a wrong accepted token, a first rejection off by
one, a wrong residual draw, garbage after the drawn token, a wrong status, a
diagnostic off by twice the tolerance, a greedy mismatch — and check that
each is reported as a failure, while genuine boundary cases built on
purpose (a uniform within 1e-7 of an acceptance ratio or of a CDF boundary)
are the only rows excused.
"""

import numpy as np
import pytest

import oracle
from oracle.compare import EPS, compare_chain
from speculative_decoding_verification_48_gb300 import workloads as W

B, G, V = 48, 4, 64


def _temps(b, v):
    return 0.0 if b % 6 == 0 else 0.4 + v


@pytest.fixture(scope="module")
def base():
    case = W.make_chain("cmp", 777, B=B, gamma=G, V=V, dtype="f32", target="normal",
                        target_sigma=1.5, draft_sigma=(0.3, 1.5), temperature=_temps)
    return case.numpy64()


def _outputs(ref):
    return (ref["tokens"].copy(), ref["num_accepted"].copy(), ref["status"].copy(),
            ref["diag"].astype(np.float32).copy())


def _check(args, ref, toks, nacc, st, diag):
    return compare_chain(args, ref, toks, nacc, st, diag, prob_tol=1e-4)


def _failed_rows(cmp):
    return {f[0] for f in cmp["failures"]}


def _stoch_rows(ref, cond):
    return [b for b in range(B) if not ref["greedy"][b] and ref["status"][b] == 0 and cond(b)]


def _far(u, r):
    return abs(u - r) > 1e-3


def test_identical_outputs_are_exact(base):
    ref = oracle.verify_chain(*base)
    cmp = _check(base, ref, *_outputs(ref))
    assert cmp["failures"] == [] and cmp["boundary"] == [] and cmp["exact"] == B


def test_wrong_accepted_token_fails(base):
    ref = oracle.verify_chain(*base)
    rows = _stoch_rows(ref, lambda b: ref["num_accepted"][b] >= 1)
    assert rows
    b = rows[0]
    toks, nacc, st, diag = _outputs(ref)
    toks[b, 0] = (toks[b, 0] + 1) % V
    cmp = _check(base, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b} and cmp["boundary"] == []


@pytest.mark.parametrize("shift", [1, -1])
def test_first_rejection_off_by_one_fails(base, shift):
    ref = oracle.verify_chain(*base)
    u = base[5]
    if shift > 0:
        # the library claims one more accepted draft than the oracle
        rows = _stoch_rows(ref, lambda b: ref["num_accepted"][b] < G
                           and _far(u[b, ref["num_accepted"][b]], ref["ratio"][b, ref["num_accepted"][b]]))
    else:
        rows = _stoch_rows(ref, lambda b: ref["num_accepted"][b] >= 1
                           and _far(u[b, ref["num_accepted"][b] - 1],
                                    ref["ratio"][b, ref["num_accepted"][b] - 1]))
    assert rows
    b = rows[0]
    j = int(ref["num_accepted"][b]) + shift
    toks, nacc, st, diag = _outputs(ref)
    xt = base[3]
    toks[b] = -1
    toks[b, :j] = xt[b, :j]
    toks[b, j] = ref["tokens"][b, ref["num_accepted"][b]]
    nacc[b] = j
    cmp = _check(base, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b} and cmp["boundary"] == []


def test_wrong_draw_fails(base):
    ref = oracle.verify_chain(*base)
    rows = _stoch_rows(ref, lambda b: True)
    toks, nacc, st, diag = _outputs(ref)
    b = rows[0]
    j = int(ref["num_accepted"][b])
    one = oracle.verify_chain(*(a[b:b + 1] if isinstance(a, np.ndarray) else a for a in base),
                              keep_cdf=True)
    cdf = one["cdf"][0]
    uu = base[5][b, G]
    # a token whose CDF interval is at least 1e-3 away from u
    lo = np.concatenate([[0.0], cdf[:-1]])
    far = [k for k in range(V) if min(abs(uu - lo[k]), abs(uu - cdf[k])) > 1e-3
           and not lo[k] <= uu < cdf[k]]
    toks[b, j] = far[0]
    cmp = _check(base, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b} and cmp["boundary"] == []


def test_padding_after_draw_fails(base):
    ref = oracle.verify_chain(*base)
    rows = _stoch_rows(ref, lambda b: ref["num_accepted"][b] < G)
    b = rows[0]
    toks, nacc, st, diag = _outputs(ref)
    toks[b, int(ref["num_accepted"][b]) + 1] = 0
    cmp = _check(base, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b}


def test_status_and_error_rows(base):
    ref = oracle.verify_chain(*base)
    toks, nacc, st, diag = _outputs(ref)
    st[3] = 2                                   # a flag the oracle does not raise
    cmp = _check(base, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {3}
    # an error row must be cleared: tokens -1 and no accepted draft
    args = list(base)
    xt = args[3].copy()
    xt[5, 1] = V                                # out of range -> BAD_TOKEN
    args[3] = xt
    ref2 = oracle.verify_chain(*args)
    assert ref2["status"][5] == oracle.ROW_BAD_TOKEN
    toks, nacc, st, diag = _outputs(ref2)
    toks[5, 0] = 7
    cmp = _check(tuple(args), ref2, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {5}


def test_diag_beyond_tolerance_fails(base):
    ref = oracle.verify_chain(*base)
    rows = _stoch_rows(ref, lambda b: True)
    toks, nacc, st, diag = _outputs(ref)
    diag[rows[1], 0, 0] += 2e-4
    diag[rows[2], 1, 1] += 0.5e-4               # within tolerance
    cmp = _check(base, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {rows[1]}
    # greedy rows carry zero diagnostics
    g = [b for b in range(B) if ref["greedy"][b]][0]
    toks, nacc, st, diag = _outputs(ref)
    diag[g, 0, 0] = 0.3
    assert _failed_rows(_check(base, ref, toks, nacc, st, diag)) == {g}


def test_greedy_mismatch_fails_even_with_near_uniforms(base):
    args = list(base)
    ref0 = oracle.verify_chain(*args)
    g = [b for b in range(B) if ref0["greedy"][b] and ref0["num_accepted"][b] < G][0]
    u = args[5].copy()
    u[g, :] = 0.5                               # unused by greedy rows
    args[5] = u
    ref = oracle.verify_chain(*args)
    toks, nacc, st, diag = _outputs(ref)
    j = int(ref["num_accepted"][g])
    toks[g, j] = (toks[g, j] + 1) % V
    cmp = _check(tuple(args), ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {g} and cmp["boundary"] == []


def _with_accept_boundary(base):
    """A stochastic row rejected at j >= 1, whose uniform at j is moved to
    1e-7 below the ratio: the oracle now accepts j."""
    ref0 = oracle.verify_chain(*base)
    rows = _stoch_rows(ref0, lambda b: 1 <= ref0["num_accepted"][b] < G
                       and ref0["ratio"][b, ref0["num_accepted"][b]] < 0.9
                       and _far(base[5][b, 0], ref0["ratio"][b, 0]))
    b = rows[0]
    j0 = int(ref0["num_accepted"][b])
    args = list(base)
    u = args[5].copy()
    u[b, j0] = ref0["ratio"][b, j0] - 1e-7
    args[5] = u
    ref = oracle.verify_chain(*args)
    assert ref["num_accepted"][b] > j0
    return tuple(args), ref, b, j0


def test_genuine_accept_boundary_is_excused(base):
    args, ref, b, j0 = _with_accept_boundary(base)
    toks, nacc, st, diag = _outputs(ref)
    # the library took the other side of the boundary: rejected at j0
    toks[b] = -1
    toks[b, :j0] = args[3][b, :j0]
    toks[b, j0] = 0
    nacc[b] = j0
    cmp = _check(args, ref, toks, nacc, st, diag)
    assert cmp["failures"] == [] and [x[:3] for x in cmp["boundary"]] == [(b, "accept", j0)]


def test_boundary_elsewhere_does_not_excuse(base):
    args, ref, b, j0 = _with_accept_boundary(base)
    assert abs(args[5][b, j0] - ref["ratio"][b, j0]) < EPS
    toks, nacc, st, diag = _outputs(ref)
    # both sides accept j0 (near its boundary); the library's first
    # rejection is off elsewhere, at position 0, far from its boundary
    toks[b] = -1
    toks[b, 0] = 1
    nacc[b] = 0
    cmp = _check(args, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b} and cmp["boundary"] == []
    # same row: decisions agree, the draw is wrong and far from any boundary
    toks, nacc, st, diag = _outputs(ref)
    j = int(ref["num_accepted"][b])
    one = oracle.verify_chain(*(a[b:b + 1] if isinstance(a, np.ndarray) else a for a in args),
                              keep_cdf=True)
    cdf = one["cdf"][0]
    uu = args[5][b, G]
    lo = np.concatenate([[0.0], cdf[:-1]])
    far = [k for k in range(V) if min(abs(uu - lo[k]), abs(uu - cdf[k])) > 1e-3
           and not lo[k] <= uu < cdf[k]]
    toks[b, j] = far[0]
    cmp = _check(args, ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b} and cmp["boundary"] == []


def test_genuine_sample_boundary_is_excused(base):
    ref0 = oracle.verify_chain(*base)
    b = _stoch_rows(ref0, lambda b: True)[3]
    one = oracle.verify_chain(*(a[b:b + 1] if isinstance(a, np.ndarray) else a for a in base),
                              keep_cdf=True)
    cdf = one["cdf"][0]
    pos = [k for k in range(V - 1) if 0.05 < cdf[k] < 0.95 and cdf[k + 1] - cdf[k] > 1e-4]
    k = pos[len(pos) // 2]
    args = list(base)
    u = args[5].copy()
    u[b, G] = cdf[k] + 1e-7                     # just past token k's interval
    args[5] = u
    ref = oracle.verify_chain(*args)
    j = int(ref["num_accepted"][b])
    assert ref["tokens"][b, j] > k
    toks, nacc, st, diag = _outputs(ref)
    toks[b, j] = k                              # the other side of the boundary
    cmp = _check(tuple(args), ref, toks, nacc, st, diag)
    assert cmp["failures"] == [] and [x[:3] for x in cmp["boundary"]] == [(b, "sample", k)]
    toks[b, j] = max(0, k - 5) if cdf[max(0, k - 5)] < cdf[k] - 1e-3 else k + 6
    cmp = _check(tuple(args), ref, toks, nacc, st, diag)
    assert _failed_rows(cmp) == {b}
