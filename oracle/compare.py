"""Comparison of library outputs with the float64 oracle (test infrastructure).

Greedy and tree outputs must be bit-exact.  A stochastic row may differ
only where a floating-point decision is within ``eps`` (1e-5) of its
boundary:

  * an accept test at a position both sides reached, with
    |u_i - p_i(x_i)/q_i(x_i)| < eps (oracle's float64 ratio), or
  * the categorical draw at the same rejected/bonus position j, where the
    library's token k' would be the oracle's choice for a uniform within eps
    of u, i.e. dist(u, [C(k'-1)/R, C(k')/R)) < eps on the oracle's CDF.

Such rows are counted as boundary cases and reported; any other difference
is a failure.  Diagnostic probabilities are compared within ``prob_tol``
(1e-4 for bf16/fp16 logits, 1e-5 for fp32).
"""

from __future__ import annotations

import numpy as np

from .spec_verify_oracle import verify_chain

EPS = 1e-5


def prob_tolerance(dtype_name: str) -> float:
    return 1e-5 if dtype_name in ("f32", "float32") else 1e-4


def compare_chain(args64, ref, tokens, nacc, status, diag=None, prob_tol=1e-4, eps=EPS):
    """args64: the oracle's inputs (float64 numpy, as from ChainCase.numpy64());
    ref: oracle result dict; tokens/nacc/status/diag: library outputs (numpy).
    Returns dict(rows, exact, boundary, failures, diag_max_err)."""
    tl, dr, probs, xt, T, u = args64
    B, G1 = tokens.shape
    g = G1 - 1
    tokens = np.asarray(tokens, np.int64)
    nacc = np.asarray(nacc, np.int64)
    status = np.asarray(status, np.int64)
    failures, boundary = [], []
    exact = 0
    diag_err = 0.0
    for b in range(B):
        if status[b] != ref["status"][b]:
            failures.append((b, "status", int(status[b]), int(ref["status"][b])))
            continue
        if status[b]:
            if nacc[b] != 0 or np.any(tokens[b] != -1):
                failures.append((b, "error row not cleared"))
            else:
                exact += 1
            continue
        same = nacc[b] == ref["num_accepted"][b] and np.array_equal(tokens[b], ref["tokens"][b])
        if not ref["greedy"][b] and diag is not None:
            d = np.asarray(diag[b], np.float64)
            err = np.max(np.abs(d[:, :3] - ref["diag"][b, :, :3]))
            err = max(err, float(np.max(np.abs(d[:, 3] - ref["diag"][b, :, 3]))) if same else err)
            diag_err = max(diag_err, float(err))
            if err > prob_tol:
                failures.append((b, "diag", float(err)))
        if same:
            exact += 1
            continue
        if ref["greedy"][b]:
            failures.append((b, "greedy mismatch", tokens[b].tolist(), ref["tokens"][b].tolist()))
            continue
        jg, jr = int(nacc[b]), int(ref["num_accepted"][b])
        lim = min(jg, jr)
        near = [i for i in range(min(lim + 1, g))
                if abs(u[b, i] - ref["ratio"][b, i]) < eps]
        if near:
            boundary.append((b, "accept", near))
            continue
        if jg == jr and np.array_equal(tokens[b, :jg], ref["tokens"][b, :jr]):
            one = verify_chain(tl[b:b + 1], dr[b:b + 1], probs, xt[b:b + 1], T[b:b + 1],
                               u[b:b + 1], keep_cdf=True)
            cdf = one["cdf"][0]
            k = int(tokens[b, jg])
            if 0 <= k < cdf.size:
                lo = 0.0 if k == 0 else cdf[k - 1]
                hi = cdf[k]
                uu = u[b, g]
                dist = 0.0 if lo <= uu < hi else min(abs(uu - lo), abs(uu - hi))
                if dist < eps:
                    boundary.append((b, "sample", k, int(ref["tokens"][b, jr]), dist))
                    continue
        failures.append((b, "stochastic mismatch", tokens[b].tolist(),
                         ref["tokens"][b].tolist()))
    return dict(rows=B, exact=exact, boundary=boundary, failures=failures,
                diag_max_err=diag_err)


def compare_exact(names_and_pairs):
    """[(name, got, want)] -> list of names whose arrays differ."""
    return [n for n, got, want in names_and_pairs
            if not np.array_equal(np.asarray(got), np.asarray(want))]
