"""Comparison of library outputs with the float64 oracle (test infrastructure).

Greedy and tree outputs must be bit-exact.  A stochastic row may differ
only where the one floating-point decision that separates the two results
lies within ``eps`` (1e-5) of its boundary:

  * the accept test at the first position where the two sides disagree
    (one accepted, the other rejected), i = min(j_lib, j_oracle) < gamma,
    with |u_i - p_i(x_i)/q_i(x_i)| < eps (the oracle's float64 ratio); the
    draft tokens before i must agree;
  * with the same first rejection j on both sides, the categorical draw at
    slot j: the library's token k' must be the oracle's choice for some
    uniform within eps of u_gamma, i.e. dist(u, [C(k'-1)/R, C(k')/R)) < eps
    on the oracle's CDF; the drafts before j and the -1 padding after j
    must agree.

Such rows are counted as boundary cases and reported; any other difference
is a failure.  Diagnostic probabilities are compared within ``prob_tol``
(1e-4 for bf16/fp16 logits, 1e-5 for fp32), the residual mass of a rejected
row only where both sides rejected at the same position.  Greedy rows carry
zero diagnostics on both sides.
"""

from __future__ import annotations

import numpy as np

from .spec_verify_oracle import verify_chain

EPS = 1e-5


def prob_tolerance(dtype_name: str) -> float:
    return 1e-5 if dtype_name in ("f32", "float32") else 1e-4


def _cdf_distance(args64, b, k, uu):
    """Distance of the uniform ``uu`` from the oracle's CDF interval of token
    ``k`` in the distribution row ``b`` drew its last token from."""
    tl, dr, probs, xt, T, u = args64
    one = verify_chain(tl[b:b + 1], dr[b:b + 1], probs, xt[b:b + 1], T[b:b + 1],
                       u[b:b + 1], keep_cdf=True)
    cdf = one["cdf"][0]
    if not 0 <= k < cdf.size:
        return np.inf
    lo = 0.0 if k == 0 else cdf[k - 1]
    hi = cdf[k]
    if np.isnan(lo) or np.isnan(hi):
        return np.inf
    return 0.0 if lo <= uu < hi else min(abs(uu - lo), abs(uu - hi))


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
        jg, jr = int(nacc[b]), int(ref["num_accepted"][b])
        same = jg == jr and np.array_equal(tokens[b], ref["tokens"][b])
        if diag is not None:
            d = np.asarray(diag[b], np.float64)
            cols = 4 if jg == jr else 3
            err = float(np.max(np.abs(d[:, :cols] - ref["diag"][b, :, :cols]), initial=0.0))
            if np.isnan(d[:, :cols]).any():
                err = np.inf
            diag_err = max(diag_err, err)
            if err > prob_tol:
                failures.append((b, "diag", err))
                continue
        if same:
            exact += 1
            continue
        if ref["greedy"][b]:
            failures.append((b, "greedy mismatch", tokens[b].tolist(), ref["tokens"][b].tolist()))
            continue
        if not (0 <= jg <= g):
            failures.append((b, "num_accepted out of range", jg))
            continue
        if jg != jr:
            # the first position whose accept decision differs
            i = min(jg, jr)
            if (np.array_equal(tokens[b, :i], ref["tokens"][b, :i])
                    and abs(u[b, i] - ref["ratio"][b, i]) < eps):
                boundary.append((b, "accept", i))
                continue
            failures.append((b, "first rejection", jg, jr, tokens[b].tolist(),
                             ref["tokens"][b].tolist()))
            continue
        j = jg
        if (not np.array_equal(tokens[b, :j], ref["tokens"][b, :j])
                or np.any(tokens[b, j + 1:] != -1)):
            failures.append((b, "accepted drafts or padding", tokens[b].tolist(),
                             ref["tokens"][b].tolist()))
            continue
        k = int(tokens[b, j])
        dist = _cdf_distance(args64, b, k, u[b, g])
        if dist < eps:
            boundary.append((b, "sample", k, int(ref["tokens"][b, j]), float(dist)))
            continue
        failures.append((b, "draw", k, int(ref["tokens"][b, j]), float(dist)))
    return dict(rows=B, exact=exact, boundary=boundary, failures=failures,
                diag_max_err=diag_err)


def compare_exact(names_and_pairs):
    """[(name, got, want)] -> list of names whose arrays differ."""
    return [n for n, got, want in names_and_pairs
            if not np.array_equal(np.asarray(got), np.asarray(want))]
