"""Float64 CPU oracle for the verification step of speculative sampling.

TEST INFRASTRUCTURE.  Only the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` import this module.  The library
package (``speculative_decoding_verification_48_gb300``) never imports it, and
the two share no code: no kernels, helpers, tables or constants.  The only
module both sides use is the seeded input generator, which holds none of the
verification arithmetic.

Sources, cited by tag:

  [SpS]        "論文解説: Speculative Sampling — ドラフトモデルによるLLMデコード高速化"
               (0h-n0.github.io/posts/paper-2302-01318), an explainer of
               Chen et al., "Accelerating Large Language Model Decoding with
               Speculative Sampling", arXiv:2302.01318.
  [SD-intro]   "投機的デコーディングとは？LLMの回答を高速化する仕組み"
               (ai-compass.weeybrid.co.jp/algorizm/speculative-decoding/).
  [SpecInfer]  SpecInfer explainer (abeam.tech/media/ai-papers/2026-08-22-
               specinfer-token-tree-speculative-decoding/), on Miao et al.,
               arXiv:2305.09781.

Everything is computed in float64 from the stored (already rounded) bf16 /
fp16 / fp32 input values.  Where the pages leave a step open this module takes
the plainest reading, stated at the function that uses it:

  * Accept test: accept draft i iff  u_i * q_i(x_i) < p_i(x_i)  (strict; the
    same as ``u < min(1, p/q)`` for q > 0).  With q = 0 and p > 0 the draft is
    accepted; with p = q = 0 it is rejected.  No epsilon is added.
  * Rows are aligned by the caller: target row i scores draft i, target row
    gamma is the bonus row; draft row i is the distribution draft i was drawn
    from.
  * Bonus: when all gamma drafts are accepted, one extra token is drawn from
    p_gamma with the last uniform ("gamma+1 tokens per round" in [SpS]
    §期待される高速化).
  * The categorical draw is the inverse CDF in ascending vocabulary order:
    the smallest k with  sum_{x<=k} w(x) > u * R,  R = sum_x w(x).
  * If the residual at a rejected position has R == 0 (only reachable through
    rounding or p = q with a zero-probability draft), the token is drawn
    from p_j instead.
  * Temperature T <= 0 selects greedy verification for that row; greedy argmax
    takes the lowest index among equal maxima (-0 == +0).  T is applied to
    target and draft logits alike; draft rows given as probabilities are used
    as given (no temperature, no renormalisation).
  * Data errors make a row report a nonzero status, ``num_accepted = 0`` and
    all tokens -1: a draft / node token outside [0, V), a NaN (or +inf /
    all -inf) row in a softmax, a NaN in an argmax row, a malformed tree,
    or a temperature that is NaN or in (0, 1e-20).  Draft rows given as
    probabilities are checked only where they are read: q(x_i) for every
    draft, and the residual mass at a rejected position (NaN propagates).

Parity status: every function here is pinned by the CPU tests (closed forms,
distribution tests, brute force and the pages' worked examples).  The exact
token chosen for one uniform depends on the inverse-CDF reading above; that
sampler is pinned against its interval definition by brute force.
"""

from __future__ import annotations

import numpy as np

# Row-status bits.  These are plain numbers of this module; the library
# defines its own copy of the same contract in its public header.
ROW_OK = 0
ROW_BAD_TOKEN = 1
ROW_NONFINITE = 2
ROW_BAD_TREE = 4
ROW_TIMEOUT = 8          # device-side only; never produced here
ROW_BAD_TEMPERATURE = 16

TINY_T = 1e-20


# --------------------------------------------------------------------------
# Building blocks
# --------------------------------------------------------------------------

def tempered_softmax(logits: np.ndarray, T: np.ndarray) -> np.ndarray:
    """p(x) = exp(l(x)/T - max_y l(y)/T) / sum_z exp(l(z)/T - max_y l(y)/T).

    [SpS] §実装のポイント, the ``speculative_decode`` listing: both models'
    rows go through softmax(logits / temperature).  ``T`` broadcasts over the
    leading axes of ``logits`` (shape ``logits.shape[:-1]``).  Rows holding a
    NaN, a +inf or only -inf come out with NaN entries.
    """
    z = logits / np.asarray(T, np.float64)[..., None]
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        m = z.max(axis=-1, keepdims=True)
        e = np.exp(z - m)
        return e / e.sum(axis=-1, keepdims=True)


def first_argmax(logits: np.ndarray) -> np.ndarray:
    """Index of the largest logit, lowest index among equal maxima.

    [SD-intro] §ドラフト生成と並列検証の仕組み: greedy verification compares the
    draft with the token the target would pick, i.e. its most probable one.
    Equality is IEEE equality, so -0.0 and +0.0 tie.  A row with a NaN returns
    an arbitrary index (the caller flags the row).
    """
    m = logits.max(axis=-1, keepdims=True)
    return (logits == m).argmax(axis=-1)


def inverse_cdf(w: np.ndarray, u: np.ndarray):
    """Categorical draw from unnormalised weights ``w`` [..., V] with uniform ``u``.

    Returns (k, C, R): k = smallest index with C(k) > u * R where
    C(k) = sum_{x<=k} w(x) and R = C(V-1).  If rounding leaves no such k, the
    last index with w > 0 is returned.  The pages call this step
    ``torch.multinomial`` ([SpS] listing) without fixing an algorithm; the
    inverse CDF in vocabulary order is the reading taken here.
    """
    C = np.cumsum(w, axis=-1)
    R = C[..., -1]
    hit = C > (u * R)[..., None]
    k = hit.argmax(axis=-1)
    none = ~hit.any(axis=-1)
    if np.any(none):
        V = w.shape[-1]
        last_pos = V - 1 - (w[..., ::-1] > 0).argmax(axis=-1)
        k = np.where(none, last_pos, k)
    return k, C, R


def residual_distribution(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """p'(x) = norm(max(0, p(x) - q(x))).

    [SpS] §修正付き棄却サンプリング, the residual ("modified rejection")
    equation.  Returns NaN rows where the residual mass is zero.
    """
    r = np.maximum(0.0, p - q)
    with np.errstate(invalid="ignore", divide="ignore"):
        return r / r.sum(axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# Chain verification
# --------------------------------------------------------------------------

def _row_any(mask: np.ndarray, axes) -> np.ndarray:
    return np.any(mask, axis=axes)


def verify_chain(target_logits, draft, draft_is_probs, draft_tokens,
                 temperatures, uniforms, keep_cdf=False):
    """One verification step of chain speculative sampling, per batch row.

    Inputs (numpy, any float dtype; converted to float64):
      target_logits [B, gamma+1, V]  row i scores draft i; row gamma = bonus row
      draft         [B, gamma, V]    draft logits, or probabilities if
                                     ``draft_is_probs``
      draft_tokens  [B, gamma]       integer ids
      temperatures  [B]              T <= 0 selects greedy verification
      uniforms      [B, gamma+1]     column i < gamma: accept draw of draft i;
                                     column gamma: the single sample draw

    Steps, in the pages' order ([SpS] §技術的詳細 ステップ3 and
    §修正付き棄却サンプリング; [SD-intro] §ドラフト生成と並列検証の仕組み):
      1. p_i = softmax(target_i / T), q_i = softmax(draft_i / T) (or q given).
      2. For i = 1..gamma in order: accept x_i iff u_i q_i(x_i) < p_i(x_i).
      3. Stop at the first rejection j; drafts after it are discarded.
      4. j < gamma: draw from norm(max(0, p_j - q_j)); j == gamma: draw the
         bonus token from p_gamma.
      5. Emit x_0..x_{j-1} and the drawn token; ``num_accepted = j``.
    Greedy rows (T <= 0): a_i = first_argmax(target_i); j = first i with
    x_i != a_i (else gamma); emit x_0..x_{j-1}, a_j.  Draft rows are unused.

    Returns a dict with
      tokens [B, gamma+1] int64 (-1 after the emitted ones), num_accepted [B],
      status [B], diag [B, gamma, 4] = (p_i(x_i), q_i(x_i), min(1, p/q),
      residual mass R at i == j of a rejected row else 0), ratio [B, gamma]
      = p_i(x_i)/q_i(x_i) (inf if q = 0 < p, 0 if p = q = 0; used to spot
      boundary cases), j [B], greedy [B];
      with ``keep_cdf``: cdf [B, V] = C/R of the distribution each stochastic
      row drew its last token from (NaN rows for greedy or failed rows).
    """
    tl = np.asarray(target_logits, np.float64)
    dr = np.asarray(draft, np.float64)
    xt = np.asarray(draft_tokens, np.int64)
    T = np.asarray(temperatures, np.float64)
    u = np.asarray(uniforms, np.float64)
    B, G1, V = tl.shape
    gamma = G1 - 1
    assert xt.shape == (B, gamma) and u.shape == (B, G1) and T.shape == (B,)
    assert dr.shape == (B, gamma, V)

    tokens = np.full((B, G1), -1, np.int64)
    n_acc = np.zeros(B, np.int64)
    status = np.zeros(B, np.int64)
    diag = np.zeros((B, gamma, 4))
    ratio = np.zeros((B, gamma))
    jj = np.zeros(B, np.int64)
    cdf = np.full((B, V), np.nan) if keep_cdf else None

    greedy = T <= 0
    bad_T = np.isnan(T) | ((T > 0) & (T < TINY_T))
    tok_ok = np.all((xt >= 0) & (xt < V), axis=1)
    status[~tok_ok] |= ROW_BAD_TOKEN
    status[bad_T] |= ROW_BAD_TEMPERATURE
    xs = np.where((xt >= 0) & (xt < V), xt, 0)        # safe gather index

    # ---- greedy rows -----------------------------------------------------
    g = np.flatnonzero(greedy)
    if g.size:
        rows = tl[g]                                   # [g, gamma+1, V]
        status[g[_row_any(np.isnan(rows), (1, 2))]] |= ROW_NONFINITE
        a = first_argmax(rows)                         # [g, gamma+1]
        match = xs[g] == a[:, :gamma]
        j = np.where(match.all(axis=1), gamma, (~match).argmax(axis=1))
        jj[g] = j
        for r, b in enumerate(g):
            if status[b]:
                continue
            tokens[b, :j[r]] = xt[b, :j[r]]
            tokens[b, j[r]] = a[r, j[r]]
            n_acc[b] = j[r]

    # ---- stochastic rows -------------------------------------------------
    s = np.flatnonzero(~greedy & ~bad_T)
    if s.size:
        Ts = T[s]
        p = tempered_softmax(tl[s], Ts[:, None])                    # step 1
        if draft_is_probs:
            q = dr[s]
        else:
            q = tempered_softmax(dr[s], Ts[:, None])
        x = xs[s]
        px = np.take_along_axis(p[:, :gamma, :], x[..., None], axis=2)[..., 0]
        qx = np.take_along_axis(q, x[..., None], axis=2)[..., 0]
        bad = ~np.all(np.isfinite(p), axis=(1, 2))
        if draft_is_probs:
            # given probabilities are only read at q(x_i) and, after a
            # rejection, over row j (checked through the residual mass below)
            bad |= ~np.all(np.isfinite(qx), axis=1)
        else:
            bad |= ~np.all(np.isfinite(q), axis=(1, 2))
        accept = u[s, :gamma] * qx < px                             # step 2
        j = np.where(accept.all(axis=1), gamma, (~accept).argmax(axis=1))  # step 3

        with np.errstate(divide="ignore", invalid="ignore"):
            rat = np.where(qx > 0, px / np.where(qx > 0, qx, 1.0),
                           np.where(px > 0, np.inf, 0.0))
        acc_prob = np.minimum(1.0, rat)

        ar = np.arange(s.size)
        pj = p[ar, j]                                               # [s, V]
        qj = q[ar, np.minimum(j, gamma - 1)]
        resid = np.maximum(0.0, pj - qj)                            # step 4
        rejected = j < gamma
        w = np.where(rejected[:, None], resid, pj)
        Rres = np.cumsum(resid, axis=-1)[:, -1]
        bad |= rejected & np.isnan(Rres)
        status[s[bad]] |= ROW_NONFINITE
        zero_mass = rejected & ~(Rres > 0)
        w = np.where(zero_mass[:, None], pj, w)
        k, C, R = inverse_cdf(w, u[s, gamma])

        for r, b in enumerate(s):
            diag[b, :, 0] = px[r]
            diag[b, :, 1] = qx[r]
            diag[b, :, 2] = acc_prob[r]
            ratio[b] = rat[r]
            jj[b] = j[r]
            if rejected[r]:
                diag[b, j[r], 3] = Rres[r]
            if status[b]:
                continue
            tokens[b, :j[r]] = xt[b, :j[r]]                         # step 5
            tokens[b, j[r]] = k[r]
            n_acc[b] = j[r]
            if keep_cdf:
                with np.errstate(invalid="ignore", divide="ignore"):
                    cdf[b] = C[r] / R[r]

    out = dict(tokens=tokens, num_accepted=n_acc, status=status, diag=diag,
               ratio=ratio, j=jj, greedy=greedy)
    if keep_cdf:
        out["cdf"] = cdf
    return out


def verify_chain_greedy(target_logits, draft_tokens):
    """Greedy chain verification ([SD-intro] §ドラフト生成と並列検証の仕組み and
    the worked example in §候補の採用と棄却を具体例で見る).

    a_i = first_argmax(target_i); accept while x_i == a_i; at the first
    mismatch j (or j = gamma) emit a_j.  Same outputs as ``verify_chain``
    with every temperature <= 0.
    """
    tl = np.asarray(target_logits, np.float64)
    B, G1, V = tl.shape
    zeros = np.zeros((B, G1 - 1, V))
    T = np.zeros(B)
    u = np.zeros((B, G1))
    r = verify_chain(tl, zeros, False, draft_tokens, T, u)
    return dict(tokens=r["tokens"], num_accepted=r["num_accepted"],
                status=r["status"])


# --------------------------------------------------------------------------
# Token-tree greedy verification
# --------------------------------------------------------------------------

def verify_tree_greedy(node_logits, parent, node_tokens, max_depth):
    """SpecInfer-style greedy verification of a token tree, per tree.

    [SpecInfer] §技術の仕組み › 基本アイデア and §推論方法: the LLM scores every
    node in one pass, giving for each node the token that should follow it;
    the verifier then walks from the root along children whose token equals
    that prediction and commits the matched run.

    Inputs: node_logits [B, N, V]; parent [B, N] with parent[0] = -1 and
    0 <= parent[n] < n; node_tokens [B, N] (node 0 is the context's last
    token and is never verified); max_depth = most accepted edges.
    Walk: cur = 0; while depth < max_depth: among children c of cur with
    node_tokens[c] == a[cur] take the lowest index; stop if none.  The token
    a[cur] of the last node reached is appended as the correction / bonus.

    Returns dict(path [B, D+1], tokens [B, D+1], num_accepted [B], status [B])
    with D = max_depth; path holds the accepted node ids then -1, tokens the
    accepted node tokens, then a[cur], then -1.
    """
    lg = np.asarray(node_logits, np.float64)
    par = np.asarray(parent, np.int64)
    ntk = np.asarray(node_tokens, np.int64)
    B, N, V = lg.shape
    D = int(max_depth)
    path = np.full((B, D + 1), -1, np.int64)
    tokens = np.full((B, D + 1), -1, np.int64)
    n_acc = np.zeros(B, np.int64)
    status = np.zeros(B, np.int64)
    for b in range(B):
        if par[b, 0] != -1 or any(not (0 <= par[b, n] < n) for n in range(1, N)):
            status[b] |= ROW_BAD_TREE
        if np.any((ntk[b, 1:] < 0) | (ntk[b, 1:] >= V)):
            status[b] |= ROW_BAD_TOKEN
        if np.any(np.isnan(lg[b])):
            status[b] |= ROW_NONFINITE
        if status[b]:
            continue
        a = first_argmax(lg[b])
        cur, walk = 0, []
        while len(walk) < D:
            nxt = -1
            for c in range(N):
                if par[b, c] == cur and ntk[b, c] == a[cur]:
                    nxt = c
                    break
            if nxt < 0:
                break
            walk.append(nxt)
            cur = nxt
        d = len(walk)
        path[b, :d] = walk
        tokens[b, :d] = ntk[b, walk]
        tokens[b, d] = a[cur]
        n_acc[b] = d
    return dict(path=path, tokens=tokens, num_accepted=n_acc, status=status)


# --------------------------------------------------------------------------
# Draft-side sampling (the draft step that produces x_i ~ q)
# --------------------------------------------------------------------------

def draft_sample(logits, temperatures, uniforms):
    """One categorical draw per row from the draft distribution.

    [SpS] §アルゴリズム Step 1 and the ``speculative_decode`` listing: the
    draft model's next-token row goes through softmax(logits / T) and one
    token is drawn from it (``torch.multinomial``).  Readings shared with
    verification: the draw is the inverse CDF in ascending vocabulary order
    with the row's uniform (``inverse_cdf``); T <= 0 takes the first argmax.

    Inputs: logits [B, V], temperatures [B], uniforms [B] in [0, 1).
    Returns dict(tokens [B] int64, probs [B] float64 = q(token) (0 for greedy
    rows), status [B], cdf_lo [B], cdf_hi [B] = C(k-1)/R and C(k)/R of the
    drawn token (NaN for greedy or failed rows), for boundary accounting).
    Status: a NaN / +inf / all -inf softmax row or a NaN argmax row flags
    ROW_NONFINITE; a NaN temperature or one in (0, 1e-20) flags
    ROW_BAD_TEMPERATURE; such rows get token -1.
    """
    l = np.asarray(logits, np.float64)
    T = np.asarray(temperatures, np.float64)
    u = np.asarray(uniforms, np.float64)
    B, V = l.shape
    tokens = np.full(B, -1, np.int64)
    probs = np.zeros(B)
    status = np.zeros(B, np.int64)
    lo = np.full(B, np.nan)
    hi = np.full(B, np.nan)
    for b in range(B):
        t = T[b]
        if np.isnan(t) or (0.0 < t < TINY_T):
            status[b] = ROW_BAD_TEMPERATURE
            continue
        if t <= 0:
            if np.isnan(l[b]).any():
                status[b] = ROW_NONFINITE
                continue
            tokens[b] = int(first_argmax(l[b]))
            continue
        p = tempered_softmax(l[b][None], np.array([t]))[0]
        if not np.all(np.isfinite(p)):
            status[b] = ROW_NONFINITE
            continue
        k, C, R = inverse_cdf(p[None], np.array([u[b]]))
        k = int(k[0])
        tokens[b] = k
        probs[b] = p[k]
        lo[b] = (C[0, k - 1] if k > 0 else 0.0) / R[0]
        hi[b] = C[0, k] / R[0]
    return dict(tokens=tokens, probs=probs, status=status, cdf_lo=lo, cdf_hi=hi)


# --------------------------------------------------------------------------
# Token-tree attention mask
# --------------------------------------------------------------------------

def tree_ancestor_mask(parent):
    """Ancestor mask of every node of every token tree.

    [SpecInfer] §技術の仕組み › 基本アイデア and §推論方法: all tree nodes are
    scored in one target pass, which needs a topology-aware attention mask —
    a node sees itself and its ancestors (the path from the root), not its
    siblings or their subtrees.  Reading: mask[b, n, m] is True iff m == n
    or m is an ancestor of n; depth[b, n] counts the edges from the root.
    A malformed tree (parent[0] != -1 or parent[n] outside [0, n)) flags
    ROW_BAD_TREE and gets an all-False mask and depth 0.

    Input: parent int [B, N].  Returns dict(mask bool [B, N, N],
    depth int64 [B, N], status [B]).
    """
    par = np.asarray(parent, np.int64)
    B, N = par.shape
    mask = np.zeros((B, N, N), bool)
    depth = np.zeros((B, N), np.int64)
    status = np.zeros(B, np.int64)
    for b in range(B):
        ok = par[b, 0] == -1 and all(0 <= par[b, n] < n for n in range(1, N))
        if not ok:
            status[b] = ROW_BAD_TREE
            continue
        for n in range(N):
            cur, d = n, 0
            while cur >= 0:
                mask[b, n, cur] = True
                cur = par[b, cur]
                d += 1
            depth[b, n] = d - 1
    return dict(mask=mask, depth=depth, status=status)


# --------------------------------------------------------------------------
# KV-cache compaction after tree verification
# --------------------------------------------------------------------------

def tree_kv_compact(kv, base, path, num_accepted):
    """Keep the accepted path's KV rows of each tree, contiguous after the context.

    [SpS] §実装のポイント: the KV cache entries of rejected tokens are discarded;
    [SpecInfer] §推論方法: the tree's nodes were all scored in one pass, so
    their KV rows sit in node order after the context.  Reading: tree node n
    (1 <= n < N; node 0 is the context's last token) was written at slot
    base[b] + n - 1; after the walk the accepted path nodes path[b, 0..d-1]
    (d = num_accepted[b]) are moved to slots base[b] + 0..d-1, in path order,
    and the cache length becomes base[b] + d.  Rows of slots outside those
    moves are unchanged.  A row whose path is not a valid accepted path
    (d outside [0, path width], a node id not above the previous one or below
    i + 1, a slot outside the cache) flags ROW_BAD_TREE and moves nothing.

    Inputs: kv [B, S, E] (any dtype), base int [B], path int [B, Wp],
    num_accepted int [B].  Returns dict(kv (a new array), length [B], status [B]).
    """
    out = np.array(kv, copy=True)
    B, S = out.shape[:2]
    base = np.asarray(base, np.int64)
    path = np.asarray(path, np.int64)
    nacc = np.asarray(num_accepted, np.int64)
    length = base.copy()
    status = np.zeros(B, np.int64)
    for b in range(B):
        d = nacc[b]
        ok = 0 <= d <= path.shape[1] and base[b] >= 0
        prev = 0
        for i in range(d if ok else 0):
            p = path[b, i]
            if p < i + 1 or p <= prev or base[b] + p - 1 >= S:
                ok = False
                break
            prev = p
        if not ok:
            status[b] = ROW_BAD_TREE
            continue
        rows = [np.array(kv[b, base[b] + path[b, i] - 1], copy=True) for i in range(d)]
        for i in range(d):
            out[b, base[b] + i] = rows[i]
        length[b] = base[b] + d
    return dict(kv=out, length=length, status=status)


# --------------------------------------------------------------------------
# Rounds of speculative decoding (the multi-round model)
# --------------------------------------------------------------------------

def acceptance_probability(target_logits, draft_logits, T=1.0):
    """Chance that a draft drawn from q passes the accept test: sum_x min(p(x), q(x)).

    [SpS] §修正付き棄却サンプリング: a draft x ~ q is kept with probability
    min(1, p(x)/q(x)), so it is kept with probability
    sum_x q(x) min(1, p(x)/q(x)) = sum_x min(p(x), q(x)).  p and q are the
    tempered softmaxes of the rows (T > 0).  Inputs [..., V]; returns [...].
    """
    target_logits = np.asarray(target_logits, np.float64)
    T = np.broadcast_to(np.asarray(T, np.float64), target_logits.shape[:-1])
    p = tempered_softmax(target_logits, T)
    q = tempered_softmax(np.asarray(draft_logits, np.float64), T)
    return np.minimum(p, q).sum(axis=-1)


def accepted_count_law(alphas):
    """Law of n_accepted in one round: P(n = k) for k = 0..gamma.

    [SpS] §技術的詳細 ステップ3 and the listing's loop: drafts are tested in
    order and the round stops at the first rejection, so with independent
    per-position acceptance probabilities alpha_0..alpha_{gamma-1}
    P(n = k) = alpha_0 ... alpha_{k-1} (1 - alpha_k) for k < gamma and
    P(n = gamma) = alpha_0 ... alpha_{gamma-1}.  The round then commits
    n + 1 tokens (the replacement or the bonus token, §期待される高速化).
    """
    a = np.asarray(alphas, np.float64)
    g = a.shape[0]
    law = np.empty(g + 1)
    reach = 1.0
    for k in range(g):
        law[k] = reach * (1.0 - a[k])
        reach *= a[k]
    law[g] = reach
    return law


def expected_tokens_per_round(alphas):
    """E[tokens committed per round] = sum_k (k + 1) P(n_accepted = k).

    [SpS] §期待される高速化 gives (1 - alpha^(gamma+1)) / (1 - alpha) for a
    constant alpha; this is the same expectation for per-position alphas.
    """
    law = accepted_count_law(alphas)
    return float(np.dot(np.arange(1, law.shape[0] + 1), law))


def speedup_estimate(tokens_per_round, gamma, c):
    """Wall-clock speedup model of [SpS] §期待される高速化.

    A round costs gamma draft forwards of relative cost c plus one target
    forward, against one target forward per token without drafting:
    speedup = E[tokens per round] / (1 + gamma c).
    """
    return float(tokens_per_round) / (1.0 + gamma * float(c))
