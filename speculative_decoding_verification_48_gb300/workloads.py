"""Seeded synthetic inputs for speculative-sampling verification.

This module only *creates* inputs: logits, draft tokens, temperatures,
uniform draws and token trees.  It holds none of the verification arithmetic
(no accept test, no residual, no argmax walk), so the library and the float64
oracle used by the tests can both consume its output without sharing code.

Every batch row (or tree) is drawn from its own torch CPU generator seeded
from ``(seed, row)``, so any subset of rows can be regenerated on its own.
Values are drawn in float32 and rounded to the storage dtype by
``torch.Tensor.to`` (round to nearest even); consumers read the rounded
values back.

Draft tokens are drawn from the draft distribution q = softmax(draft / T)
with ``torch.multinomial`` (draft generation, step 1 of the method, as in the
pages' own drafting loop); greedy rows (T <= 0) use the draft's own top
token.  None of this is verification.

Workloads (the pages measure on XSum, HumanEval, WMT and Alpaca; these
synthetic shapes stand in for them):
  c1  chain, B=256 rounds, gamma=4, V=1000, fp32; target ~ N(0, 2^2),
      draft = target + N(0, 0.5^2), T = 1.
  c2  chain, 4096 rounds, gamma=5, V=32000, bf16; Zipf-biased target
      N(0,1) - 1.1 ln(rank), draft = target + N(0,1), T in {0, 0.7, 1.0}.
  c3  chain, B=64, gamma=7, V=128256, bf16; Zipf-biased target, per-row draft
      noise sigma ~ U[0.3, 2.0], per-row T ~ U[0, 1.2) with T = 0 on rows
      b % 8 == 0 (greedy rows).
  c4  token trees, 16 trees x 64 nodes, depth <= 8, 1..4 children per node,
      fp16 node logits ~ N(0, 2^2), one planted root path matching the
      target argmax with probability 0.8 per step.
  c5  chain, B=256, gamma=4, V=256000; bf16 Zipf-biased target at T = 0.8;
      draft given as fp32 probabilities softmax(target + N(0, 0.7^2)) (the
      input data, computed here once); rows b % 16 == 0 have their accept
      draws set to 0 (all drafts accepted, bonus token drawn).
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def seed_for(*keys: int) -> int:
    """63-bit seed derived from the integer keys (SeedSequence mixing)."""
    st = np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in keys]).generate_state(2, np.uint32)
    return int((int(st[0]) << 31) ^ int(st[1])) & ((1 << 63) - 1)


def gen_for(*keys: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed_for(*keys))
    return g


def uniform(g: torch.Generator, lo: float = 0.0, hi: float = 1.0) -> float:
    return lo + (hi - lo) * float(torch.rand((), generator=g, dtype=torch.float64))


def round_to(x, dtype: str) -> torch.Tensor:
    """Round float data to the storage dtype (round to nearest even)."""
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return x.to(torch.float32).to(DTYPES[dtype])


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Stored values as float64 numpy (exact for fp32 / bf16 / fp16)."""
    return t.detach().to("cpu", torch.float64).numpy()


def zipf_bias(seed: int, V: int) -> torch.Tensor:
    """-1.1 * ln(rank(x)) with rank = perm(x) + 1, one permutation per seed."""
    perm = torch.randperm(V, generator=gen_for(seed, 0x7FFFFFFF)).to(torch.float64)
    return (-1.1 * torch.log(perm + 1.0)).to(torch.float32)


@dataclass
class ChainCase:
    name: str
    target: torch.Tensor          # [B, gamma+1, V] storage dtype (CPU)
    draft: torch.Tensor           # [B, gamma, V] logits, or fp32 probabilities
    draft_is_probs: bool
    draft_tokens: torch.Tensor    # int32 [B, gamma]
    temperatures: torch.Tensor    # fp32 [B]
    uniforms: torch.Tensor        # fp32 [B, gamma+1]
    meta: dict = field(default_factory=dict)

    @property
    def B(self): return self.target.shape[0]
    @property
    def gamma(self): return self.target.shape[1] - 1
    @property
    def V(self): return self.target.shape[2]

    def select(self, rows: Sequence[int]) -> "ChainCase":
        idx = torch.as_tensor(list(rows), dtype=torch.long)
        return ChainCase(self.name, self.target[idx].contiguous(), self.draft[idx].contiguous(),
                         self.draft_is_probs, self.draft_tokens[idx].contiguous(),
                         self.temperatures[idx].contiguous(), self.uniforms[idx].contiguous(),
                         dict(self.meta))

    def numpy64(self):
        """Arguments for the float64 oracle, in its argument order."""
        return (to_f64(self.target), to_f64(self.draft), self.draft_is_probs,
                self.draft_tokens.numpy().astype(np.int64),
                to_f64(self.temperatures), to_f64(self.uniforms))


@dataclass
class TreeCase:
    name: str
    node_logits: torch.Tensor     # [B, N, V] storage dtype (CPU)
    parent: torch.Tensor          # int32 [B, N]
    node_tokens: torch.Tensor     # int32 [B, N]
    max_depth: int
    meta: dict = field(default_factory=dict)

    @property
    def B(self): return self.node_logits.shape[0]
    @property
    def N(self): return self.node_logits.shape[1]
    @property
    def V(self): return self.node_logits.shape[2]

    def numpy64(self):
        return (to_f64(self.node_logits), self.parent.numpy().astype(np.int64),
                self.node_tokens.numpy().astype(np.int64), self.max_depth)


def make_chain(name: str, seed: int, B: int, gamma: int, V: int, dtype: str = "bf16",
               target: str = "zipf", target_sigma: float = 1.0,
               draft_sigma: tuple = (1.0, 1.0),
               temperature: Callable[[int, float], float] | float = 1.0,
               draft_probs: bool = False, draft_probs_T: float = 1.0,
               force_accept_every: int = 0, row0: int = 0) -> ChainCase:
    """General chain workload; row b uses the generator (seed, row0 + b), so
    a batch starting at ``row0`` continues the same row stream.

    target: "zipf" -> N(0, target_sigma^2) - 1.1 ln(rank); "normal" ->
    N(0, target_sigma^2).  Draft logits = target (before rounding) + N(0, s_b^2)
    with s_b ~ U[draft_sigma].  ``temperature`` is a constant or a callable
    (b, v) -> T of a per-row uniform v in [0, 1).  With ``draft_probs`` the
    draft is stored as fp32 probabilities softmax((target + noise) /
    draft_probs_T) and the target keeps the row temperature.
    """
    bias = zipf_bias(seed, V) if target == "zipf" else None
    tgt = torch.empty((B, gamma + 1, V), dtype=DTYPES[dtype])
    ddt = "f32" if draft_probs else dtype
    dft = torch.empty((B, gamma, V), dtype=DTYPES[ddt])
    toks = torch.empty((B, gamma), dtype=torch.int32)
    temps = torch.empty(B, dtype=torch.float32)
    unif = torch.empty((B, gamma + 1), dtype=torch.float32)
    for i in range(B):
        b = row0 + i
        g = gen_for(seed, b)
        base = torch.randn((gamma + 1, V), generator=g) * float(target_sigma)
        if bias is not None:
            base += bias
        s_b = uniform(g, draft_sigma[0], draft_sigma[1])
        dl = base[:gamma] + torch.randn((gamma, V), generator=g) * float(s_b)
        v = uniform(g)
        T = float(temperature(b, v)) if callable(temperature) else float(temperature)
        temps[i] = T
        unif[i] = torch.rand(gamma + 1, generator=g)
        if force_accept_every and b % force_accept_every == 0:
            unif[i, :gamma] = 0.0
        tgt[i] = base.to(DTYPES[dtype])
        if draft_probs:
            q = torch.softmax(dl / draft_probs_T, dim=-1)
            dft[i] = q
            toks[i] = torch.multinomial(q, 1, generator=g)[:, 0].to(torch.int32)
        else:
            dft[i] = dl.to(DTYPES[dtype])
            dr = dft[i].to(torch.float32)
            if T <= 0:
                toks[i] = torch.argmax(dr, dim=-1).to(torch.int32)
            else:
                q = torch.softmax(dr / T, dim=-1)
                toks[i] = torch.multinomial(q, 1, generator=g)[:, 0].to(torch.int32)
    return ChainCase(name, tgt, dft, draft_probs, toks, temps, unif,
                     dict(seed=seed, dtype=dtype, draft_dtype=ddt))


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def c1_spec(rounds: int = 256, seed: int = 1001) -> dict:
    """Keyword arguments of ``make_chain`` for C1 (any subset of its rows can
    be regenerated with ``make_chain(**{**spec, "B": n, "row0": r0})``)."""
    return dict(name=f"c1_chain_B1x{rounds}rounds_g4_V1000_f32", seed=seed, B=rounds, gamma=4,
                V=1000, dtype="f32", target="normal", target_sigma=2.0, draft_sigma=(0.5, 0.5),
                temperature=1.0)


def c2_spec(T: float, rounds: int = 4096, seed: int = 1002) -> dict:
    return dict(name=f"c2_chain_B1x{rounds}rounds_g5_V32000_bf16_T{T}", seed=seed, B=rounds,
                gamma=5, V=32000, dtype="bf16", target="zipf", draft_sigma=(1.0, 1.0),
                temperature=float(T))


def _c3_temperature(b: int, v: float) -> float:
    return 0.0 if b % 8 == 0 else 1.2 * v


def c3_spec(B: int = 64, gamma: int = 7, V: int = 128256, seed: int = 1003) -> dict:
    return dict(name=f"c3_chain_B{B}_g{gamma}_V{V}_bf16", seed=seed, B=B, gamma=gamma, V=V,
                dtype="bf16", target="zipf", draft_sigma=(0.3, 2.0), temperature=_c3_temperature)


def c5_spec(B: int = 256, gamma: int = 4, V: int = 256000, seed: int = 1005) -> dict:
    return dict(name=f"c5_chain_B{B}_g{gamma}_V{V}_bf16_f32probs", seed=seed, B=B, gamma=gamma,
                V=V, dtype="bf16", target="zipf", draft_sigma=(0.7, 0.7), temperature=0.8,
                draft_probs=True, draft_probs_T=1.0, force_accept_every=16)


def c1_chain_fp32_v1000(rounds: int = 256, seed: int = 1001) -> ChainCase:
    return make_chain(**c1_spec(rounds, seed))


def c2_chain_bf16_v32000(T: float, rounds: int = 4096, seed: int = 1002) -> ChainCase:
    return make_chain(**c2_spec(T, rounds, seed))


def c3_chain_bf16_v128256(B: int = 64, gamma: int = 7, V: int = 128256,
                          seed: int = 1003) -> ChainCase:
    return make_chain(**c3_spec(B, gamma, V, seed))


def c5_chain_bf16_probs_v256000(B: int = 256, gamma: int = 4, V: int = 256000,
                                seed: int = 1005) -> ChainCase:
    return make_chain(**c5_spec(B, gamma, V, seed))


def concat_chain(parts: Sequence[ChainCase], name: Optional[str] = None) -> ChainCase:
    """One case holding the rows of ``parts`` in order."""
    cat = lambda f: torch.cat([getattr(c, f) for c in parts])  # noqa: E731
    return ChainCase(name or parts[0].name, cat("target"), cat("draft"), parts[0].draft_is_probs,
                     cat("draft_tokens"), cat("temperatures"), cat("uniforms"),
                     dict(parts[0].meta))


def make_tree(name: str, seed: int, B: int = 16, N: int = 64, V: int = 32000,
              max_depth: int = 8, kmin: int = 1, kmax: int = 4, dtype: str = "f16",
              sigma: float = 2.0, p_match: float = 0.8) -> TreeCase:
    """Token trees given as parent-index arrays (BFS numbering, parent[n] < n).

    Each node gets kmin..kmax children until N nodes exist; no node deeper than
    ``max_depth``.  Sibling tokens are distinct.  Along one random root-to-leaf
    path, each step is planted: with probability ``p_match`` the parent's logit
    row is raised at the child's token (to the row maximum + 1) so the target's
    top token is that child; otherwise the parent's logit at the child's token
    is set below the row minimum so the child does not match.
    """
    logits = torch.empty((B, N, V), dtype=DTYPES[dtype])
    parents = np.empty((B, N), np.int32)
    tokens = np.empty((B, N), np.int32)
    for b in range(B):
        rng = np.random.Generator(np.random.SFC64(seed_for(seed, b, 1)))
        g = gen_for(seed, b)
        par, dep = [-1], [0]
        queue = deque([0])
        while len(par) < N:
            if not queue:
                queue = deque(n for n in range(len(par)) if dep[n] < max_depth)
                if not queue:
                    raise ValueError("tree cannot reach N nodes within max_depth")
            n = queue.popleft()
            if dep[n] >= max_depth:
                continue
            k = int(rng.integers(kmin, kmax + 1))
            for _ in range(k):
                if len(par) >= N:
                    break
                par.append(n)
                dep.append(dep[n] + 1)
                queue.append(len(par) - 1)
        par_a = np.asarray(par, np.int32)
        children = [np.flatnonzero(par_a == n) for n in range(N)]
        tok = np.empty(N, np.int32)
        tok[0] = rng.integers(0, V)
        for n in range(N):
            if len(children[n]):
                tok[children[n]] = rng.choice(V, size=len(children[n]), replace=False)
        lg = torch.randn((N, V), generator=g) * float(sigma)
        cur = 0
        while len(children[cur]):
            c = int(rng.choice(children[cur]))
            if rng.random() < p_match:
                lg[cur, int(tok[c])] = lg[cur].max() + 1.0
            else:
                lg[cur, int(tok[c])] = lg[cur].min() - 1.0
            cur = c
        logits[b] = lg.to(DTYPES[dtype])
        parents[b] = par_a
        tokens[b] = tok
    return TreeCase(name, logits, torch.from_numpy(parents), torch.from_numpy(tokens),
                    max_depth, dict(seed=seed, dtype=dtype))


def c4_tree_f16_v32000(B: int = 16, N: int = 64, V: int = 32000, seed: int = 1004) -> TreeCase:
    return make_tree(f"c4_tree_B{B}_N{N}_V{V}_f16", seed, B, N, V, max_depth=8)


# Algorithmic bytes: every logit byte the verification needs, read once.

def chain_algorithmic_bytes(case: ChainCase, num_accepted: Optional[np.ndarray] = None) -> int:
    """Target rows of every batch row; draft logit rows of stochastic rows;
    in probability mode the draft row at the rejected position only (needs
    the call's ``num_accepted``); plus draft tokens, temperatures, uniforms."""
    B, g, V = case.B, case.gamma, case.V
    te = case.target.element_size()
    de = case.draft.element_size()
    T = case.temperatures.numpy()
    stoch = T > 0
    nbytes = B * (g + 1) * V * te
    if case.draft_is_probs:
        if num_accepted is not None:
            rej = stoch & (np.asarray(num_accepted) < g)
            nbytes += int(rej.sum()) * V * de
        nbytes += int(stoch.sum()) * g * de         # gathers q(x)
    else:
        nbytes += int(stoch.sum()) * g * V * de
    nbytes += B * g * 4 + B * 4 + B * (g + 1) * 4
    return int(nbytes)


def tree_algorithmic_bytes(case: TreeCase) -> int:
    B, N, V = case.B, case.N, case.V
    return int(B * N * V * case.node_logits.element_size() + 2 * B * N * 4)


@dataclass
class DraftCase:
    """Draft-side draws: one logit row per batch entry."""
    name: str
    logits: torch.Tensor        # [B, V]
    temperatures: torch.Tensor  # [B]
    uniforms: torch.Tensor      # [B]
    meta: dict = field(default_factory=dict)

    @property
    def B(self): return self.logits.shape[0]

    @property
    def V(self): return self.logits.shape[1]

    def numpy64(self):
        return to_f64(self.logits), self.temperatures.double().numpy(), self.uniforms.double().numpy()


def make_draft(name: str, seed: int, B: int, V: int, dtype: str = "bf16", target: str = "zipf",
               sigma: float = 1.0, temperature: Callable[[int, float], float] | float = 1.0,
               row0: int = 0) -> DraftCase:
    """Draft-model next-token rows: N(0, sigma^2) (+ Zipf bias -1.1 ln(rank)),
    a temperature per row (constant or (b, v) -> T of a per-row uniform v)
    and one uniform per row; row b uses the generator (seed, row0 + b)."""
    bias = zipf_bias(seed, V) if target == "zipf" else None
    logits = torch.empty((B, V), dtype=DTYPES[dtype])
    temps = torch.empty(B, dtype=torch.float32)
    unif = torch.empty(B, dtype=torch.float32)
    for i in range(B):
        g = gen_for(seed, row0 + i)
        row = torch.randn(V, generator=g) * float(sigma)
        if bias is not None:
            row += bias
        v = uniform(g)
        temps[i] = float(temperature(row0 + i, v)) if callable(temperature) else float(temperature)
        unif[i] = torch.rand(1, generator=g)[0]
        logits[i] = row.to(DTYPES[dtype])
    return DraftCase(name, logits, temps, unif, dict(seed=seed, dtype=dtype))


@dataclass
class AlphaPair:
    """One target row and one draft row whose distributions overlap by a
    known amount: sum_x min(p(x), q(x)) = alpha, where p and q are the
    distributions the stored fp32 logits define at T = 1.

    p is a random distribution, p(x) proportional to exp(N(0, sigma^2)),
    stored as target logits log p.  q moves weight w of p onto the least
    likely token k, q = (1 - w) p + w e_k, stored as draft logits log q.
    The overlap of such a pair is 1 - w (1 - p(k)), so
    w = (1 - alpha) / (1 - p(k)) gives alpha exactly; the fp32 rounding of
    the stored logits moves it by about 1e-7.
    """
    target_logits: torch.Tensor    # fp32 [V]
    draft_logits: torch.Tensor     # fp32 [V]
    alpha: float
    k: int
    w: float


def make_alpha_pair(seed: int, V: int, alpha: float, sigma: float = 1.5) -> AlphaPair:
    if not 0.0 < alpha <= 1.0:
        raise ValueError("alpha must lie in (0, 1]")
    if V < 2:
        raise ValueError("V must be at least 2")
    g = gen_for(seed, 0xA1FA)
    z = torch.randn(V, generator=g, dtype=torch.float64) * sigma
    p = torch.exp(z - z.max())
    p = p / p.sum()
    k = int(torch.argmin(p))
    w = (1.0 - alpha) / (1.0 - float(p[k]))
    q = (1.0 - w) * p
    q[k] += w
    return AlphaPair(torch.log(p).to(torch.float32), torch.log(q).to(torch.float32),
                     float(alpha), k, float(w))
