"""Multi-round speculative decoding driven through the library's kernels.

One round of the method ("論文解説: Speculative Sampling", §投機的サンプリングの
アルゴリズム and §技術的詳細 ステップ1–3):

- the draft proposes gamma tokens, each drawn from q (``spec_draft_sample``);
- the target verifies them (``spec_verify_chain``);
- the round commits n_accepted + 1 tokens.

The page's §期待される高速化 models the tokens per round as
(1 - alpha^(gamma+1)) / (1 - alpha) and the wall-clock speedup as
E / (1 + gamma c). ``simulate`` measures the tokens per round on the GPU
and reports that model beside it. ``sweep`` runs one alpha over
gamma = 1..8: the look-ahead sweep the page describes from the paper's
Figure 5.

Inputs:

- One synthetic target row and one draft row of known overlap alpha
  (``workloads.make_alpha_pair``), the same at every position and in every
  round.
- These synthetic distributions do not depend on the context. So rounds are
  independent draws, and committed tokens need not be fed back.
- Each of ``sequences`` sequences runs rounds until it has committed
  ``tokens`` tokens. The last round's surplus counts, as a decoder would
  commit it too.
- All sequences of one round share one draft-sample call and one verify
  call. Uniforms come from a seeded torch generator on the device.
"""

from __future__ import annotations

import argparse
import json
from dataclasses import asdict, dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import binding as B
from . import workloads as W


@dataclass
class RoundStats:
    gamma: int
    alpha: float                 # design overlap of the p / q pair
    c: float                     # draft forward cost relative to the target's
    sequences: int
    tokens_per_sequence: int
    rounds: int                  # rounds run, over all sequences
    tokens: int                  # tokens committed, over all sequences
    tokens_per_round: float      # measured E[tokens per round]
    tokens_per_round_se: float   # its standard error
    accept_rate: List[float]     # per draft position: accepted / tested
    n_accepted_hist: List[int]   # rounds with n_accepted = 0..gamma
    model_tokens_per_round: float  # (1 - alpha^(gamma+1)) / (1 - alpha)
    speedup_model: float         # measured E / (1 + gamma c)
    us_per_round: float          # device time between events recorded before the draft-sample
                                 # call and after the verify call (host launch gaps included)
    V: int


def _closed_form(alpha: float, gamma: int) -> float:
    if alpha >= 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def simulate(gamma: int, alpha: float, *, sequences: int = 1024, tokens: int = 128,
             V: int = 4096, c: float = 0.05, seed: int = 0,
             device: Optional[torch.device] = None) -> RoundStats:
    """Run rounds of draft sampling + verification on the GPU until every
    sequence has committed ``tokens`` tokens.  Work is enqueued on torch's
    current stream of ``device``."""
    if gamma < 1 or sequences < 1 or tokens < 1:
        raise ValueError("gamma, sequences and tokens must be positive")
    dev = torch.device(device) if device is not None else torch.device("cuda")
    if dev.type != "cuda":
        raise ValueError("the simulator runs the library's CUDA kernels; give a CUDA device")
    pair = W.make_alpha_pair(seed, V, alpha)
    S = sequences
    target = pair.target_logits.to(dev).expand(S, gamma + 1, V).contiguous()
    draft = pair.draft_logits.to(dev).expand(S, gamma, V).contiguous()
    temps = torch.ones(S, dtype=torch.float32, device=dev)
    dtemps = torch.ones(S * gamma, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(W.seed_for(seed, gamma, 0x5151))

    d_tok = torch.empty(S * gamma, dtype=torch.int32, device=dev)
    d_prob = torch.empty(S * gamma, dtype=torch.float32, device=dev)
    d_st = torch.empty(S * gamma, dtype=torch.int32, device=dev)
    v_tok = torch.empty((S, gamma + 1), dtype=torch.int32, device=dev)
    v_nacc = torch.empty(S, dtype=torch.int32, device=dev)
    v_st = torch.empty(S, dtype=torch.int32, device=dev)
    committed = torch.zeros(S, dtype=torch.int64, device=dev)
    hist = torch.zeros(gamma + 1, dtype=torch.int64, device=dev)
    bad = torch.zeros((), dtype=torch.bool, device=dev)
    stream = torch.cuda.current_stream(dev)
    events = []
    rounds = 0
    while True:
        active = committed < tokens
        n_active = int(active.sum())
        if n_active == 0:
            break
        ud = torch.rand(S * gamma, generator=gen, device=dev)
        uv = torch.rand((S, gamma + 1), generator=gen, device=dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        B.spec_draft_sample(draft.view(S * gamma, V), dtemps, ud, out_tokens=d_tok,
                            out_probs=d_prob, out_row_status=d_st)
        B.spec_verify_chain(target, draft, d_tok.view(S, gamma), temps, uv, out_tokens=v_tok,
                            out_num_accepted=v_nacc, out_row_status=v_st, want_diag=False)
        b.record(stream)
        events.append((a, b))
        n = v_nacc.to(torch.int64)
        hist += torch.bincount(n[active], minlength=gamma + 1)
        committed += torch.where(active, n + 1, torch.zeros_like(n))
        bad |= (d_st != 0).any() | (v_st != 0).any()
        rounds += n_active
    torch.cuda.synchronize(dev)
    if bool(bad):
        raise RuntimeError("a draft-sample or verify row reported a data error")
    h = hist.cpu().numpy().astype(np.int64)
    k = np.arange(gamma + 1)
    E = float(((k + 1) * h).sum() / rounds)
    var = float(((k + 1 - E) ** 2 * h).sum() / max(rounds - 1, 1))
    reach = np.cumsum(h[::-1])[::-1]                 # rounds with n_accepted >= i
    acc = [float(reach[i + 1] / reach[i]) if reach[i] else float("nan") for i in range(gamma)]
    us = float(np.median([x.elapsed_time(y) for x, y in events]) * 1e3)
    return RoundStats(gamma=gamma, alpha=float(alpha), c=float(c), sequences=S,
                      tokens_per_sequence=tokens, rounds=rounds,
                      tokens=int(committed.sum()), tokens_per_round=E,
                      tokens_per_round_se=float(np.sqrt(var / rounds)), accept_rate=acc,
                      n_accepted_hist=h.tolist(),
                      model_tokens_per_round=_closed_form(alpha, gamma),
                      speedup_model=E / (1.0 + gamma * c), us_per_round=us, V=V)


def sweep(alpha: float, gammas: Sequence[int] = range(1, 9), **kw) -> List[RoundStats]:
    """``simulate`` at each look-ahead in ``gammas``."""
    return [simulate(g, alpha, **kw) for g in gammas]


def _parse_gammas(s: str) -> List[int]:
    if "-" in s:
        lo, hi = s.split("-")
        return list(range(int(lo), int(hi) + 1))
    return [int(x) for x in s.split(",")]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--alpha", type=float, default=0.8)
    ap.add_argument("--c", type=float, default=0.05)
    ap.add_argument("--gammas", default="1-8")
    ap.add_argument("--sequences", type=int, default=1024)
    ap.add_argument("--tokens", type=int, default=128)
    ap.add_argument("--vocab", type=int, default=4096)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--json", action="store_true", help="one JSON line per gamma")
    a = ap.parse_args(argv)
    res = sweep(a.alpha, _parse_gammas(a.gammas), sequences=a.sequences, tokens=a.tokens,
                V=a.vocab, c=a.c, seed=a.seed)
    if a.json:
        for r in res:
            print(json.dumps(asdict(r)))
        return
    print(f"alpha = {a.alpha}, c = {a.c}, {a.sequences} sequences x {a.tokens} tokens, "
          f"V = {a.vocab}")
    print(" gamma  tokens/round (measured)  model  speedup (model, measured E)  us/round")
    for r in res:
        print(f"{r.gamma:6d}  {r.tokens_per_round:10.4f} +- {r.tokens_per_round_se:.4f}  "
              f"{r.model_tokens_per_round:8.4f}  {r.speedup_model:10.3f}  {r.us_per_round:12.1f}")
    best = max(res, key=lambda r: r.speedup_model)
    print(f"best gamma by the speedup model: {best.gamma}")


if __name__ == "__main__":
    main()
