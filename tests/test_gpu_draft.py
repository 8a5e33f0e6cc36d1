"""GPU parity of the draft-side draw (spec_draft_sample through the C ABI)
against the float64 oracle on the same seeded inputs.

Greedy rows must give the oracle's token exactly.  A stochastic row must give
the oracle's token unless its uniform lies within 1e-5 of a CDF boundary of
the drawn token (counted, at most 1% of rows); q(token) must match within
1e-4 for bf16/fp16 logits and 1e-5 for fp32.
"""

import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
from oracle.compare import prob_tolerance
from speculative_decoding_verification_48_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
EPS = 1e-5


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as pkg
    pkg.lib()
    return pkg


def _run(sv, case):
    out = sv.spec_draft_sample(case.logits.to(DEV), case.temperatures.to(DEV),
                               case.uniforms.to(DEV))
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def _check(sv, case, max_boundary_frac=0.01):
    tok, prob, st = _run(sv, case)
    l, T, u = case.numpy64()
    ref = oracle.draft_sample(l, T, u)
    assert np.array_equal(st, ref["status"])
    tol = prob_tolerance(case.meta["dtype"])
    boundary = 0
    for b in range(case.B):
        if ref["status"][b]:
            assert tok[b] == -1
            continue
        if T[b] <= 0:
            assert tok[b] == ref["tokens"][b], b
            continue
        if tok[b] == ref["tokens"][b]:
            assert abs(prob[b] - ref["probs"][b]) <= tol, (b, prob[b], ref["probs"][b])
            continue
        # a different token is allowed only at a CDF boundary of the oracle's CDF
        p = special.softmax(l[b] / T[b])
        C = np.cumsum(p)
        k = int(tok[b])
        lo = C[k - 1] / C[-1] if k > 0 else 0.0
        hi = C[k] / C[-1]
        dist = 0.0 if lo <= u[b] < hi else min(abs(u[b] - lo), abs(u[b] - hi))
        assert dist < EPS, (b, k, ref["tokens"][b], u[b], lo, hi)
        boundary += 1
    assert boundary <= max(2, int(max_boundary_frac * case.B)), boundary
    return tok, ref


def _temps(b, v):
    return [0.0, 0.7, 1.0, 1.3, 0.05, 2.0][b % 6] if b % 6 != 5 else 0.2 + 1.5 * v


@pytest.mark.parametrize("dtype,V,B", [("bf16", 128256, 64), ("f16", 32000, 33),
                                       ("f32", 1000, 300), ("bf16", 8, 500)])
def test_draft_sample_matches_oracle(sv, dtype, V, B):
    case = W.make_draft(f"draft_{dtype}_{V}", 5000 + V, B, V, dtype, temperature=_temps)
    tok, ref = _check(sv, case)
    assert len(set(tok.tolist())) > 2


def test_draft_sample_edge_rows(sv):
    case = W.make_draft("draft_edges", 5100, 8, 4096, "f32", target="normal", sigma=2.0,
                        temperature=1.0)
    lg = case.logits
    lg[1, 7] = float("nan")                    # NaN logit
    lg[2, :] = float("-inf")                   # all -inf
    lg[3, ::2] = float("-inf")                 # half the vocabulary impossible
    lg[4, :] = 1.0                             # flat row: exact ties
    case.temperatures[5] = float("nan")        # invalid temperature
    case.temperatures[6] = 0.0                 # greedy with ties below
    lg[6, :] = 0.0
    lg[6, 100] = 3.0
    lg[6, 3000] = 3.0
    case.temperatures[7] = 1e-3                # very small T
    tok, ref = _check(sv, case)
    assert ref["status"][1] and ref["status"][2] and ref["status"][5]
    assert tok[6] == 100
    assert tok[3] % 2 == 1


def test_draft_sample_distribution_on_gpu(sv):
    """Many rows of one V = 8 distribution: the drawn tokens follow
    softmax(l / T) (chi-square against scipy's softmax)."""
    V, n, T = 8, 200000, 0.9
    base = torch.tensor([0.3, -1.0, 2.0, 0.0, 1.1, -0.4, 0.8, -2.0], dtype=torch.float32)
    logits = base.repeat(n, 1).to(DEV)
    g = torch.Generator().manual_seed(77)
    u = torch.rand(n, generator=g).to(DEV)
    tok, prob, st = sv.spec_draft_sample(logits, torch.full((n,), T, device=DEV), u)
    torch.cuda.synchronize()
    tok = tok.cpu().numpy()
    assert not st.cpu().numpy().any()
    obs = np.bincount(tok, minlength=V)
    exp = special.softmax(base.numpy().astype(np.float64) / T) * n
    assert stats.chisquare(obs, exp * (obs.sum() / exp.sum())).pvalue > 1e-3


@pytest.mark.parametrize("dtype,V", [("bf16", 1001), ("f16", 70001), ("f32", 4099), ("bf16", 3)])
def test_draft_sample_unaligned_rows(sv, dtype, V):
    """Rows that do not start on 16-byte boundaries (odd V in 16-bit types,
    V not a multiple of 4 in fp32): each row's chunks sit on the row's own
    16-byte grid and its edge vectors are read element by element.  Greedy
    and tiny-T rows included."""
    case = W.make_draft(f"draft_odd_{dtype}_{V}", 5200 + V % 97, 13, V, dtype,
                        temperature=_temps)
    _check(sv, case)


def test_draft_sample_unaligned_view(sv):
    """A view that starts 2 bytes into an allocation: every row is off the
    16-byte grid, including the first."""
    case = W.make_draft("draft_view", 5300, 9, 4096, "bf16", temperature=_temps)
    buf = torch.empty(case.B * case.V + 1, dtype=torch.bfloat16, device=DEV)
    view = buf[1:].view(case.B, case.V)
    view.copy_(case.logits.to(DEV))
    tok, prob, st = sv.spec_draft_sample(view, case.temperatures.to(DEV), case.uniforms.to(DEV))
    torch.cuda.synchronize()
    l, T, u = case.numpy64()
    ref = oracle.draft_sample(l, T, u)
    assert np.array_equal(st.cpu().numpy(), ref["status"])
    greedy = T <= 0
    assert np.array_equal(tok.cpu().numpy()[greedy], ref["tokens"][greedy])
