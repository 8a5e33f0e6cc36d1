"""GPU parity: the CUDA library (called through the C ABI) against the float64
oracle on the same seeded inputs.

Greedy and tree outputs are bit-exact.  Stochastic rows must match exactly
except boundary cases (a uniform within 1e-5 of an acceptance ratio or CDF
boundary), which are counted; diagnostic probabilities match within 1e-4
(bf16/fp16 logits) or 1e-5 (fp32 logits).
"""

import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
from oracle.compare import compare_chain, prob_tolerance
import chunked_oracle as CO
from speculative_decoding_verification_48_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as pkg
    pkg.lib()
    return pkg


DEV = torch.device("cuda:0")


def run_chain(sv, case):
    out = sv.spec_verify_chain(case.target.to(DEV), case.draft.to(DEV),
                               case.draft_tokens.to(DEV), case.temperatures.to(DEV),
                               case.uniforms.to(DEV), draft_is_probs=case.draft_is_probs)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def check_chain(sv, case, rows=None, max_boundary=None):
    toks, nacc, diag, st = run_chain(sv, case)
    sub = case if rows is None else case.select(rows)
    if rows is not None:
        toks, nacc, diag, st = toks[rows], nacc[rows], diag[rows], st[rows]
    args = sub.numpy64()
    ref = oracle.verify_chain(*args)
    tol = prob_tolerance(case.meta.get("dtype", "bf16"))
    cmp = compare_chain(args, ref, toks, nacc, st, diag, prob_tol=tol)
    assert not cmp["failures"], cmp["failures"][:5]
    B = len(toks)
    lim = max(2, int(0.01 * B)) if max_boundary is None else max_boundary
    assert len(cmp["boundary"]) <= lim, cmp["boundary"]
    return cmp, ref, (toks, nacc, diag, st)


def run_tree(sv, case):
    out = sv.spec_verify_tree_greedy(case.node_logits.to(DEV), case.parent.to(DEV),
                                     case.node_tokens.to(DEV), case.max_depth)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def check_tree(sv, case):
    path, toks, nacc, st = run_tree(sv, case)
    ref = oracle.verify_tree_greedy(*case.numpy64())
    assert np.array_equal(st, ref["status"])
    assert np.array_equal(nacc, ref["num_accepted"])
    assert np.array_equal(toks, ref["tokens"])
    assert np.array_equal(path, ref["path"])
    return ref


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def test_c1_chain_fp32_v1000(sv):
    cmp, ref, _ = check_chain(sv, W.c1_chain_fp32_v1000())
    assert cmp["exact"] + len(cmp["boundary"]) == 256


@pytest.fixture(scope="module")
def pool():
    p = CO.spawn_pool()
    yield p
    p.close()
    p.join()


def check_full(sv, pool, spec, gen_chunk, cmp_chunk, tol):
    """All rows of a workload through one library call, compared with the
    oracle chunk by chunk in the pool."""
    case = CO.generate(pool, spec, gen_chunk)
    B = case.B
    outs = run_chain(sv, case)
    del case
    cmp = CO.compare(pool, spec, outs, cmp_chunk, tol)
    assert not cmp["failures"], cmp["failures"][:5]
    assert len(cmp["boundary"]) <= max(2, int(0.01 * B)), cmp["boundary"]
    assert cmp["exact"] + len(cmp["boundary"]) == B
    return cmp, outs


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_c2_chain_bf16_v32000_all_rounds(sv, pool, T):
    """C2 in full: all 4096 rounds at each temperature in one batched call."""
    cmp, _ = check_full(sv, pool, W.c2_spec(T), 256, 128, 1e-4)
    if T == 0.0:
        assert cmp["greedy"].all()
    assert len(set(cmp["num_accepted"].tolist())) >= 3


def _single_rounds(sv, case, rounds):
    """One library call per round (B = 1), the call shape the bench times."""
    args = [t.to(DEV) for t in (case.target, case.draft, case.draft_tokens, case.temperatures,
                                case.uniforms)]
    ws = torch.zeros(sv.spec_verify_workspace_bytes(1, 2 * case.gamma + 1, case.V),
                     dtype=torch.uint8, device=DEV)
    outs = []
    for r in rounds:
        o = sv.spec_verify_chain(*(a[r:r + 1] for a in args), draft_is_probs=case.draft_is_probs,
                                 workspace=ws)
        outs.append([t.clone() for t in o])
    torch.cuda.synchronize()
    return [np.concatenate([o[k].cpu().numpy() for o in outs]) for k in range(4)]


def test_c1_single_round_calls(sv):
    """C1's 256 rounds, each as its own B = 1 call on one shared workspace."""
    case = W.c1_chain_fp32_v1000()
    toks, nacc, diag, st = _single_rounds(sv, case, range(case.B))
    args = case.numpy64()
    cmp = compare_chain(args, oracle.verify_chain(*args), toks, nacc, st, diag, prob_tol=1e-5)
    assert not cmp["failures"], cmp["failures"][:5]
    assert cmp["exact"] + len(cmp["boundary"]) == 256 and len(cmp["boundary"]) <= 2


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
def test_c2_single_round_calls(sv, T):
    """The first 64 of C2's rounds, each as its own B = 1 call."""
    case = W.c2_chain_bf16_v32000(T, rounds=64)
    toks, nacc, diag, st = _single_rounds(sv, case, range(case.B))
    args = case.numpy64()
    cmp = compare_chain(args, oracle.verify_chain(*args), toks, nacc, st, diag, prob_tol=1e-4)
    assert not cmp["failures"], cmp["failures"][:5]
    assert len(cmp["boundary"]) <= 2


def test_c3_chain_bf16_v128256_full(sv):
    case = W.c3_chain_bf16_v128256()
    cmp, ref, out = check_chain(sv, case)
    assert ref["greedy"].sum() == 8
    # all rows verified; the batch mixes rejections at every position
    assert len(set(out[1].tolist())) > 3


def test_c4_tree_f16_full(sv):
    ref = check_tree(sv, W.c4_tree_f16_v32000())
    assert ref["num_accepted"].max() >= 3


@pytest.mark.parametrize("B,N,dtype", [(13, 96, "f16"), (5, 200, "bf16"), (1, 1024, "f16")])
def test_trees_filling_the_grid(sv, B, N, dtype):
    """Tree calls whose stats grid would fill every SM launch a few stats CTAs
    fewer, so that the decide CTAs (one per tree) are resident from the start
    and merge each tree as its partials arrive.  An odd number of trees, a
    single tree of the largest size, and both 16-bit dtypes: bit-exact
    against the oracle."""
    case = W.make_tree(f"grid_trees_B{B}_N{N}", 7100 + B, B=B, N=N, V=32000, max_depth=8,
                       dtype=dtype, p_match=0.9)
    ref = check_tree(sv, case)
    assert ref["num_accepted"].max() >= 1


def test_c5_chain_probs_all_rows(sv, pool):
    """C5 in full: all 256 rows in one call (bf16 target, fp32 draft
    probabilities, forced all-accept rows drawing the bonus token)."""
    cmp, outs = check_full(sv, pool, W.c5_spec(), 16, 8, 1e-4)
    forced = np.arange(256) % 16 == 0
    assert np.all(cmp["num_accepted"][forced] == 4)
    assert (cmp["num_accepted"] == 4).sum() > forced.sum()   # natural all-accepts too


# ---------------------------------------------------------------------------
# Shapes: ragged tiles, unaligned rows, dtype pairs, gamma extremes
# ---------------------------------------------------------------------------

def _temps_mix(b, v):
    return [0.0, 0.01, 0.5, 1.0, 1.7, -1.0][b % 6] if b % 6 != 4 else 0.3 + v


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("V", [20000, 8193])
def test_chain_ragged_tiles(sv, dtype, V):
    case = W.make_chain("ragged", 3000 + V, B=12, gamma=5, V=V, dtype=dtype,
                        draft_sigma=(0.2, 2.0), temperature=_temps_mix)
    check_chain(sv, case)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chain_probs_mode_ragged(sv, dtype):
    case = W.make_chain("probs", 3100, B=16, gamma=4, V=20001, dtype=dtype,
                        draft_sigma=(0.5, 0.9), temperature=0.8, draft_probs=True,
                        force_accept_every=4)
    check_chain(sv, case)


@pytest.mark.parametrize("V", [1001, 7, 1, 3])
@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
def test_chain_unaligned_rows(sv, V, dtype):
    case = W.make_chain("unaligned", 3200 + V, B=9, gamma=3, V=V, dtype=dtype,
                        target="normal", target_sigma=2.0, draft_sigma=(0.5, 1.5),
                        temperature=_temps_mix)
    check_chain(sv, case)


def test_c3_shape_unaligned_rows_full(sv):
    """C3's shape with V = 128257: every bf16 row starts at an odd multiple
    of 2 bytes from the 16-byte grid, target and draft rows alike."""
    case = W.make_chain("c3_unaligned", 1003, 64, 7, 128257, "bf16", target="zipf",
                        draft_sigma=(0.3, 2.0), temperature=W._c3_temperature)
    cmp, ref, out = check_chain(sv, case)
    assert ref["greedy"].sum() == 8 and len(set(out[1].tolist())) > 3


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_tree_unaligned_rows(sv, dtype):
    check_tree(sv, W.make_tree(f"tree_odd_{dtype}", 4600, B=5, N=40, V=9001, max_depth=8,
                               kmin=1, kmax=3, dtype=dtype, p_match=0.9))


def test_chain_mixed_dtypes(sv):
    base = W.make_chain("mixed", 3300, B=10, gamma=4, V=9000, dtype="bf16",
                        draft_sigma=(0.3, 1.0), temperature=_temps_mix)
    for ddt in (torch.float32, torch.float16):
        case = W.ChainCase("mixed", base.target, base.draft.to(ddt), False, base.draft_tokens,
                           base.temperatures, base.uniforms, dict(dtype="bf16"))
        check_chain(sv, case)


@pytest.mark.parametrize("gamma", [1, 31])
def test_chain_gamma_extremes(sv, gamma):
    case = W.make_chain("gamma", 3400 + gamma, B=20, gamma=gamma, V=600, dtype="bf16",
                        draft_sigma=(0.05, 0.4), temperature=_temps_mix)
    check_chain(sv, case)


# ---------------------------------------------------------------------------
# Degenerate cases and data errors
# ---------------------------------------------------------------------------

def _chain_case(tl, dl, x, T, u, probs=False, dtype="f32"):
    dt = W.DTYPES[dtype]
    return W.ChainCase("edge", torch.tensor(tl, dtype=torch.float32).to(dt),
                       torch.tensor(dl, dtype=torch.float32).to(torch.float32 if probs else dt),
                       probs, torch.tensor(x, dtype=torch.int32),
                       torch.tensor(T, dtype=torch.float32), torch.tensor(u, dtype=torch.float32),
                       dict(dtype=dtype))


def test_chain_edge_cases(sv):
    rng = np.random.default_rng(5)
    B, g, V = 12, 3, 40
    tl = rng.normal(size=(B, g + 1, V)) * 2
    dl = tl[:, :g] + rng.normal(size=(B, g, V))
    x = rng.integers(0, V, size=(B, g))
    T = np.ones(B)
    u = rng.random((B, g + 1))
    x[0, 1] = V                      # token out of range
    x[1, 0] = -1
    tl[2, 1, 5] = np.nan             # NaN in a softmax row
    tl[3, 3, :] = -np.inf            # an all -inf bonus row
    T[4] = np.nan                    # bad temperatures
    T[5] = 1e-30
    T[6] = 0.0
    tl[6, 0, 3] = np.nan             # NaN in a greedy row
    T[7] = 0.0
    dl[7, :, :] = np.nan             # draft rows of a greedy row are never read
    tl[8, :, 10:] = -np.inf          # -inf logits: p = 0 there
    dl[8, :, :20] = -np.inf          # q = 0 on [0, 20)
    x[8] = [5, 25, 3]                # q(5) = 0 < p(5): accept; 25: p = 0 -> reject
    u[8, :g] = 0.5
    tl[9, 0, :] = 1.0                # flat target row
    dl[9, 0, :] = 1.0                # identical draft row -> ratio 1 -> accept
    u[10, :g] = 0.0                  # forced accept: bonus draw from p_gamma
    tl[11, 0] = np.where(np.arange(V) == 7, -np.inf, tl[11, 0])
    dl[11, 0] = tl[11, 0]            # p = q with p(x) = q(x) = 0 at x = 7
    x[11, 0] = 7                     # -> reject, zero residual mass -> draw from p_0
    case = _chain_case(tl, dl, x, T, u)
    cmp, ref, out = check_chain(sv, case, max_boundary=0)
    st = out[3]
    assert st[0] & 1 and st[1] & 1 and st[2] & 2 and st[3] & 2
    assert st[4] & 16 and st[5] & 16 and st[6] & 2 and st[7] == 0
    assert out[1][8] == 1 and out[1][9] >= 1 and out[1][10] == g and out[1][11] == 0


def test_chain_probs_mode_errors(sv):
    rng = np.random.default_rng(6)
    B, g, V = 4, 2, 50
    tl = rng.normal(size=(B, g + 1, V))
    q = special.softmax(rng.normal(size=(B, g, V)), axis=-1)
    x = np.array([[1, 2]] * B)
    u = np.full((B, g + 1), 0.4)
    q[0, 1, 2] = np.nan              # q(x) NaN -> error
    q[1, 1, 30] = np.nan             # never read when row 1 accepts all
    u[1, :g] = 0.0
    q[2, 0, 40] = np.nan             # read by the residual sweep after a rejection
    u[2, 0] = 0.999999
    q[2, 0, 1] = 1.0
    case = _chain_case(tl, q, x, np.full(B, 0.9), u, probs=True)
    cmp, ref, out = check_chain(sv, case, max_boundary=0)
    assert out[3][0] & 2 and out[3][1] == 0 and out[3][2] & 2


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_argmax_ties_across_tiles(sv, dtype):
    """Exact ties (and -0 / +0) spread over several tiles: lowest index wins."""
    rng = np.random.default_rng(7)
    B, g, V = 6, 3, 30000
    tl = rng.integers(-4, 3, size=(B, g + 1, V)).astype(np.float32)
    tl[0, 0, :] = -0.0
    tl[0, 0, 20000] = 0.0
    tl[1, 1, [9000, 17000, 25000]] = 9.0
    tl[2, 2, :] = -np.inf
    x = np.zeros((B, g), np.int64)
    x[0, 0] = 0
    x[1] = [int(np.argmax(tl[1, 0])), 9000, 3]
    x[3] = [int(np.argmax(tl[3, i])) for i in range(g)]
    case = _chain_case(tl, np.zeros((B, g, V)), x, np.zeros(B), np.zeros((B, g + 1)),
                       dtype=dtype)
    check_chain(sv, case, max_boundary=0)
    tg = sv.spec_verify_chain_greedy(case.target.to(DEV), case.draft_tokens.to(DEV))
    ref = oracle.verify_chain_greedy(W.to_f64(case.target), case.draft_tokens.numpy())
    assert np.array_equal(tg[0].cpu().numpy(), ref["tokens"])
    assert np.array_equal(tg[1].cpu().numpy(), ref["num_accepted"])


def test_greedy_entry_matches_chain_at_T0(sv):
    case = W.make_chain("greedy", 3500, B=40, gamma=6, V=12345, dtype="bf16",
                        draft_sigma=(0.0, 0.3), temperature=0.0)
    toks, nacc, diag, st = run_chain(sv, case)
    g_t, g_n, g_s = sv.spec_verify_chain_greedy(case.target.to(DEV), case.draft_tokens.to(DEV))
    ref = oracle.verify_chain_greedy(W.to_f64(case.target), case.draft_tokens.numpy())
    assert np.array_equal(g_t.cpu().numpy(), ref["tokens"]) and np.array_equal(toks, ref["tokens"])
    assert np.array_equal(g_n.cpu().numpy(), ref["num_accepted"])
    assert np.all(g_s.cpu().numpy() == 0)
    assert ref["num_accepted"].max() > 0


def test_greedy_worked_example_through_abi(sv):
    import json
    import os
    gdn = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                      "sd_intro_greedy_example.json")))
    words = sorted(set(gdn["draft"]) | set(gdn["target_choice"]))
    vocab = {w: i for i, w in enumerate(words)}
    V, gamma = 8, len(gdn["draft"])
    tl = np.random.default_rng(8).normal(size=(1, gamma + 1, V))
    for i, w in enumerate(gdn["target_choice"]):
        tl[0, i, vocab[w]] = tl[0, i].max() + 1.0
    x = torch.tensor([[vocab[w] for w in gdn["draft"]]], dtype=torch.int32, device=DEV)
    t, n, s = sv.spec_verify_chain_greedy(torch.tensor(tl, dtype=torch.float32, device=DEV), x)
    inv = {i: w for w, i in vocab.items()}
    got = [inv[int(v)] for v in t[0].cpu().tolist() if v >= 0]
    assert got == gdn["committed"] and int(n[0]) == gdn["accepted"]


# ---------------------------------------------------------------------------
# Trees
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kmax,p_match,D", [(2, 1.0, 8), (4, 0.8, 8), (3, 1.0, 2), (2, 1.0, 0)])
def test_tree_variants(sv, kmax, p_match, D):
    case = W.make_tree("tree", 4000 + kmax * 10 + D, B=12, N=64, V=9001, max_depth=max(D, 1),
                       kmin=1, kmax=kmax, p_match=p_match)
    case.max_depth = D
    check_tree(sv, case)


def test_tree_large_and_single_node(sv):
    check_tree(sv, W.make_tree("big", 4100, B=3, N=1024, V=700, max_depth=31, kmin=1, kmax=2,
                               p_match=1.0))
    check_tree(sv, W.make_tree("one", 4101, B=4, N=1, V=300, max_depth=5))


def test_tree_errors_and_duplicate_siblings(sv):
    case = W.make_tree("err", 4200, B=5, N=20, V=500, max_depth=8, p_match=1.0)
    par = case.parent.clone()
    tok = case.node_tokens.clone()
    par[0, 0] = 0                    # root must have parent -1
    par[1, 5] = 7                    # parent after child
    tok[2, 3] = 500                  # token out of range
    lg = case.node_logits.clone()
    lg[3, 2, 17] = float("nan")      # NaN node row
    # tree 4: two children of the root carry the root's argmax -> lowest index
    a0 = int(torch.argmax(lg[4, 0].float()))
    kids = (par[4] == 0).nonzero().flatten().tolist()
    if len(kids) >= 2:
        tok[4, kids[0]] = a0
        tok[4, kids[1]] = a0
    bad = W.TreeCase("err", lg, par, tok, 8)
    ref = check_tree(sv, bad)
    assert ref["status"][0] & 4 and ref["status"][1] & 4 and ref["status"][2] & 1
    assert ref["status"][3] & 2 and ref["status"][4] == 0


# ---------------------------------------------------------------------------
# Workspace reuse and determinism
# ---------------------------------------------------------------------------

def test_workspace_reuse_across_entry_points(sv):
    chain = W.make_chain("ws", 4300, B=8, gamma=4, V=17000, dtype="bf16",
                         temperature=_temps_mix)
    tree = W.make_tree("ws", 4301, B=4, N=32, V=17000)
    nb = max(sv.spec_verify_workspace_bytes(8, 9, 17000),
             sv.spec_verify_workspace_bytes(4, 32, 17000))
    ws = torch.full((nb,), 0xAB, dtype=torch.uint8, device=DEV)   # no initialisation needed
    c_args = [t.to(DEV) for t in (chain.target, chain.draft, chain.draft_tokens,
                                  chain.temperatures, chain.uniforms)]
    t_args = [t.to(DEV) for t in (tree.node_logits, tree.parent, tree.node_tokens)]
    first = None
    for _ in range(4):
        a = [o.cpu().clone() for o in sv.spec_verify_chain(*c_args, workspace=ws)]
        b = [o.cpu().clone() for o in sv.spec_verify_tree_greedy(*t_args, 8, workspace=ws)]
        c = [o.cpu().clone() for o in sv.spec_verify_chain_greedy(c_args[0], c_args[2],
                                                                   workspace=ws)]
        if first is None:
            first = (a, b, c)
        else:
            for x, y in zip(first[0] + first[1] + first[2], a + b + c):
                assert torch.equal(x, y)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) > 0                        # partials were written


# ---------------------------------------------------------------------------
# Statistics on the GPU (the pages' theorems)
# ---------------------------------------------------------------------------

def test_gpu_theorem1_chi_square(sv):
    """Emitted tokens, slot by slot, follow p (10^6 rounds, V = 8)."""
    rng = np.random.default_rng(9)
    n, V, g, T = 1_000_000, 8, 3, 0.9
    tl = rng.normal(size=(g + 1, V)) * 1.5
    dl = tl[:g] + rng.normal(size=(g, V)) * 1.2
    q = special.softmax(dl / T, axis=-1)
    x = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(g)], axis=1)
    tgt = torch.tensor(tl, dtype=torch.float32, device=DEV).expand(n, g + 1, V).contiguous()
    dft = torch.tensor(dl, dtype=torch.float32, device=DEV).expand(n, g, V).contiguous()
    u = torch.rand((n, g + 1), generator=torch.Generator().manual_seed(3)).to(DEV)
    toks, nacc, _, st = sv.spec_verify_chain(tgt, dft, torch.tensor(x, dtype=torch.int32,
                                                                     device=DEV),
                                             torch.full((n,), T, device=DEV), u,
                                             want_diag=False)
    toks, nacc = toks.cpu().numpy(), nacc.cpu().numpy()
    assert np.all(st.cpu().numpy() == 0)
    for i in range(g + 1):
        p = special.softmax(tl[i] / T)
        reached = nacc >= i
        obs = np.bincount(toks[reached, i], minlength=V)
        assert stats.chisquare(obs, p * reached.sum()).pvalue > 1e-3, i
    alpha0 = np.minimum(special.softmax(tl[0] / T), q[0]).sum()
    acc0 = (nacc >= 1).mean()
    assert abs(acc0 - alpha0) < 5 * np.sqrt(alpha0 * (1 - alpha0) / n)


def test_gpu_expected_tokens_constant_alpha(sv):
    """Mean tokens per round = (1 - a^(g+1)) / (1 - a) at constant alpha."""
    rng = np.random.default_rng(10)
    n, V, g, alpha = 1_000_000, 8, 4, 0.75
    tl = np.full((g + 1, V), -np.inf)
    tl[:, :4] = rng.normal(size=(g + 1, 4))
    q = np.zeros((g, V))
    for i in range(g):
        s = np.zeros(V)
        s[4:] = rng.random(4) + 0.1
        q[i] = alpha * special.softmax(tl[i]) + (1 - alpha) * s / s.sum()
    x = np.stack([rng.choice(V, size=n, p=q[i] / q[i].sum()) for i in range(g)], axis=1)
    tgt = torch.tensor(tl, dtype=torch.float32, device=DEV).expand(n, g + 1, V).contiguous()
    dft = torch.tensor(q, dtype=torch.float32, device=DEV).expand(n, g, V).contiguous()
    u = torch.rand((n, g + 1), generator=torch.Generator().manual_seed(4)).to(DEV)
    toks, nacc, _, st = sv.spec_verify_chain(tgt, dft, torch.tensor(x, dtype=torch.int32,
                                                                     device=DEV),
                                             torch.ones(n, device=DEV), u, draft_is_probs=True,
                                             want_diag=False)
    emitted = nacc.cpu().numpy() + 1
    want = (1 - alpha ** (g + 1)) / (1 - alpha)
    assert abs(emitted.mean() - want) < 4 * emitted.std() / np.sqrt(n)


@pytest.mark.parametrize("V,N,B,dtype,D", [(704, 1024, 3, "f16", 31), (70000, 40, 2, "f16", 8),
                                           (20000, 64, 5, "f32", 8), (32000, 64, 6, "bf16", 6)])
def test_tree_aligned_rows(sv, V, N, B, dtype, D):
    """Rows on 16-byte boundaries take the streaming pair: node-row merges of
    at most 32 chunks (grouped per warp) and of more (V = 70000 fp16)."""
    check_tree(sv, W.make_tree(f"tree_al_{V}", 4300 + V % 97, B=B, N=N, V=V, max_depth=D,
                               kmin=1, kmax=3, dtype=dtype, p_match=0.9))


def test_tree_errors_aligned_rows(sv):
    case = W.make_tree("err_al", 4400, B=4, N=48, V=4096, max_depth=8, p_match=1.0)
    par = case.parent.clone()
    tok = case.node_tokens.clone()
    lg = case.node_logits.clone()
    par[0, 9] = 30                   # parent after child
    tok[1, 4] = -2                   # token out of range
    lg[2, 40, 1000] = float("nan")   # NaN node row
    lg[3, 7, :] = float("-inf")      # an all -inf node row: argmax at index 0
    ref = check_tree(sv, W.TreeCase("err_al", lg, par, tok, 8))
    assert ref["status"][0] & 4 and ref["status"][1] & 1 and ref["status"][2] & 2


def test_chain_maximum_vocabulary(sv):
    """V = 2^26, the library's limit: 32768 stats chunks and 65536 residual
    chunks per bf16 row, so the long-row merge and the streamed crossing
    search run.  Row 0 drafts the draft row's top token; row 1 drafts a token
    far down the target's order, a rejection with a residual draw over all
    2^26 entries.  Draft tokens are chosen here (a categorical draw over 2^26
    entries is beyond the input generator's sampler)."""
    V = 1 << 26
    g = torch.Generator().manual_seed(2026)
    bias = W.zipf_bias(2026, V)
    tgt = (torch.randn((2, 2, V), generator=g) + bias).to(torch.bfloat16)
    dft = (tgt[:, :1].float() + 0.5 * torch.randn((2, 1, V), generator=g)).to(torch.bfloat16)
    toks = torch.empty((2, 1), dtype=torch.int32)
    toks[0, 0] = int(torch.argmax(dft[0, 0].float()))
    toks[1, 0] = int(torch.argmin(tgt[1, 0].float() - dft[1, 0].float()))
    case = W.ChainCase("max_vocab", tgt, dft, False, toks,
                       torch.tensor([0.9, 1.1], dtype=torch.float32),
                       torch.tensor([[0.3, 0.77], [0.999, 0.41]], dtype=torch.float32))
    cmp, ref, _ = check_chain(sv, case)
    assert ref["num_accepted"][1] == 0           # the far-down draft is rejected


def test_chain_large_batch(sv):
    """4096 batch rows of short aligned rows: one decide CTA per row, a
    decide grid far larger than one wave, every row checked."""
    case = W.make_chain("large_batch", 4500, B=4096, gamma=3, V=1024, dtype="bf16",
                        draft_sigma=(0.2, 2.0),
                        temperature=lambda b, v: 0.0 if b % 5 == 0 else 0.3 + 1.2 * v)
    cmp, ref, _ = check_chain(sv, case)
    assert len(set(ref["num_accepted"].tolist())) == 4
