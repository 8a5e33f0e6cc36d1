"""Both execution paths on the same small shapes.

Small calls run on the cluster path (one launch, a thread-block cluster per
batch row or tree); the diagnostics switch spec_verify_force_stream_path
sends them through the two-launch streaming path instead.  Each case here
runs on both paths against the float64 oracle, and the two paths' greedy and
tree outputs must agree bit for bit.
"""

import numpy as np
import pytest
import torch

import test_gpu_parity as TP
from speculative_decoding_verification_48_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = TP.DEV


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as pkg
    pkg.lib()
    return pkg


@pytest.fixture(params=["cluster", "stream"])
def svp(sv, request):
    prev = sv.spec_verify_force_stream_path(request.param == "stream")
    yield sv
    sv.spec_verify_force_stream_path(prev)


def test_edge_cases(svp):
    TP.test_chain_edge_cases(svp)


def test_probs_mode_errors(svp):
    TP.test_chain_probs_mode_errors(svp)


def test_mixed_dtypes(svp):
    TP.test_chain_mixed_dtypes(svp)


@pytest.mark.parametrize("tdt,ddt", [("bf16", torch.float32), ("f32", torch.bfloat16),
                                     ("bf16", torch.float16)])
def test_mixed_dtypes_rows_off_grid(svp, tdt, ddt):
    """Target and draft rows of different widths and odd V, so that the
    rows start at shifting offsets from the 16-byte grid: on the streaming
    path the draft row's vectors are rebuilt from aligned blocks of its own
    grid (16- and 8-byte vectors)."""
    base = W.make_chain(f"mixed_odd_{tdt}", 3400, B=9, gamma=4, V=9001, dtype=tdt,
                        draft_sigma=(0.3, 1.0), temperature=TP._temps_mix)
    case = W.ChainCase("mixed_odd", base.target, base.draft.to(ddt), False, base.draft_tokens,
                       base.temperatures, base.uniforms, dict(dtype="bf16"))
    TP.check_chain(svp, case)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_ragged_odd_vocabulary(svp, dtype):
    TP.test_chain_ragged_tiles(svp, dtype, 8193)


@pytest.mark.parametrize("gamma", [1, 31])
def test_gamma_extremes(svp, gamma):
    TP.test_chain_gamma_extremes(svp, gamma)


@pytest.mark.parametrize("dtype,V", [("bf16", 1001), ("f32", 7), ("f16", 3), ("f32", 1)])
def test_unaligned_rows(svp, dtype, V):
    TP.test_chain_unaligned_rows(svp, V, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_argmax_ties(svp, dtype):
    TP.test_argmax_ties_across_tiles(svp, dtype)


def test_greedy_entry(svp):
    TP.test_greedy_entry_matches_chain_at_T0(svp)


def test_c1_rounds(svp):
    TP.test_c1_single_round_calls(svp)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_c2_rounds(svp, T):
    TP.test_c2_single_round_calls(svp, T)


@pytest.mark.parametrize("kmax,p_match,D", [(2, 1.0, 8), (4, 0.8, 8), (2, 1.0, 0)])
def test_tree_variants(svp, kmax, p_match, D):
    TP.test_tree_variants(svp, kmax, p_match, D)


def test_tree_errors(svp):
    TP.test_tree_errors_and_duplicate_siblings(svp)


def test_c4_trees(svp):
    TP.test_c4_tree_f16_full(svp)


def test_paths_agree_on_greedy_and_trees(sv):
    """Greedy chains and tree walks are deterministic: both paths give the
    same bits."""
    chain = W.make_chain("paths_greedy", 9100, B=6, gamma=6, V=30001, dtype="bf16",
                         temperature=0.0)
    tree = W.make_tree("paths_tree", 9101, B=4, N=48, V=24000, max_depth=8, kmin=1, kmax=3,
                       dtype="f16", p_match=0.9)
    outs = []
    for force in (False, True):
        prev = sv.spec_verify_force_stream_path(force)
        try:
            outs.append((TP.run_chain(sv, chain)[:2], TP.run_tree(sv, tree)))
        finally:
            sv.spec_verify_force_stream_path(prev)
    (c0, t0), (c1, t1) = outs
    for a, b in zip(c0, c1):
        assert np.array_equal(a, b)
    for a, b in zip(t0, t1):
        assert np.array_equal(a, b)
