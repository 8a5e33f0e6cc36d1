"""GPU parity of the token-tree ancestor mask (spec_tree_mask through the C
ABI) against the oracle: mask bits, depths and row status bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_48_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as pkg
    pkg.lib()
    return pkg


def _bits(words, N):
    """[B, N, W] int64 words -> bool [B, N, N] (bit m % 64 of word m / 64)."""
    w = words.astype(np.uint64)
    B, n, Wd = w.shape
    out = np.zeros((B, n, Wd * 64), bool)
    for k in range(Wd):
        for bit in range(64):
            out[:, :, k * 64 + bit] = (w[:, :, k] >> np.uint64(bit)) & np.uint64(1)
    return out[:, :, :N]


def _check(sv, parent):
    mask, depth, st = sv.spec_tree_mask(torch.as_tensor(parent, dtype=torch.int32).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.tree_ancestor_mask(parent)
    N = parent.shape[1]
    assert np.array_equal(st.cpu().numpy(), ref["status"])
    assert np.array_equal(depth.cpu().numpy(), ref["depth"])
    assert np.array_equal(_bits(mask.cpu().numpy(), N), ref["mask"])
    return ref


def test_tree_mask_token_trees(sv):
    tree = W.c4_tree_f16_v32000()
    ref = _check(sv, tree.parent.numpy())
    assert ref["depth"].max() >= 3


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 129, 1000, 1024])
def test_tree_mask_random_trees(sv, N):
    rng = np.random.default_rng(40 + N)
    par = np.stack([np.array([-1] + [int(rng.integers(max(0, n - 5), n)) for n in range(1, N)])
                    for _ in range(3)])
    _check(sv, par)


def test_tree_mask_chain_star_and_bad_trees(sv):
    N = 1024
    chain = np.array([-1] + list(range(N - 1)))
    star = np.array([-1] + [0] * (N - 1))
    bad1 = chain.copy()
    bad1[700] = 900                       # parent after the child
    bad2 = star.copy()
    bad2[0] = 3                           # root with a parent
    ref = _check(sv, np.stack([chain, star, bad1, bad2]))
    assert ref["depth"][0, -1] == N - 1
    assert list(ref["status"][2:]) == [oracle.ROW_BAD_TREE] * 2
