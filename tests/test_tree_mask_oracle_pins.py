"""Pins for the oracle's tree attention mask (CPU only).

The mask is checked against the transitive closure of the parent relation
computed with boolean matrix powers (numpy matmul, independent of the
oracle's parent walk), against closed forms for chains and stars, and against
its own invariants (depth = set bits - 1, a row contains its parent's row).
"""

import numpy as np

import oracle
from speculative_decoding_verification_48_gb300 import workloads as W


def _closure(par):
    """I + A + A^2 + ... with A[n, parent[n]] = 1, by repeated squaring."""
    N = len(par)
    A = np.zeros((N, N), np.int64)
    for n in range(1, N):
        A[n, par[n]] = 1
    R = np.eye(N, dtype=np.int64) + A
    for _ in range(int(np.ceil(np.log2(max(N, 2)))) + 1):
        R = np.minimum(R @ R, 1)
    return R.astype(bool)


def test_mask_is_the_transitive_closure_of_the_parent_relation():
    rng = np.random.default_rng(31)
    for _ in range(40):
        N = int(rng.integers(1, 60))
        par = np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)])
        r = oracle.tree_ancestor_mask(par[None])
        assert np.array_equal(r["mask"][0], _closure(par))
        assert np.array_equal(r["depth"][0], r["mask"][0].sum(axis=1) - 1)
        for n in range(1, N):
            assert np.all(r["mask"][0, n] >= r["mask"][0, par[n]])


def test_mask_closed_forms_chain_and_star():
    N = 17
    chain = np.array([-1] + list(range(N - 1)))
    r = oracle.tree_ancestor_mask(chain[None])
    assert np.array_equal(r["mask"][0], np.tril(np.ones((N, N), bool)))
    assert np.array_equal(r["depth"][0], np.arange(N))
    star = np.array([-1] + [0] * (N - 1))
    r = oracle.tree_ancestor_mask(star[None])
    want = np.eye(N, dtype=bool)
    want[:, 0] = True
    assert np.array_equal(r["mask"][0], want)


def test_mask_of_the_token_trees_and_bad_trees():
    tree = W.make_tree("mask_pin", 32, B=3, N=40, V=50, max_depth=6)
    par = tree.parent.numpy().copy()
    r = oracle.tree_ancestor_mask(par)
    assert not r["status"].any() and r["depth"].max() <= 6
    par[1, 5] = 7                                 # a parent after its child
    par[2, 0] = 0                                 # a root with a parent
    r = oracle.tree_ancestor_mask(par)
    assert list(r["status"]) == [0, oracle.ROW_BAD_TREE, oracle.ROW_BAD_TREE]
    assert not r["mask"][1:].any()
