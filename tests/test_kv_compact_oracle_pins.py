"""Pins for the oracle's KV-cache compaction after tree verification (CPU).

Checked against rows tagged with their own slot number (so every moved row
names where it came from), the identity case of a fully accepted chain tree,
brute-force path enumeration on real token trees, and the bad-path flags.
"""

import numpy as np

import oracle
from speculative_decoding_verification_48_gb300 import workloads as W


def _tagged(B, S, E):
    kv = np.zeros((B, S, E), np.int32)
    for b in range(B):
        for s in range(S):
            kv[b, s] = 1000 * b + s            # every element names its slot
    return kv


def test_rows_move_from_node_slots_to_contiguous_slots():
    kv = _tagged(2, 40, 3)
    base = np.array([10, 5])
    path = np.array([[2, 5, 9, -1], [1, 4, -1, -1]])
    r = oracle.tree_kv_compact(kv, base, path, np.array([3, 2]))
    assert list(r["length"]) == [13, 7] and not r["status"].any()
    assert list(r["kv"][0, 10:13, 0]) == [11, 14, 18]      # slots base + path - 1
    assert list(r["kv"][1, 5:7, 0]) == [1005, 1008]
    untouched = np.ones((2, 40), bool)
    untouched[0, 10:13] = False
    untouched[1, 5:7] = False
    assert np.array_equal(r["kv"][:, :, 0][untouched], kv[:, :, 0][untouched])


def test_fully_accepted_chain_tree_is_the_identity():
    kv = _tagged(1, 20, 2)
    path = np.array([[1, 2, 3, 4, 5]])
    r = oracle.tree_kv_compact(kv, np.array([4]), path, np.array([5]))
    assert np.array_equal(r["kv"], kv) and r["length"][0] == 9


def test_compaction_of_walked_token_trees():
    tree = W.make_tree("kv_pin", 33, B=4, N=30, V=40, max_depth=5)
    walk = oracle.verify_tree_greedy(*tree.numpy64())
    kv = _tagged(4, 64, 2)
    base = np.array([3, 0, 10, 20])
    r = oracle.tree_kv_compact(kv, base, walk["path"], walk["num_accepted"])
    par = tree.parent.numpy()
    for b in range(4):
        d = walk["num_accepted"][b]
        moved = r["kv"][b, base[b]:base[b] + d, 0] - 1000 * b - base[b] + 1
        assert list(moved) == list(walk["path"][b, :d])
        node = 0                                     # the moved nodes form a root path
        for n in moved:
            assert par[b, n] == node
            node = n


def test_bad_paths_move_nothing():
    kv = _tagged(4, 16, 1)
    path = np.array([[2, 2, -1], [0, 3, -1], [1, 20, -1], [1, 2, 3]])
    r = oracle.tree_kv_compact(kv, np.array([1, 1, 1, 1]), path, np.array([2, 1, 2, 4]))
    assert list(r["status"]) == [oracle.ROW_BAD_TREE] * 4
    assert np.array_equal(r["kv"], kv) and list(r["length"]) == [1, 1, 1, 1]
