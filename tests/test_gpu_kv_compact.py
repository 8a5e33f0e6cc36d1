"""GPU parity of the KV-cache compaction (spec_tree_kv_compact through the C
ABI) against the oracle: the whole cache, new lengths and row status
bit-exact, on paths walked by the GPU tree verifier and by the oracle."""

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


def _random_kv(B, S, E, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-30000, 30000, (B, S, E), generator=g, dtype=torch.int32).to(dtype) \
        if dtype != torch.int32 else torch.randint(-2**31, 2**31 - 1, (B, S, E), generator=g,
                                                   dtype=torch.int32)


def _check(sv, kv, base, path, nacc):
    ref = oracle.tree_kv_compact(kv.view(torch.int16 if kv.element_size() == 2 else kv.dtype)
                                 .numpy(), base, path, nacc)
    g = kv.to(DEV)
    length, st = sv.spec_tree_kv_compact(
        g, torch.as_tensor(base, dtype=torch.int32).to(DEV),
        torch.as_tensor(path, dtype=torch.int32).to(DEV),
        torch.as_tensor(nacc, dtype=torch.int32).to(DEV))
    torch.cuda.synchronize()
    got = g.cpu()
    got = got.view(torch.int16 if got.element_size() == 2 else got.dtype).numpy()
    assert np.array_equal(st.cpu().numpy(), ref["status"])
    assert np.array_equal(length.cpu().numpy(), ref["length"])
    assert np.array_equal(got, ref["kv"])
    return ref


def test_kv_compact_after_gpu_tree_walk(sv):
    """The paths come from spec_verify_tree_greedy on the GPU (its own parity
    against the oracle is tested elsewhere); the compaction of a 4 KB-row
    bf16 cache matches the oracle's on those paths."""
    tree = W.c4_tree_f16_v32000()
    B, N = tree.parent.shape
    path, _, nacc, st = sv.spec_verify_tree_greedy(
        tree.node_logits.to(DEV), tree.parent.to(DEV), tree.node_tokens.to(DEV), tree.max_depth)
    torch.cuda.synchronize()
    assert not st.cpu().numpy().any()
    walk = oracle.verify_tree_greedy(*tree.numpy64())
    assert np.array_equal(nacc.cpu().numpy(), walk["num_accepted"])
    S = 64 + N
    base = np.arange(B) % 7 * 3 + 17
    kv = _random_kv(B, S, 2048, torch.bfloat16, 1)
    ref = _check(sv, kv, base, path.cpu().numpy(), nacc.cpu().numpy())
    assert (ref["length"] - base).max() >= 2


@pytest.mark.parametrize("E,dtype", [(4, torch.int32), (8, torch.float16), (264, torch.int32),
                                     (1032, torch.bfloat16), (5000, torch.int32)])
def test_kv_compact_ragged_rows(sv, E, dtype):
    """Row sizes of one 16-byte unit, within one 1 KB tile, and several tiles
    with a ragged last tile; paths from the oracle's walk of random trees."""
    tree = W.make_tree(f"kv_{E}", 60 + E, B=6, N=40, V=50, max_depth=8)
    walk = oracle.verify_tree_greedy(*tree.numpy64())
    S = 50
    base = np.array([0, 1, 5, 9, 10, 2])
    kv = _random_kv(6, S, E, dtype, E)
    _check(sv, kv, base, walk["path"], walk["num_accepted"])


def test_kv_compact_full_depth_and_bad_paths(sv):
    """A fully accepted 31-deep chain (the widest path), the identity case,
    d = 0, and each kind of bad path (which must leave its tree untouched)."""
    W_ = 32
    S = 64
    B = 8
    path = np.full((B, W_), -1)
    nacc = np.zeros(B, int)
    base = np.full(B, 3)
    path[0, :31] = np.arange(1, 32) + np.r_[np.zeros(16, int), np.ones(15, int)]  # one gap
    nacc[0] = 31
    path[1, :31] = np.arange(1, 32)             # identity
    nacc[1] = 31
    nacc[2] = 0                                 # nothing accepted
    path[3, :3] = [2, 2, 5]                     # not increasing
    nacc[3] = 3
    path[4, :2] = [0, 4]                        # below i + 1
    nacc[4] = 2
    path[5, :2] = [1, 62]                       # slot 3 + 62 - 1 >= S
    nacc[5] = 2
    nacc[6] = 33                                # d above the path width
    base[7] = -1                                # negative base
    path[7, :1] = [1]
    nacc[7] = 1
    kv = _random_kv(B, S, 12, torch.int32, 7)
    ref = _check(sv, kv, base, path, nacc)
    assert list(ref["status"]) == [0, 0, 0] + [oracle.ROW_BAD_TREE] * 5
    assert ref["length"][0] == 34


def test_kv_compact_many_trees(sv):
    """4096 trees of a 64-slot cache with 1 KB rows, random valid paths
    (distinct sorted node ids, so entry i is at least i + 1)."""
    rng = np.random.default_rng(9)
    B, S, Wp = 4096, 64, 8
    base = rng.integers(0, 17, B)
    nacc = rng.integers(0, Wp + 1, B)
    path = np.full((B, Wp), -1)
    for b in range(B):
        path[b, :nacc[b]] = np.sort(rng.choice(np.arange(1, 48), size=nacc[b], replace=False))
    kv = _random_kv(B, S, 256, torch.int32, 11)
    ref = _check(sv, kv, base, path, nacc)
    assert not ref["status"].any()


def test_kv_compact_rejects_misaligned_rows(sv):
    kv = torch.zeros((2, 8, 3), dtype=torch.int32, device=DEV)     # 12-byte rows
    z = torch.zeros(2, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_tree_kv_compact(kv, z, torch.zeros((2, 4), dtype=torch.int32, device=DEV), z)
