"""The C ABI without a GPU: the library loads, exports every declared entry
point, sizes workspaces, and rejects bad arguments before any CUDA call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    from speculative_decoding_verification_48_gb300 import binding
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SV_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("spec_verify_chain", "spec_verify_chain_greedy", "spec_verify_tree_greedy",
              "spec_verify_workspace_bytes", "spec_verify_status_string", "spec_draft_sample",
              "spec_tree_mask", "spec_tree_kv_compact", "spec_verify_chain_no_alloc",
              "spec_verify_wait_selftest", "spec_verify_set_call_counter",
              "spec_verify_force_stream_path"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_no_torch_types_in_header():
    text = open(HEADER).read()
    assert "torch" not in text.lower() and "at::" not in text and "Tensor" not in text


def test_status_strings(L):
    from speculative_decoding_verification_48_gb300 import binding
    for s in range(5):
        assert binding.spec_verify_status_string(s).startswith("SV_")
    assert "unknown" in binding.spec_verify_status_string(99)


def test_workspace_bytes(L):
    from speculative_decoding_verification_48_gb300 import binding as bd
    assert bd.spec_verify_workspace_bytes(0, 3, 10) == 0
    assert bd.spec_verify_workspace_bytes(1, 0, 10) == 0
    assert bd.spec_verify_workspace_bytes(1, 1, 0) == 0
    a = bd.spec_verify_workspace_bytes(64, 15, 128256)
    b = bd.spec_verify_workspace_bytes(64, 15, 128257 + 8192)
    c = bd.spec_verify_workspace_bytes(128, 15, 128256)
    assert 0 < a < b and a < c
    assert a % 256 == 0


FAKE = 1 << 20   # never dereferenced: every call below fails host validation


def _chain(L, **kw):
    args = dict(target=FAKE, tdt=1, draft=FAKE, ddt=1, probs=0, toks=FAKE, temps=FAKE,
                unif=FAKE, B=4, gamma=3, V=100, otok=FAKE, onacc=FAKE, odiag=None,
                ostat=None, ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    return L.spec_verify_chain(*args.values())


def test_chain_rejects_bad_arguments(L):
    INVALID, UNSUPPORTED = 1, 2
    assert _chain(L, target=None) == INVALID
    assert _chain(L, draft=None) == INVALID
    assert _chain(L, toks=None) == INVALID
    assert _chain(L, temps=None) == INVALID
    assert _chain(L, unif=None) == INVALID
    assert _chain(L, otok=None) == INVALID
    assert _chain(L, onacc=None) == INVALID
    assert _chain(L, ws=None) == INVALID
    assert _chain(L, B=0) == INVALID
    assert _chain(L, gamma=0) == INVALID
    assert _chain(L, gamma=32) == INVALID
    assert _chain(L, V=0) == INVALID
    assert _chain(L, V=(1 << 26) + 1) == INVALID
    assert _chain(L, tdt=7) == INVALID
    assert _chain(L, ddt=-1) == INVALID
    assert _chain(L, probs=1, ddt=1) == UNSUPPORTED
    assert _chain(L, wsb=16) == INVALID
    assert _chain(L, ws=FAKE + 4) == INVALID
    assert _chain(L, target=FAKE + 1) == INVALID      # misaligned bf16 logits
    assert _chain(L, toks=FAKE + 2) == INVALID
    assert _chain(L, odiag=FAKE + 4) == INVALID       # diag needs 16-byte alignment


def test_greedy_and_tree_reject_bad_arguments(L):
    INVALID = 1
    g = L.spec_verify_chain_greedy
    assert g(None, 1, FAKE, 2, 3, 50, FAKE, FAKE, None, FAKE, 1 << 30, None) == INVALID
    assert g(FAKE, 1, FAKE, 2, 40, 50, FAKE, FAKE, None, FAKE, 1 << 30, None) == INVALID
    assert g(FAKE, 1, FAKE, 2, 3, 50, FAKE, FAKE, None, FAKE, 8, None) == INVALID
    t = L.spec_verify_tree_greedy
    ok = [FAKE, 2, FAKE, FAKE, 2, 16, 100, 4, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return t(*a)
    assert call(a0=None) == INVALID
    assert call(a2=None) == INVALID
    assert call(a5=0) == INVALID          # N
    assert call(a5=1025) == INVALID
    assert call(a7=-1) == INVALID         # max_depth
    assert call(a7=32) == INVALID
    assert call(a13=16) == INVALID        # workspace too small


def test_binding_refuses_cpu_tensors():
    import torch
    from speculative_decoding_verification_48_gb300 import binding
    x = torch.zeros(2, 3, 10)
    with pytest.raises((ValueError, RuntimeError)):
        binding.spec_verify_chain(x, torch.zeros(2, 2, 10), torch.zeros(2, 2, dtype=torch.int32),
                                  torch.ones(2), torch.zeros(2, 3))


def test_simulator_host_checks():
    """The simulator runs only the library's CUDA kernels: without a CUDA
    device it refuses, before any work."""
    from speculative_decoding_verification_48_gb300 import simulate
    with pytest.raises(ValueError):
        simulate.simulate(4, 0.8, device="cpu")
    with pytest.raises(ValueError):
        simulate.simulate(0, 0.8, device="cpu")
    assert simulate._parse_gammas("1-4") == [1, 2, 3, 4]
    assert simulate._parse_gammas("2,5") == [2, 5]
