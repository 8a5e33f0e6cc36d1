"""Bounded device-side waits give up and report instead of hanging.

Each wait the kernels contain runs on a flag that nothing sets (through the
library's diagnostics entry point).  It must return SV_ROW_TIMEOUT within
its bound, and the context must stay usable: a verification call right
after still matches the oracle.
"""

import time

import pytest
import torch

import oracle
from oracle.compare import compare_chain
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


@pytest.mark.parametrize("which", [0, 1], ids=["counter_reset_wait", "partial_tag_poll"])
def test_bounded_wait_gives_up_and_reports(sv, which):
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = sv.spec_verify_wait_selftest(which, device=DEV)
    dt = time.perf_counter() - t0
    print(f"wait {which}: status {st} after {dt:.2f} s")
    assert st == sv.SV_ROW_TIMEOUT
    assert dt < 20.0


def test_context_usable_after_timeouts(sv):
    sv.spec_verify_wait_selftest(0, device=DEV)
    case = W.make_chain("after_timeout", 77, B=4, gamma=3, V=4096, dtype="bf16",
                        temperature=lambda b, v: 0.0 if b == 0 else 0.8)
    toks, nacc, diag, status = sv.spec_verify_chain(
        case.target.to(DEV), case.draft.to(DEV), case.draft_tokens.to(DEV),
        case.temperatures.to(DEV), case.uniforms.to(DEV))
    torch.cuda.synchronize()
    args = case.numpy64()
    ref = oracle.verify_chain(*args)
    cmp = compare_chain(args, ref, toks.cpu().numpy(), nacc.cpu().numpy(), status.cpu().numpy(),
                        diag.cpu().numpy(), prob_tol=1e-4)
    assert not cmp["failures"], cmp["failures"]
