"""spec_verify_chain_no_alloc, the entry point for callers that cannot
allocate device memory (for example a plugin in a serving engine that has
already reserved the whole GPU, or a decode loop that must not call
cudaMalloc because it can synchronise the device).  Its scratch memory is a
fixed 8 MiB array inside the library instead of a caller-provided workspace.

The test calls it through the C ABI three times in a row, with different
shapes, and checks each result against the regular spec_verify_chain on the same
inputs: the same accepted counts and tokens, and diagnostics within the
probability tolerance the parity tests use.  It also checks that a shape
whose workspace would not fit in the array is refused before anything is
enqueued.  This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle.compare import prob_tolerance
from speculative_decoding_verification_48_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SV_OK, SV_ERR_UNSUPPORTED = 0, 2
SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as pkg
    L = pkg.lib()
    vp, i = ctypes.c_void_p, ctypes.c_int
    L.spec_verify_chain_no_alloc.argtypes = [vp, i, vp, i, i, vp, vp, vp, i, i, i,
                                             vp, vp, vp, vp, vp]
    L.spec_verify_chain_no_alloc.restype = i
    return pkg


def _dt(t):
    return {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[t.dtype]


def _no_alloc_call(sv, dev_in, probs, outs, B=None):
    t, d, x, T, u = dev_in
    Bc, G1, V = t.shape
    stream = torch.cuda.current_stream(DEV).cuda_stream
    return sv.lib().spec_verify_chain_no_alloc(
        t.data_ptr(), _dt(t), d.data_ptr(), _dt(d), int(probs), x.data_ptr(), T.data_ptr(),
        u.data_ptr(), Bc if B is None else B, G1 - 1, V, outs[0].data_ptr(), outs[1].data_ptr(),
        outs[2].data_ptr(), outs[3].data_ptr(), stream)


def _check_against_regular(sv, case):
    dev_in = [a.to(DEV) for a in (case.target, case.draft, case.draft_tokens,
                                  case.temperatures, case.uniforms)]
    B, g = case.B, case.gamma
    ref = sv.spec_verify_chain(*dev_in, draft_is_probs=case.draft_is_probs)
    # outputs pre-filled with junk, so a call that writes nothing is caught
    outs = [torch.full((B, g + 1), 12345, dtype=torch.int32, device=DEV),
            torch.full((B,), 12345, dtype=torch.int32, device=DEV),
            torch.full((B, g, 4), 7.0, dtype=torch.float32, device=DEV),
            torch.full((B,), 12345, dtype=torch.int32, device=DEV)]
    st = _no_alloc_call(sv, dev_in, case.draft_is_probs, outs)
    assert st == SV_OK, sv.spec_verify_status_string(st)
    torch.cuda.synchronize()
    r = [o.cpu().numpy() for o in ref]
    o = [x.cpu().numpy() for x in outs]
    assert np.array_equal(o[3], r[3])            # row status
    assert np.array_equal(o[1], r[1])            # accepted counts
    assert np.array_equal(o[0], r[0])            # tokens
    tol = prob_tolerance(case.meta.get("dtype", "bf16"))
    np.testing.assert_allclose(o[2], r[2], rtol=0, atol=tol)
    return o


def test_no_alloc_matches_regular_entry_point_three_calls_in_a_row(sv):
    # first call: batched chain with greedy rows and rejections everywhere
    first = W.make_chain("no_alloc_a", 4101, B=24, gamma=7, V=50000, dtype="bf16",
                         target="zipf", draft_sigma=(0.3, 2.0),
                         temperature=lambda b, v: 0.0 if b % 8 == 0 else 1.2 * v + 0.05)
    o1 = _check_against_regular(sv, first)
    assert len(set(o1[1].tolist())) > 2
    # second call, right after, on the same scratch array: another shape,
    # fp32 logits and a ragged vocabulary
    second = W.make_chain("no_alloc_b", 4102, B=40, gamma=4, V=20001, dtype="f32",
                          draft_sigma=(0.2, 1.5), temperature=lambda b, v: 0.3 + v)
    _check_against_regular(sv, second)
    # third call: rows on 16-byte boundaries again, with another batch size
    # and gamma, and the draft given as fp32 probabilities (forced all-accept
    # rows draw the bonus token)
    third = W.make_chain("no_alloc_c", 4103, B=33, gamma=5, V=32000, dtype="bf16",
                         target="zipf", draft_sigma=(0.7, 0.7), temperature=0.8,
                         draft_probs=True, force_accept_every=4)
    o3 = _check_against_regular(sv, third)
    assert np.all(o3[1][::4] == 5)


def test_no_alloc_refuses_shapes_beyond_the_scratch_array(sv):
    big_B = 1 << 16
    assert sv.spec_verify_workspace_bytes(big_B, 7, 4096) > SCRATCH_BYTES
    assert sv.spec_verify_workspace_bytes(64, 15, 128256) <= SCRATCH_BYTES
    # Every pointer is NULL: the size check must refuse the call before any
    # pointer is looked at (a call that got past it would stop at the NULL
    # checks of spec_verify_chain instead, with SV_ERR_INVALID_ARG).
    st = sv.lib().spec_verify_chain_no_alloc(None, 1, None, 1, 0, None, None, None, big_B, 3,
                                             4096, None, None, None, None, None)
    assert st == SV_ERR_UNSUPPORTED, sv.spec_verify_status_string(st)
