"""Calls captured into a CUDA graph and replayed on new inputs.

A replay reuses the kernel parameters fixed at capture.  Every replay must
still verify the inputs it finds in the buffers: two input sets written into
the same buffers between replays each match the oracle.  The call is large
enough that, outside a graph, its decide kernel would merge partials as they
arrive.
"""

import ctypes
import os

import numpy as np
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


def _case(seed):
    return W.make_chain(f"graph_{seed}", seed, B=512, gamma=3, V=32768, dtype="bf16",
                        draft_sigma=(0.3, 1.5),
                        temperature=lambda b, v: 0.0 if b % 7 == 0 else 0.4 + v)


def test_graph_replays_verify_their_own_inputs(sv):
    cases = [_case(601), _case(602)]
    c0 = cases[0]
    B, g, V = c0.B, c0.gamma, c0.V
    bufs = [c0.target.to(DEV), c0.draft.to(DEV), c0.draft_tokens.to(DEV),
            c0.temperatures.to(DEV), c0.uniforms.to(DEV)]
    toks = torch.empty((B, g + 1), dtype=torch.int32, device=DEV)
    nacc = torch.empty((B,), dtype=torch.int32, device=DEV)
    diag = torch.empty((B, g, 4), dtype=torch.float32, device=DEV)
    st = torch.empty((B,), dtype=torch.int32, device=DEV)
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, 2 * g + 1, V, sv.SV_BF16),
                     dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream(DEV)

    def call():
        sv.spec_verify_chain(*bufs, out_tokens=toks, out_num_accepted=nacc, out_diag=diag,
                             out_row_status=st, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()                                   # outside the graph first
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for case in cases + cases[:1]:
        for buf, src in zip(bufs, (case.target, case.draft, case.draft_tokens,
                                   case.temperatures, case.uniforms)):
            buf.copy_(src.to(DEV))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        args = case.numpy64()
        ref = oracle.verify_chain(*args)
        cmp = compare_chain(args, ref, toks.cpu().numpy(), nacc.cpu().numpy(), st.cpu().numpy(),
                            diag.cpu().numpy(), prob_tol=1e-4)
        assert not cmp["failures"], (case.name, cmp["failures"][:3])
        assert len(cmp["boundary"]) <= 5


# Header words of a workspace of the two-launch path (byte offsets of the
# 4 KB state header): the claim-failure word, the counter-reset word, the
# counters' validity stamp and the epoch of the last completed call.
CLAIM_BYTES, ERR, READY, STAMP, EPOCH_BASE = 2048, 2048, 2176, 2304, 2432


def _u64(ws, off):
    return int(ws[off:off + 8].cpu().view(torch.int64).item())


def _put_u64(ws, off, v):
    ws[off:off + 8].copy_(torch.tensor([v], dtype=torch.int64).view(torch.uint8).to(DEV))


def test_graph_replays_ignore_words_left_by_earlier_replays(sv):
    """Every replay runs with its own device-side epoch.  Before every other
    replay, the words a failed earlier replay could have left are planted:
    the claim-failure word and the counter-reset word hold the last epoch,
    the stamp is cleared, and the claim counters and every partial slot hold
    garbage.  The replay must reset the counters itself (waiting for its own
    reset, not an earlier one), so that every partial is rewritten, report
    no timeout and match the oracle."""
    case = _case(603)
    B, g, V = case.B, case.gamma, case.V
    bufs = [t.to(DEV) for t in (case.target, case.draft, case.draft_tokens, case.temperatures,
                                case.uniforms)]
    toks = torch.empty((B, g + 1), dtype=torch.int32, device=DEV)
    nacc = torch.empty((B,), dtype=torch.int32, device=DEV)
    diag = torch.empty((B, g, 4), dtype=torch.float32, device=DEV)
    st = torch.empty((B,), dtype=torch.int32, device=DEV)
    ws = torch.zeros(sv.spec_verify_workspace_bytes(B, 2 * g + 1, V, sv.SV_BF16),
                     dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream(DEV)

    def call():
        sv.spec_verify_chain(*bufs, out_tokens=toks, out_num_accepted=nacc, out_diag=diag,
                             out_row_status=st, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    args = case.numpy64()
    ref = oracle.verify_chain(*args)
    epochs = []
    for rep in range(4):
        last = _u64(ws, EPOCH_BASE)
        epochs.append(last)
        if rep % 2 == 1:
            _put_u64(ws, ERR, last)
            _put_u64(ws, READY, last)
            _put_u64(ws, STAMP, 0)
            ws[:CLAIM_BYTES].fill_(0x7F)
            ws[4096:].fill_(0x3F)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert not (st.cpu().numpy() & sv.SV_ROW_TIMEOUT).any()
        cmp = compare_chain(args, ref, toks.cpu().numpy(), nacc.cpu().numpy(), st.cpu().numpy(),
                            diag.cpu().numpy(), prob_tol=1e-4)
        assert not cmp["failures"], (rep, cmp["failures"][:3])
    # one epoch per call: the first call, then each replay
    assert epochs == list(range(epochs[0], epochs[0] + 4)) and epochs[0] >= 1
    assert _u64(ws, EPOCH_BASE) == epochs[-1] + 1


def _tag(call_id):
    return (((call_id << 1) | 1) * 0x9E3779B1) & 0xFFFFFFFF


def _tag_wrap_body():
    """Runs in a fresh process: calls numbered across 2^31, each on a
    workspace whose partial slots all carry the tag its own partials get, as
    partials left by the call numbered 2^31 below it would.  Calls at or past
    2^31 must not merge partials as they arrive; every call matches the
    oracle."""
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as svm
    case = _case(604)
    B, g, V = case.B, case.gamma, case.V
    bufs = [t.to(DEV) for t in (case.target, case.draft, case.draft_tokens, case.temperatures,
                                case.uniforms)]
    nb = svm.spec_verify_workspace_bytes(B, 2 * g + 1, V, svm.SV_BF16)
    ws = torch.zeros(nb, dtype=torch.uint8, device=DEV)
    args = case.numpy64()
    ref = oracle.verify_chain(*args)
    first = (1 << 31) - 2
    svm.spec_verify_set_call_counter(first - 1)
    for call_id in range(first, first + 5):
        if call_id >= 1 << 31:
            # a stale partial of the same tag in every slot: max 30, sum 1
            word = (_tag(call_id) << 32) | int(np.float32(30.0).view(np.uint32))
            ws[4096:].view(torch.int64)[:] = word - (1 << 64 if word >= 1 << 63 else 0)
            torch.cuda.synchronize()
        toks, nacc, diag, st = svm.spec_verify_chain(*bufs, workspace=ws)
        torch.cuda.synchronize()
        cmp = compare_chain(args, ref, toks.cpu().numpy(), nacc.cpu().numpy(),
                            st.cpu().numpy(), diag.cpu().numpy(), prob_tol=1e-4)
        assert not cmp["failures"], (call_id, cmp["failures"][:3])


def test_partial_tags_never_repeat_for_polling_calls(sv):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = "import test_gpu_graphs as t; t._tag_wrap_body(); print('tag wrap ok')"
    r = subprocess.run([sys.executable, "-c", code], cwd=os.path.join(root, "tests"),
                       env={**os.environ, "PYTHONPATH": root}, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "tag wrap ok" in r.stdout, r.stdout[-2000:] + r.stderr[-3000:]
