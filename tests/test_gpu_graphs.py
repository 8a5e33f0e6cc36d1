"""Calls captured into a CUDA graph and replayed on new inputs.

A replay reuses the kernel parameters fixed at capture.  Every replay must
still verify the inputs it finds in the buffers: two input sets written into
the same buffers between replays each match the oracle.  The call is large
enough that, outside a graph, its decide kernel would merge partials as they
arrive.
"""

import ctypes

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
