"""CPU check of the chunked full-size comparison used by the GPU parity
tests: a workload generated in pool chunks equals the one generated whole,
and a mismatch planted in one row of a later chunk is reported at its row
of the whole workload."""

import numpy as np
import torch

import chunked_oracle as CO
import oracle
from speculative_decoding_verification_48_gb300 import workloads as W


def test_chunked_generation_and_comparison():
    spec = W.c2_spec(0.7, rounds=10)
    spec = {**spec, "V": 512}
    whole = W.make_chain(**spec)
    with CO.spawn_pool(2) as pool:
        case = CO.generate(pool, spec, 4)
        for f in ("target", "draft", "draft_tokens", "temperatures", "uniforms"):
            assert torch.equal(getattr(case, f), getattr(whole, f))
        ref = oracle.verify_chain(*whole.numpy64())
        outs = [ref["tokens"].copy(), ref["num_accepted"].copy(),
                ref["diag"].astype(np.float32), ref["status"].copy()]
        cmp = CO.compare(pool, spec, outs, 3, 1e-4)
        assert cmp["failures"] == [] and cmp["exact"] == 10
        assert np.array_equal(cmp["num_accepted"], ref["num_accepted"])
        outs[0][7, 0] = -5
        cmp = CO.compare(pool, spec, outs, 3, 1e-4)
        assert [f[0] for f in cmp["failures"]] == [7]
