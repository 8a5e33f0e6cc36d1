"""Float64 CPU oracle for speculative-sampling verification (test infrastructure).

Imported only by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py``; the library never imports it.
"""
from .spec_verify_oracle import (  # noqa: F401
    ROW_OK, ROW_BAD_TOKEN, ROW_NONFINITE, ROW_BAD_TREE, ROW_TIMEOUT,
    ROW_BAD_TEMPERATURE, tempered_softmax, first_argmax, inverse_cdf,
    residual_distribution, verify_chain, verify_chain_greedy,
    verify_tree_greedy, draft_sample, tree_ancestor_mask, tree_kv_compact,
    acceptance_probability, accepted_count_law, expected_tokens_per_round,
    speedup_estimate,
)
