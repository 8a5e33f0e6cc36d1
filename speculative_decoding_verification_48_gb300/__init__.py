"""GB300 (sm_103a) verification step of speculative decoding.

The compute path is the CUDA library ``lib/libspec_verify.so`` (C ABI in
include/spec_verify.h); ``binding`` wraps it with the same function names.
``workloads`` creates seeded synthetic inputs.  Importing this package does
not load the library; the first call does, and raises if it is missing.
"""

from .binding import (  # noqa: F401
    SV_BF16, SV_F16, SV_F32, SV_ROW_BAD_TEMPERATURE, SV_ROW_BAD_TOKEN, SV_ROW_BAD_TREE,
    SV_ROW_NONFINITE, SV_ROW_OK, SV_ROW_TIMEOUT, SpecVerifyError, lib, library_path,
    spec_draft_sample, spec_tree_kv_compact, spec_tree_mask, spec_verify_chain,
    spec_verify_chain_greedy, spec_verify_force_stream_path, spec_verify_set_call_counter, spec_verify_status_string,
    spec_verify_tree_greedy, spec_verify_wait_selftest, spec_verify_workspace_bytes,
)
