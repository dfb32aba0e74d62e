"""GB300 (sm_103a) library for the data-parallel hot path of batch
speculative decoding: greedy and stochastic verification of k draft tokens
against k+1 target logit rows, realignment of a contiguous left-padded KV
cache with its position IDs and attention mask, and same-length grouping.

The C ABI is include/specverify.h (libspecverify.so); this package is a thin
ctypes binding with the same function names.
"""
from .api import (  # noqa: F401
    FLAG_BAD_TOKEN,
    FLAG_NONFINITE,
    FLAG_Q_ZERO,
    FLAG_ZERO_RESIDUAL,
    MAX_GROUP_N,
    MAX_K,
    REALIGN_CAPACITY,
    REALIGN_EMIT,
    REALIGN_LAYOUT,
    REALIGN_OK,
    REALIGN_TIMEOUT,
    SpecError,
    Workspace,
    spec_commit_ragged,
    spec_group_by_length,
    spec_repad_gather,
    spec_unpad_scatter,
    MAX_POOL,
    spec_realign_kv,
    spec_realign_kv_multi,
    MAX_CACHES,
    spec_rebuild_pos_mask,
    spec_round_greedy,
    spec_round_sample,
    spec_verify_greedy,
    spec_verify_greedy_static,
    STATIC_SCRATCH_BYTES,
    spec_verify_sample,
    spec_verify_sample_filtered,
    spec_workspace_bytes,
)
from .graph import RoundGraph  # noqa: F401,E402
