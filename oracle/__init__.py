"""CPU oracle for batch speculative-decoding verification and realignment.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library's product
path never does.  The arithmetic lives in ``oracle.c`` (plain scalar C, fp64
probabilities); this module compiles it with gcc and marshals numpy arrays.

Parity pins for every function are in ``tests/test_oracle_*.py``.  The
length-grouping policy is this project's own construction (the pages' EXSPEC
scheduling appendix has no body): its parity is UNPINNED by the pages.
"""
from .core import (  # noqa: F401
    DT_BF16,
    DT_F16,
    DT_F32,
    MUTANTS,
    build,
    filter_cut,
    filter_info,
    commit_ragged,
    repad_gather,
    unpad_scatter,
    group_by_length,
    mutant,
    set_threads,
    threads,
    threads_available,
    realign_kv,
    realign_plan,
    rebuild_pos_mask,
    shift_slab,
    softmax_row,
    verify_greedy,
    verify_sample,
)
