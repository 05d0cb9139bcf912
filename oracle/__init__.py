"""CPU oracle for the decode-time sampler (test infrastructure; never imported by the library).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  Parity of each function is pinned by the ``-m "not gpu"`` tests (hand cases from
the pages' rules, closed forms, invariants, brute force against a second formulation, Philox
known answers and the cuRAND host generator).
"""
from .philox import philox4x32_10, row_uniform  # noqa: F401
from .sampling import (  # noqa: F401
    Params, params_valid, widen, history_counts, apply_penalties, rank_order, min_p_cut, top_p_cut,
    draw_index, log_softmax, allowed_renorm, sample_row, logprobs_row, sample_call, logprobs_call,
    c_logf, BOUNDARY_EPS, accept_window, verify_call, history_call, history_append, history_tail,
    HISTORY_RING_CAP, shard_record, merge_records,
)
