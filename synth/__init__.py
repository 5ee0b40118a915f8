"""Seeded synthetic inputs for the compressed sparse attention hot path.

This package is the only code that both the CUDA side (tests, bench) and the
oracle side draw their inputs from.  It holds random draws, rounding of those
draws to their storage type, workload shapes and paged-block bookkeeping --
none of the method's arithmetic.
"""

from .workloads import (  # noqa: F401
    LayerSpec,
    SeqSpec,
    Workload,
    WORKLOADS,
    workload,
    layer_params,
    seq_raw,
    seq_history,
    seq_index_keys,
    index_key_case,
    seq_queries,
    block_table,
    physical_row,
    random_subset,
    round_bf16,
    CACHE_KINDS,
    BLOCK_POSITIONS,
)
