"""Seeded synthetic workloads shaped like the GrowPage paper's 8B-model runs.

This package only draws random inputs (paged K/V caches, block tables,
query streams).  It holds none of the method's arithmetic: no summary
update, no calibration or rotary embedding, no scoring, no selection.  Both
the CUDA path's tests/bench and the oracle consume what it produces.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    ModelShape,
    Workload,
    config_seed,
    low_freq_directions,
    make_workload,
    query_step,
    fill_page,
    fill_pages,
    batch_kinds,
)
