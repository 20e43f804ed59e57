"""Seeded synthetic inputs for the CSA / HCA hybrid compressed attention.

This package is shared by the tests, the benchmark and the smoke check. It draws random
tensors and holds the table of workload shapes; it performs none of the method's arithmetic
(no pooling, scoring, selection or attention), so neither the CUDA library nor the oracle
depends on the other through it.
"""
from .workloads import (  # noqa: F401
    CONFIGS,
    LayerShape,
    Workload,
    generate_layer,
    index_key_rows,
    get_config,
)
