"""Seeded synthetic workloads shared by the tests, the bench and the oracle runs.

This package holds no arithmetic of the compression method itself: it only
draws token ids and Q/K/V tensors with planted attention structure, from a
counter-based generator, so that any single head can be regenerated alone.
"""
from .generator import (  # noqa: F401
    Config,
    CONFIGS,
    HEAD_TYPES,
    head_types,
    kv_of,
    make_head,
    make_kv,
    make_q,
    make_ids,
    make_workload,
    make_workload_split,
    punct_ids,
    special_ids,
)
