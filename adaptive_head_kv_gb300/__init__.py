"""GB300 (sm_103a) implementation of the FastGen hot path: prompt profiling,
per-head compaction and windowed decode attention, behind a C ABI
(include/fastgen.h, libfastgen.so) with a ctypes binding."""
from . import fastgen  # noqa: F401
from .fastgen import FastGenError, Params, PlanInfo  # noqa: F401
