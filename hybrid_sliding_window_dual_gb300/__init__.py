"""Hybrid sliding-window attention over a dual KV pool, native to GB300.

The compute lives in libhswa.so (CUDA for sm_103a behind a C ABI declared in
include/hswa.h); this package is its thin ctypes binding plus the build step.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import Config, Layer, HswaError, NoSpace, lib, library_path  # noqa: F401
