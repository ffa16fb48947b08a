"""GB300-native Gated Bidirectional Linear Attention (GBLA) layer.

The compute lives in libgbla.so (CUDA for sm_103a, C ABI in include/gbla.h);
``gbla`` is its thin Python binding and ``workloads`` draws seeded synthetic
inputs.  Build the library with ``build.build()``.
"""
from . import workloads  # noqa: F401

__all__ = ["gbla", "workloads", "build"]
