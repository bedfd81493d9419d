"""GB300-native sparse MLA (DSA) attention: forward and backward.

The compute path is the CUDA library built from ``csrc/`` (see ``include/dsa.h``);
``dsa`` is its Python binding and ``workloads`` builds seeded synthetic inputs.
"""
from . import dsa  # noqa: F401
from .dsa import bwd, fwd, topk_compact  # noqa: F401
