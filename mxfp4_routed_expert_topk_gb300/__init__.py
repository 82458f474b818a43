"""GB300 (sm_103a) routed-expert MXFP4 MoE layer.

The compute lives in libmoe.so (hand-written CUDA kernels behind the C ABI of
include/moe.h); this package is its thin Python binding.  PyTorch supplies device
memory and streams only.
"""
from ._lib import *  # noqa: F401,F403
from ._lib import Pool, StreamPool, MoeError, lib, workspace, exact_fallbacks, status_string  # noqa: F401
from ._lib import moe_trace_begin, moe_trace_end  # noqa: F401


def build(verbose: bool = False) -> str:
    """Compile libmoe.so in-tree for sm_103a."""
    from .nvcc_build import build as _build
    return _build(verbose=verbose)
