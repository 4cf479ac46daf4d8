"""GB300-native (sm_103a) hot path of Attention Residuals.

The depth-wise softmax aggregation -- Full, Block and the two-phase Block
inference scheme -- as hand-written CUDA kernels behind a C ABI
(include/attnres.h, libattnres.so), with thin PyTorch wrappers.

``workloads`` (seeded synthetic inputs) imports without the CUDA library;
everything in ``api`` needs libattnres.so and raises if it is missing.
"""
from . import workloads  # noqa: F401

__all__ = [
    "depth_aggregate", "block_phase1", "block_phase2_merge", "partial_update",
    "full_stack_forward", "TwoPhaseBlock", "block_two_phase", "block_schedule",
    "atomic_block_size", "workloads",
]


def __getattr__(name):
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
