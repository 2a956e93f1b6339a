"""Single-GPU (sm_103a) routed Mixture-of-Experts FFN layer.

The layer -- router, top-k with renormalised softmax weights, expert-grouped
permutation, SwiGLU expert GEMMs on the tensor cores, unpermutation with the
shared-expert add -- runs in the CUDA kernels of libmoe (include/moe.h),
reached through the ctypes binding in ``_lib``.  ``MoELayer`` holds one layer's
weights and workspace on the device; ``synth`` draws seeded synthetic inputs.
"""
from .layer import MoELayer  # noqa: F401
from . import synth  # noqa: F401
