"""GB300 (sm_103a) block-sparse FlexAttention forward.

``flexattn`` is the Python binding of the C-ABI (include/flexattn.h); it
loads libflexattn.so on first use and raises if it is missing.
``workloads`` holds the seeded synthetic inputs.
"""
from . import flexattn, workloads  # noqa: F401

__all__ = ["flexattn", "workloads"]
