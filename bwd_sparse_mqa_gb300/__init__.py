"""GB300-native (sm_103a) top-k sparse multi-query attention with an attention
sink: forward and backward as hand-written tcgen05/TMA CUDA kernels behind a
C ABI (include/sparse_mqa.h).

    from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_interface, sparse_mqa_bwd_interface

The library is loaded on first use; importing this package does not touch
the GPU.
"""
from .api import (bwd_workspace_bytes, device_status, sparse_mqa_bwd_interface,  # noqa: F401
                  sparse_mqa_fwd_interface)

__all__ = ["sparse_mqa_fwd_interface", "sparse_mqa_bwd_interface", "bwd_workspace_bytes",
           "device_status"]
