"""GB300-native (sm_103a) top-k sparse multi-query attention with an attention
sink: forward and backward as hand-written tcgen05/TMA CUDA kernels behind a
C ABI (include/sparse_mqa.h).

    from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_interface, sparse_mqa_bwd_interface
    from bwd_sparse_mqa_gb300 import sparse_mqa   # autograd: grads for q, kv, attn_sink
    from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_bwd_host   # host tensors in and out

The library is loaded on first use; importing this package does not touch
the GPU.
"""
from .api import (SparseMQAFunction, batched_indexer_bwd, bwd_workspace_bytes,  # noqa: F401
                  device_status, fwd_bwd_host_workspace_bytes, fwd_host_workspace_bytes, fwd_workspace_bytes,
                  sparse_mqa, sparse_mqa_bwd_interface, sparse_mqa_fwd_bwd_host,
                  indexer_bwd_interface, set_wait_limit_ns, sparse_mqa_fwd_host,
                  sparse_mqa_fwd_interface)

__all__ = ["sparse_mqa_fwd_interface", "sparse_mqa_bwd_interface", "sparse_mqa",
           "SparseMQAFunction", "bwd_workspace_bytes", "fwd_workspace_bytes", "device_status",
           "sparse_mqa_fwd_host", "sparse_mqa_fwd_bwd_host", "fwd_host_workspace_bytes",
           "fwd_bwd_host_workspace_bytes", "set_wait_limit_ns", "indexer_bwd_interface",
           "batched_indexer_bwd"]
