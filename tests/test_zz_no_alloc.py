"""The entry points for callers that cannot allocate device memory
(smqa_fwd_static_scratch, smqa_bwd_static_scratch): they must give what the
ordinary smqa_fwd / smqa_bwd give, call after call, using only the library's
static scratch buffer.

Such callers -- code under a memory planner that owns all device memory,
plugins handed only their tensors, hot paths that must not risk cudaMalloc's
synchronisation -- cannot pass smqa_fwd / smqa_bwd a workspace.  This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import pytest
import torch

from bwd_sparse_mqa_gb300 import _lib, inputs
from tests import _parity as P


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_scratch_rejects_oversized_shape_without_gpu_work():
    """Too large for the static buffer: rejected on the host, nothing runs."""
    lib = _lib.load()
    big = _lib.Shape(1, 8192, 65536, 128, 512, 2048)   # 128 MiB accumulator alone
    head = _lib.Shape(1, 8192, 8192, 128, 512, 2048)   # the H=128 D=512 benchmark shape
    assert lib.smqa_bwd_workspace_bytes(head, 0) <= _lib.STATIC_SCRATCH_BYTES
    assert lib.smqa_bwd_workspace_bytes(head, _lib.FLAG_DETERMINISTIC_DKV) <= \
        _lib.STATIC_SCRATCH_BYTES
    need = lib.smqa_bwd_workspace_bytes(big, 0)
    assert need > _lib.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    rc = lib.smqa_bwd_static_scratch(*([fake] * 7), big, 0.0, fake, fake, None, 0, None)
    assert rc == _lib.SMQA_ERR_UNSUPPORTED
    assert b"static buffer" in lib.smqa_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("fp32_dkv", [False, True])
def test_static_scratch_matches_workspace_backward_twice(fp32_dkv):
    lib = _lib.load()
    x = inputs.custom(2, 96, 512, 128, 512, 200, recipe="causal_masked10", seed=21)
    g = P.to_dev(x)
    o, lse = P.run_fwd(g)
    B, S, H, D = g["q"].shape
    S_kv, K = g["kv"].shape[1], g["topk_idxs"].shape[2]
    shp = _lib.Shape(B, S, S_kv, H, D, K)
    flags = _lib.FLAG_RETURN_DKV_FP32 if fp32_dkv else 0
    assert lib.smqa_bwd_workspace_bytes(shp, flags) <= _lib.STATIC_SCRATCH_BYTES
    dkv_dtype = torch.float32 if fp32_dkv else torch.bfloat16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [_p(g["q"]), _p(g["kv"]), _p(g["attn_sink"]), _p(o), _p(g["do"]),
            _p(g["topk_idxs"]), _p(lse)]

    # Reference: the workspace backward.
    ws = torch.empty(lib.smqa_bwd_workspace_bytes(shp, flags), dtype=torch.uint8, device="cuda")
    dq_ref = torch.empty_like(g["q"])
    dkv_ref = torch.empty((B, S_kv, D), dtype=dkv_dtype, device="cuda")
    _lib.check("smqa_bwd", lib.smqa_bwd(*args, shp, 0.0, _p(dq_ref), _p(dkv_ref), None, _p(ws),
                                        ws.numel(), flags, stream))
    torch.cuda.synchronize()

    # Two calls in a row through the static-scratch entry point: the second
    # must not see the first one's accumulator.
    for _ in range(2):
        dq = torch.full_like(g["q"], float("nan"))
        dkv = torch.full((B, S_kv, D), float("nan"), dtype=dkv_dtype, device="cuda")
        _lib.check("smqa_bwd_static_scratch",
                   lib.smqa_bwd_static_scratch(*args, shp, 0.0, _p(dq), _p(dkv), None, flags,
                                               stream))
        torch.cuda.synchronize()
        assert lib.smqa_device_status(1) == 0
        assert torch.equal(dq, dq_ref)  # dq has no atomics: identical
        e = P.rel_err(dkv, dkv_ref.double().cpu().numpy())
        assert e <= P.TOL["dkv"], f"dkv differs from the workspace backward: {e:.3e}"


@pytest.mark.gpu
def test_static_scratch_forward_matches_workspace_forward_twice():
    lib = _lib.load()
    x = inputs.custom(2, 96, 512, 128, 512, 200, recipe="causal_masked10", seed=22)
    g = P.to_dev(x)
    B, S, H, D = g["q"].shape
    S_kv, K = g["kv"].shape[1], g["topk_idxs"].shape[2]
    shp = _lib.Shape(B, S, S_kv, H, D, K)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [_p(g["q"]), _p(g["kv"]), _p(g["attn_sink"]), _p(g["topk_idxs"])]
    ws = torch.empty(lib.smqa_fwd_workspace_bytes(shp), dtype=torch.uint8, device="cuda")
    o_ref = torch.empty_like(g["q"])
    lse_ref = torch.empty((B, S, H), dtype=torch.float32, device="cuda")
    _lib.check("smqa_fwd", lib.smqa_fwd(*args, shp, 0.0, _p(o_ref), _p(lse_ref), _p(ws),
                                        ws.numel(), 0, stream))
    torch.cuda.synchronize()
    for _ in range(2):
        o = torch.full_like(g["q"], float("nan"))
        lse = torch.full((B, S, H), float("nan"), device="cuda")
        _lib.check("smqa_fwd_static_scratch",
                   lib.smqa_fwd_static_scratch(*args, shp, 0.0, _p(o), _p(lse), 0, stream))
        torch.cuda.synchronize()
        assert lib.smqa_device_status(1) == 0
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
