"""Host-buffer entry points (smqa_fwd_host, smqa_fwd_bwd_host): the chunked,
overlapped copies and kernels give the oracle's results, and exactly the
results of the device-buffer entry points (O, LSE, dQ, dsink always; dKV in
the deterministic mode, within fp32-atomic rounding otherwise)."""
import ctypes

import pytest
import torch

import oracle
from bwd_sparse_mqa_gb300 import (_lib, inputs, sparse_mqa_fwd_bwd_host, sparse_mqa_fwd_host)
from tests import _parity as P

# (B, S, S_kv, H, D, topk, recipe): chunks of at least 256 tokens rounded up
# to whole waves (the minimum decides at these sizes; smqa_host_chunk_plan
# gives the plan) -- on a 152-SM GB300
#   1 x 1100 -> three pieces of S of 304 tokens and a last one of 188;
#   2 x 600  -> two pieces per batch element (kv and dKV offsets per b);
#   5 x 100  -> whole batch elements, three in a chunk and a last chunk of two.
CASES = [(1, 1100, 500, 32, 512, 96, "causal_masked10"),
         (2, 600, 300, 128, 512, 64, "hot4096_masked10"),
         (5, 100, 120, 32, 64, 64, "causal_uniform")]


def _pinned(x: dict) -> dict:
    return {k: v.pin_memory() for k, v in x.items()}


def _plan(shape) -> list:
    lib = _lib.load()
    n = lib.smqa_host_chunk_plan(shape, None, 0)
    buf = (ctypes.c_int32 * (4 * n))()
    lib.smqa_host_chunk_plan(shape, buf, n)
    return [tuple(buf[4 * c:4 * c + 4]) for c in range(n)]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])))
def test_fwd_bwd_host_matches_device_path_and_oracle(case):
    B, S, S_kv, H, D, K, recipe = case
    plan = _plan(_lib.Shape(B, S, S_kv, H, D, K))
    assert len(plan) >= 2  # the case spans several chunks
    x = inputs.custom(B, S, S_kv, H, D, K, recipe=recipe, seed=21)
    h = _pinned(x)
    o, lse, dq, dkv, dsink = sparse_mqa_fwd_bwd_host(
        h["q"], h["kv"], h["attn_sink"], h["topk_idxs"], h["do"], return_dsink=True)
    assert P.device_status() == 0
    assert o.device.type == "cpu" and dkv.dtype == torch.bfloat16

    g = P.to_dev(x)
    o_d, lse_d = P.run_fwd(g)
    dq_d, dkv_d, dsink_d = P.run_bwd(g, o_d, lse_d, g["do"], return_dsink=True)
    assert torch.equal(o, o_d.cpu()) and torch.equal(lse, lse_d.cpu())
    assert torch.equal(dq, dq_d.cpu()) and torch.equal(dsink, dsink_d.cpu())
    assert P.rel_err(dkv, dkv_d.double().cpu().numpy()) < 8e-3

    o_ref, lse_ref = oracle.fwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"])
    P.assert_close("o", o, o_ref)
    P.assert_close("lse", lse, lse_ref)
    dq_ref, dkv_ref, dsink_ref, _ = oracle.bwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"],
                                               x["do"])
    P.assert_close("dq", dq, dq_ref)
    P.assert_close("dkv", dkv, dkv_ref)
    P.assert_close("dsink", dsink, dsink_ref)


@pytest.mark.gpu
@pytest.mark.parametrize("fp32_out", [False, True])
def test_fwd_bwd_host_deterministic_is_bit_exact(fp32_out):
    x = inputs.custom(2, 600, 300, 128, 512, 96, recipe="causal_masked10", seed=22)
    h = _pinned(x)
    g = P.to_dev(x)
    o_d, lse_d = P.run_fwd(g)
    dq_d, dkv_d = P.run_bwd(g, o_d, lse_d, g["do"], deterministic=True,
                            return_dkv_accum_dtype=fp32_out)
    ws = torch.empty((int(_lib.load().smqa_fwd_bwd_host_workspace_bytes(
        _lib.Shape(2, 600, 300, 128, 512, 96),
        _lib.FLAG_DETERMINISTIC_DKV | (_lib.FLAG_RETURN_DKV_FP32 if fp32_out else 0))),),
        dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the same workspace twice: nothing carries over
        o, lse, dq, dkv = sparse_mqa_fwd_bwd_host(
            h["q"], h["kv"], h["attn_sink"], h["topk_idxs"], h["do"], workspace=ws,
            deterministic=True, return_dkv_accum_dtype=fp32_out)
        assert P.device_status() == 0
        assert dkv.dtype == (torch.float32 if fp32_out else torch.bfloat16)
        assert torch.equal(o, o_d.cpu()) and torch.equal(lse, lse_d.cpu())
        assert torch.equal(dq, dq_d.cpu()) and torch.equal(dkv, dkv_d.cpu())


@pytest.mark.gpu
@pytest.mark.parametrize("case", [CASES[0], CASES[2]], ids=["d512", "d64"])
def test_fwd_host_matches_device_path(case):
    B, S, S_kv, H, D, K, recipe = case
    x = inputs.custom(B, S, S_kv, H, D, K, recipe=recipe, seed=23)
    h = _pinned(x)
    out = {"o": torch.empty(B, S, H, D, dtype=torch.bfloat16).pin_memory(),
           "lse": torch.empty(B, S, H, dtype=torch.float32).pin_memory()}
    o, lse = sparse_mqa_fwd_host(h["q"], h["kv"], h["attn_sink"], h["topk_idxs"], out=out,
                                 reference_rounding=True)
    assert o is out["o"] and lse is out["lse"]
    g = P.to_dev(x)
    o_d, lse_d = P.run_fwd(g, reference_rounding=True)
    assert torch.equal(o, o_d.cpu()) and torch.equal(lse, lse_d.cpu())


@pytest.mark.gpu
def test_host_entry_rejects_device_buffers():
    """A device pointer where host memory is expected, or a host workspace,
    is refused before anything is queued."""
    lib = _lib.load()
    x = inputs.custom(1, 64, 64, 16, 64, 32, seed=24)
    shp = _lib.Shape(1, 64, 64, 16, 64, 32)
    h = _pinned(x)
    g = P.to_dev(x)
    need = int(lib.smqa_fwd_host_workspace_bytes(shp))
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(h["q"]).pin_memory()
    lse = torch.empty(1, 64, 16, dtype=torch.float32).pin_memory()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.smqa_fwd_host(ptr(g["q"]), ptr(h["kv"]), ptr(h["attn_sink"]), ptr(h["topk_idxs"]),
                           shp, 0.0, ptr(o), ptr(lse), ptr(ws), need, 0, stream)
    assert st == _lib.SMQA_ERR_INVALID_ARG and b"device memory" in lib.smqa_last_error()
    host_ws = torch.empty((need,), dtype=torch.uint8).pin_memory()
    st = lib.smqa_fwd_host(ptr(h["q"]), ptr(h["kv"]), ptr(h["attn_sink"]), ptr(h["topk_idxs"]),
                           shp, 0.0, ptr(o), ptr(lse), ptr(host_ws), need, 0, stream)
    assert st == _lib.SMQA_ERR_INVALID_ARG and b"workspace" in lib.smqa_last_error()
    torch.cuda.synchronize()
    assert P.device_status() == 0
