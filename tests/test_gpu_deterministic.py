"""Deterministic dKV (SMQA_FLAG_DETERMINISTIC_DKV): 64-bit fixed-point integer
accumulation (binary point chosen per call from the inputs' magnitudes) gives
bit-identical dkv from run to run, equal to the oracle within the tolerance
and to the fp32-atomic path within its rounding.  Gradient-sized and large
inputs are covered by tests/test_gpu_magnitudes.py."""
import pytest
import torch

import oracle
from bwd_sparse_mqa_gb300 import inputs
from tests import _parity as P


def _bwd(g, o, lse, **kw):
    return P.run_bwd(g, o, lse, g["do"], **kw)


@pytest.mark.gpu
@pytest.mark.parametrize("D,H,fp32_out", [(512, 64, False), (512, 128, True), (64, 32, False)])
def test_deterministic_dkv_small(D, H, fp32_out):
    x = inputs.custom(2, 40, 100, H, D, 96, recipe="causal_masked10", seed=14)
    g = P.to_dev(x)
    o, lse = P.run_fwd(g)
    dq1, dkv1 = _bwd(g, o, lse, deterministic=True, return_dkv_accum_dtype=fp32_out)
    dq2, dkv2 = _bwd(g, o, lse, deterministic=True, return_dkv_accum_dtype=fp32_out)
    assert dkv1.dtype == (torch.float32 if fp32_out else torch.bfloat16)
    assert torch.equal(dkv1, dkv2) and torch.equal(dq1, dq2)
    dq_ref, dkv_ref, _, _ = oracle.bwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], x["do"])
    P.assert_close("dq", dq1, dq_ref)
    P.assert_close("dkv", dkv1, dkv_ref)
    _, dkv_atomic = _bwd(g, o, lse, return_dkv_accum_dtype=True)
    assert P.rel_err(dkv1, dkv_atomic.double().cpu().numpy()) < 8e-3


@pytest.mark.gpu
def test_deterministic_dkv_scatter_heavy_full_size():
    """The 4096-hot-row workload (each hot row receives ~4000 tokens'
    contributions): two deterministic backwards are bit-identical and match
    the fp32-atomic backward."""
    cfg = inputs.by_name("hot4096_h128_d512_k2048")
    g = inputs.make_inputs(cfg, device="cuda")
    o, lse = P.run_fwd(g)
    _, dkv1 = _bwd(g, o, lse, deterministic=True, return_dkv_accum_dtype=True)
    _, dkv2 = _bwd(g, o, lse, deterministic=True, return_dkv_accum_dtype=True)
    assert torch.equal(dkv1, dkv2)
    _, dkv_atomic = _bwd(g, o, lse, return_dkv_accum_dtype=True)
    err = (dkv1 - dkv_atomic).abs().max().item() / dkv_atomic.abs().max().item()
    assert err < 1e-5, err
