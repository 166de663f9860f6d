"""The autograd wrapper (sparse_mqa): gradients of a loss through O reach q,
kv and attn_sink, and equal the oracle's dQ, dKV and dsink for the same dO."""
import pytest
import torch

import oracle
from bwd_sparse_mqa_gb300 import inputs, sparse_mqa
from tests import _parity as P


@pytest.mark.gpu
@pytest.mark.parametrize("D,H", [(512, 64), (64, 16)])
def test_autograd_gradients_match_oracle(D, H):
    x = inputs.custom(1, 40, 120, H, D, 96, recipe="causal_masked10", seed=13)
    g = P.to_dev(x)
    q = g["q"].clone().requires_grad_(True)
    kv = g["kv"].clone().requires_grad_(True)
    sink = g["attn_sink"].clone().requires_grad_(True)
    o, lse = sparse_mqa(q, kv, sink, g["topk_idxs"])
    assert not lse.requires_grad
    w = g["do"]  # bf16: d(loss)/dO is exactly w
    (o.float() * w.float()).sum().backward()
    torch.cuda.synchronize()
    assert q.grad.dtype == torch.bfloat16 and kv.grad.dtype == torch.bfloat16
    assert sink.grad.dtype == torch.float32 and sink.grad.shape == (H,)
    dq_ref, dkv_ref, dsink_ref, _ = oracle.bwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"],
                                               x["do"])
    P.assert_close("dq", q.grad.reshape(-1, H, D), dq_ref)
    P.assert_close("dkv", kv.grad, dkv_ref)
    P.assert_close("dsink", sink.grad, dsink_ref)
