"""The parity helpers' own arithmetic (CPU only): the dsink scale is the sum
over tokens of |p_sink * Delta| per head, so it bounds |dsink| from above and
equals it when every token's term has the same sign."""
import numpy as np
import torch

import oracle
from bwd_sparse_mqa_gb300 import inputs
from tests import _parity as P


def _case(same_sign: bool):
    x = inputs.custom(2, 9, 40, 8, 64, 24, recipe="causal_masked10", seed=31)
    if same_sign:
        # dO = O (rounded to bf16): Delta = <O, O> > 0 on every token that has
        # a valid slot, 0 on the others, so no two terms cancel.
        o, _ = oracle.fwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"])
        x["do"] = torch.from_numpy(o).to(torch.bfloat16).reshape(x["q"].shape)
    _, lse = oracle.fwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"])
    _, _, dsink, delta = oracle.bwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], x["do"])
    return x, lse, dsink, delta


def test_dsink_scale_bounds_dsink():
    x, lse, dsink, delta = _case(same_sign=False)
    scale = P.dsink_scale(x["attn_sink"], lse, delta)
    assert scale >= float(np.max(np.abs(dsink))) * (1 - 1e-12)
    # Random dO mixes signs, so the bound is strict here.
    assert scale > 1.05 * float(np.max(np.abs(dsink)))


def test_dsink_scale_equals_dsink_without_cancellation():
    x, lse, dsink, delta = _case(same_sign=True)
    assert np.all(np.asarray(delta) >= 0)
    scale = P.dsink_scale(x["attn_sink"], lse, delta)
    np.testing.assert_allclose(scale, float(np.max(np.abs(dsink))), rtol=1e-9)


def test_scaled_tolerance_reduces_to_plain_one():
    ref = np.array([0.5, -2.0, 1.0])
    gpu = torch.tensor([0.51, -2.0, 1.0])
    plain = P.rel_err(gpu, ref)
    assert abs(plain - 0.01 / 2.0) < 1e-6
    # A scale below max|ref| leaves the check as it was; a larger one divides
    # the error by it instead.
    assert abs(P.assert_close("dsink", gpu, ref, scale=1.0) - plain) < 1e-12
    assert abs(P.assert_close("dsink", gpu, ref, scale=4.0) - 0.01 / 4.0) < 1e-6
