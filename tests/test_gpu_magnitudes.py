"""GPU against the fp64 oracle at input magnitudes away from N(0,1).

Training gradients are small (a loss averaged over many tokens gives dO of
1e-6 and below), and trained queries can give peaked softmaxes with logits in
the tens.  The definition is exactly linear in dO and depends on q only
through the scaled logits, so these cases have the same relative tolerances
as the N(0,1) ones (tests/_parity.py): an error that grows as dO shrinks, or
as the logits grow, is a defect of the kernel's number formats, not a
property of the method.  Every scaling is by a power of two, which is exact in
bf16, so the oracle sees exactly the values the GPU reads.
"""
import pytest
import torch

import oracle
from bwd_sparse_mqa_gb300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu


def _inputs(D, seed, q_scale=1.0, do_scale=1.0):
    x = inputs.custom(2, 40, 300, 128, D, 200, recipe="causal_masked10", seed=seed)
    x["q"] = (x["q"].float() * q_scale).to(torch.bfloat16)
    x["do"] = (x["do"].float() * do_scale).to(torch.bfloat16)
    return x


def _check_bwd(x, deterministic):
    g = P.to_dev(x)
    o, lse = P.run_fwd(g)
    kw = dict(return_dsink=True)
    if deterministic:
        kw.update(deterministic=True, return_dkv_accum_dtype=True)
    dq, dkv, dsink = P.run_bwd(g, o, lse, g["do"], **kw)
    dq_ref, dkv_ref, dsink_ref, _ = oracle.bwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"],
                                               x["do"])
    errs = {"dq": P.assert_close("dq", dq, dq_ref), "dkv": P.assert_close("dkv", dkv, dkv_ref),
            "dsink": P.assert_close("dsink", dsink, dsink_ref)}
    if deterministic:
        dq2, dkv2, _ = P.run_bwd(g, o, lse, g["do"], **kw)
        assert torch.equal(dkv, dkv2) and torch.equal(dq, dq2)
    return errs


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("do_scale", [2.0 ** -20, 2.0 ** -30, 2.0 ** 10],
                         ids=["dO_2^-20", "dO_2^-30", "dO_2^10"])
@pytest.mark.parametrize("D", [512, 64])
def test_gradient_scale(D, do_scale, deterministic):
    """dO scaled by 2^-20, 2^-30 (gradient-sized) and 2^10."""
    print(_check_bwd(_inputs(D, 31, do_scale=do_scale), deterministic))


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "det"])
@pytest.mark.parametrize("q_scale", [8.0, 16.0], ids=["q_x8", "q_x16"])
@pytest.mark.parametrize("D", [512, 64])
def test_peaked_softmax(D, q_scale, deterministic):
    """q scaled by 8 and 16: logits with standard deviation 8 and 16 (natural
    units), so each row's softmax is dominated by a few slots."""
    x = _inputs(D, 32, q_scale=q_scale)
    print(P.check_full(x, bwd=False))
    print(_check_bwd(x, deterministic))


@pytest.mark.parametrize("D", [512, 64])
def test_flat_softmax_and_tiny_gradients(D):
    """q scaled by 2^-20 (every logit ~0: the softmax is flat, the partial
    scores are tiny) together with dO scaled by 2^-24."""
    x = _inputs(D, 33, q_scale=2.0 ** -20, do_scale=2.0 ** -24)
    print(P.check_full(x, bwd=False))
    print(_check_bwd(x, False))
