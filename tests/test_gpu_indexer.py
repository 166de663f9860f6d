"""Lightning-indexer backward (tilelang_indexer_bwd page) on the GPU against
the fp64 oracle, element by element.

Tolerance: max(|dq_gpu - dq_ref| - slack) <= 2e-2 * max|dq_ref|, where the
oracle leaves out of dq_ref every (token, head, slot) whose logit <q,k_j>
lies within 2^-12 * sum_d |q_d k_jd| of 0 and reports the size of its term
as slack: there the ReLU gate is decided by rounding (the GPU forms the
logit in fp32 on the tensor core), and either decision is correct.  Pairs
outside that band must match exactly in their gate.
"""
import numpy as np
import pytest
import torch

import oracle
from bwd_sparse_mqa_gb300 import batched_indexer_bwd, indexer_bwd_interface, inputs
from bwd_sparse_mqa_gb300.api import device_status

pytestmark = pytest.mark.gpu

AMB = 2.0 ** -12
TOL = 2e-2


def _err(gpu, ref, slack):
    a = gpu.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    over = np.maximum(np.abs(a - ref) - slack, 0.0)
    return float(np.max(over)) / max(float(np.max(np.abs(ref))), 1e-30)


def _single(x, b):
    """Batch element b of the per-element layouts, on the GPU."""
    return {k: v[b].contiguous().cuda() for k, v in x.items()}


def _check_single(x, tokens=None):
    errs = []
    for b in range(x["index_q"].shape[0]):
        g = _single(x, b)
        dq = indexer_bwd_interface(g["index_q"], g["weights"], g["index_k"], g["topk_indices"],
                                   g["grad_scores"])
        torch.cuda.synchronize()
        assert device_status() == 0
        ref, slack = oracle.indexer_bwd(x["index_q"][b], x["weights"][b], x["index_k"][b],
                                        x["topk_indices"][b], x["grad_scores"][b],
                                        tokens=tokens, amb=AMB)
        got = dq if tokens is None else dq[torch.as_tensor(tokens, device=dq.device)]
        e = _err(got, ref, slack)
        assert np.isfinite(e) and e <= TOL, f"dq: rel err {e:.3e} > {TOL}"
        errs.append(e)
    return errs


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("H", [64, 128, 48, 1])
def test_indexer_every_token(H, D):
    """Several 64-slot blocks and a ragged tail (topk = 150), 10% masked
    slots, every token, for H on and off the 16-row grid."""
    x = inputs.indexer_custom(2, 40, 200, H, D, 150, recipe="causal_masked10", seed=70 + H)
    print(_check_single(x))


def test_indexer_masked_rows_duplicates_and_closed_gates():
    x = inputs.indexer_custom(1, 16, 90, 64, 128, 100, seed=71)
    idx = x["topk_indices"]
    idx[0, 2] = -1            # every slot masked: dq = 0
    idx[0, 3, :] = 90         # masked by S_kv
    idx[0, 5, :12] = 7        # one key row listed twelve times
    x["index_q"][0, 9] = -x["index_q"][0, 9].abs()    # token 9: every gate closed
    x["index_k"][0] = x["index_k"][0].abs()
    print(_check_single(x))
    g = _single(x, 0)
    dq = indexer_bwd_interface(g["index_q"], g["weights"], g["index_k"], g["topk_indices"],
                               g["grad_scores"])
    assert torch.all(dq[2] == 0) and torch.all(dq[3] == 0) and torch.all(dq[9] == 0)


def test_batched_layout():
    """The page's batched layouts, all batch elements in one launch, against
    the oracle run per element."""
    x = inputs.indexer_custom(3, 24, 130, 64, 128, 96, recipe="causal_masked10", seed=72,
                              batched_layout=True)
    g = {k: v.cuda() for k, v in x.items()}
    dq = batched_indexer_bwd(g["index_q"], g["weights"], g["index_k"], g["topk_indices"],
                             g["grad_scores"])
    torch.cuda.synchronize()
    assert device_status() == 0
    ref, slack = oracle.indexer_bwd_batched(x["index_q"], x["weights"], x["index_k"],
                                            x["topk_indices"], x["grad_scores"], amb=AMB)
    e = _err(dq, ref, slack)
    assert e <= TOL, f"batched dq: rel err {e:.3e}"
    # Element b of the batched call equals the single-element call on it.
    for b in range(3):
        d1 = indexer_bwd_interface(g["index_q"][:, b].contiguous(), g["weights"][:, b].contiguous(),
                                   g["index_k"][:, b].contiguous(),
                                   g["topk_indices"][b].contiguous(),
                                   g["grad_scores"][b].contiguous())
        assert torch.equal(d1, dq[:, b])


def test_indexer_full_size_sampled():
    """The H=64 D=128 topk=2048 S=8192 indexer workload, run whole, checked
    on a seeded sample of 256 tokens (plus the first, the topk-th and the
    last)."""
    from tests import _parity as P
    cfg = inputs.INDEXER_CONFIGS[0]
    x = inputs.make_indexer_inputs(cfg, device="cuda")
    tokens = P.sample_tokens(1, cfg.S, cfg.topk, 256, seed=120)
    xc = {k: v.cpu() for k, v in x.items()}
    print(_check_single(xc, tokens=tokens))
