"""The persistent main kernels: every CTA pair (every CTA for D = 64) works
through many tokens, taken from a counter (D = 512) or in a fixed order
(D = 64), as one sequence of slot blocks whose barrier phases run on across
token boundaries.  These cases give each pair several tokens and put the
boundary cases in the middle of its sequence -- tokens without any valid
slot (no MMA at all: nothing loaded, O / dQ written as zeros), tokens of a
single valid slot, full tokens next to empty ones -- and compare every
token with the fp64 oracle (forward and backward), then repeat the call to
check that a second launch on the same workspace gives the same bits."""
import numpy as np
import pytest
import torch

from bwd_sparse_mqa_gb300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu


def _boundary_mix(x: dict, seed: int) -> dict:
    """Every third token of a run fully masked (-1 or S_kv), every seventh
    of a single valid slot at a random position; the rest as drawn."""
    idx = x["topk_idxs"]
    B, S, K = idx.shape
    S_kv = x["kv"].shape[1]
    rng = np.random.default_rng(seed)
    for b in range(B):
        for s in range(S):
            r = rng.random()
            if r < 0.2:
                idx[b, s, :] = -1
            elif r < 0.3:
                idx[b, s, :] = S_kv
            elif r < 0.45:
                keep = int(rng.integers(0, K))
                row = int(rng.integers(0, S_kv))
                idx[b, s, :] = -1
                idx[b, s, keep] = row
    # Runs of empty tokens, so a pair meets several in a row.
    idx[0, 40:52, :] = -1
    return x


@pytest.mark.parametrize("D,H,K,seed", [(512, 32, 130, 31), (512, 128, 64, 32), (64, 48, 100, 33)])
def test_many_tokens_per_cta_with_empty_and_single_slot_tokens(D, H, K, seed):
    # 2 x 480 tokens: more than 76 pairs (or 152+ CTAs) can hold, so every
    # pair handles several tokens.
    x = _boundary_mix(inputs.custom(2, 480, 200, H, D, K, recipe="causal_masked10", seed=seed), seed)
    print(P.check_full(x))
    g = P.to_dev(x)
    o1, lse1 = P.run_fwd(g)
    o2, lse2 = P.run_fwd(g)
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    dq1, _ = P.run_bwd(g, o1, lse1, g["do"])
    dq2, _ = P.run_bwd(g, o1, lse1, g["do"])
    assert torch.equal(dq1, dq2)
    empty = (x["topk_idxs"] < 0) | (x["topk_idxs"] >= x["kv"].shape[1])
    empty_tok = empty.all(dim=-1).cuda()
    assert int(empty_tok.sum()) > 20
    assert torch.all(o1[empty_tok] == 0) and torch.all(dq1[empty_tok] == 0)


def test_every_token_empty():
    """No token has a valid slot: no MMA runs anywhere; O and dQ are zero,
    the LSE is the sink's, dKV is zero."""
    x = inputs.custom(1, 300, 64, 16, 512, 64, seed=34)
    x["topk_idxs"][:] = -1
    g = P.to_dev(x)
    o, lse = P.run_fwd(g)
    assert torch.all(o == 0)
    sink2 = g["attn_sink"] / np.log(2.0)
    assert torch.allclose(lse[0], sink2.expand_as(lse[0]), rtol=1e-5, atol=1e-6)
    dq, dkv = P.run_bwd(g, o, lse, g["do"])
    assert torch.all(dq == 0) and torch.all(dkv == 0)
    assert P.device_status() == 0
