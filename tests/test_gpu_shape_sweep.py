"""A seeded sweep over shapes the C ABI accepts: every case runs the forward
and the backward on every token against the fp64 oracle (tolerances of
tests/_parity.py).  The shapes are drawn once from a fixed generator, so the
list is the same on every run: batch 1-3, up to 64 queries, 1-600 key rows,
any head count 1-128, D = 64 or 512, topk 1-520 (from a single slot to a
ragged ninth 64-slot block), every index recipe, with or without an explicit
sm_scale.  Short rows (topk above the causal row length) pad with -1, so
those cases hold masked tails and tokens without a valid slot; half of the
cases replace the causal rows by long ones (distinct uniform rows of all of
S_kv, 10 % of the slots masked by -1 or S_kv, the rest in random order), so
that most slot blocks are full.  Every fourth shape also runs the
deterministic backward with fp32 dKV, and 16 more shapes (D = 64 or 128)
run the lightning-indexer backward in the batched layout."""
import numpy as np
import pytest
import torch

import oracle
from bwd_sparse_mqa_gb300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu

_RECIPES = ["causal_uniform", "causal_masked10", "causal_recent512", "causal_window64",
            "hot4096_masked10"]


def _shapes(n=32, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        S = int(rng.integers(1, 65))
        S_kv = int(rng.integers(1, 601))
        H = int(rng.integers(1, 129))
        D = 512 if i % 2 == 0 else 64
        topk = int(rng.integers(1, 521))
        recipe = _RECIPES[int(rng.integers(0, len(_RECIPES)))]
        sm_scale = None if rng.random() < 0.5 else float(rng.uniform(0.02, 0.2))
        dense = bool(i % 4 >= 2)
        out.append((B, S, S_kv, H, D, topk, recipe, sm_scale, 100 + i, dense))
    return out


def _dense_rows(B, S, S_kv, topk, seed):
    """int32 [B, S, topk]: per token min(topk, S_kv) distinct rows drawn
    uniformly from [0, S_kv), the rest -1, then 10 % of all slots masked
    (half by -1, half by S_kv), slots shuffled."""
    gen = torch.Generator().manual_seed(seed)
    k = min(topk, S_kv)
    keys = torch.rand((B, S, S_kv), generator=gen)
    rows = torch.argsort(keys, dim=2)[:, :, :k].to(torch.int32)
    if k < topk:
        rows = torch.cat([rows, torch.full((B, S, topk - k), -1, dtype=torch.int32)], dim=2)
    hit = torch.rand((B, S, topk), generator=gen) < 0.10
    coin = torch.rand((B, S, topk), generator=gen) < 0.5
    repl = torch.where(coin, torch.full_like(rows, -1), torch.full_like(rows, S_kv))
    rows = torch.where(hit, repl, rows)
    perm = torch.argsort(torch.rand((B, S, topk), generator=gen), dim=2)
    return torch.gather(rows, 2, perm).contiguous()


_CASES = _shapes()


@pytest.mark.parametrize("case", _CASES, ids=[
    f"B{c[0]}_S{c[1]}_Skv{c[2]}_H{c[3]}_D{c[4]}_k{c[5]}_{'dense' if c[9] else c[6]}"
    for c in _CASES])
def test_random_shape_every_token(case):
    B, S, S_kv, H, D, topk, recipe, sm_scale, seed, dense = case
    x = inputs.custom(B, S, S_kv, H, D, topk, recipe=recipe, seed=seed)
    if dense:
        x["topk_idxs"] = _dense_rows(B, S, S_kv, topk, seed)
    print(P.check_full(x, sm_scale=sm_scale))


@pytest.mark.parametrize("case", _CASES[::4], ids=[
    f"B{c[0]}_S{c[1]}_Skv{c[2]}_H{c[3]}_D{c[4]}_k{c[5]}" for c in _CASES[::4]])
def test_random_shape_deterministic_fp32_dkv(case):
    """Every fourth shape through the deterministic backward with fp32 dKV
    output: dQ, dKV and dsink against the oracle, and a second call
    bit-identical."""
    B, S, S_kv, H, D, topk, recipe, sm_scale, seed, dense = case
    x = inputs.custom(B, S, S_kv, H, D, topk, recipe=recipe, seed=seed)
    if dense:
        x["topk_idxs"] = _dense_rows(B, S, S_kv, topk, seed)
    g = P.to_dev(x)
    o, lse = P.run_fwd(g, sm_scale)
    kw = dict(return_dkv_accum_dtype=True, return_dsink=True, deterministic=True)
    dq, dkv, dsink = P.run_bwd(g, o, lse, g["do"], sm_scale, **kw)
    dq2, dkv2, dsink2 = P.run_bwd(g, o, lse, g["do"], sm_scale, **kw)
    assert dkv.dtype == torch.float32
    assert torch.equal(dq, dq2) and torch.equal(dkv, dkv2) and torch.equal(dsink, dsink2)
    _, lse_ref = oracle.fwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], sm_scale)
    dq_ref, dkv_ref, dsink_ref, delta_ref = oracle.bwd(x["q"], x["kv"], x["attn_sink"],
                                                       x["topk_idxs"], x["do"], sm_scale)
    P.assert_close("dq", dq, dq_ref)
    P.assert_close("dkv", dkv, dkv_ref)
    P.assert_close("dsink", dsink, dsink_ref,
                   scale=P.dsink_scale(x["attn_sink"], lse_ref, delta_ref))


def _indexer_shapes(n=16, seed=2025):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        S = int(rng.integers(1, 65))
        S_kv = int(rng.integers(1, 601))
        H = int(rng.integers(1, 129))
        D = 128 if i % 2 == 0 else 64
        topk = int(rng.integers(1, 521))
        recipe = _RECIPES[int(rng.integers(0, len(_RECIPES)))]
        out.append((B, S, S_kv, H, D, topk, recipe, 200 + i, bool(i % 4 >= 2)))
    return out


_ICASES = _indexer_shapes()


@pytest.mark.parametrize("case", _ICASES, ids=[
    f"B{c[0]}_S{c[1]}_Skv{c[2]}_H{c[3]}_D{c[4]}_k{c[5]}_{'dense' if c[8] else c[6]}"
    for c in _ICASES])
def test_random_indexer_shape_every_token(case):
    """The lightning-indexer backward, batched layout, every token against
    the oracle run per batch element (gate-ambiguity band and tolerance of
    tests/test_gpu_indexer.py)."""
    from bwd_sparse_mqa_gb300 import batched_indexer_bwd
    from bwd_sparse_mqa_gb300.api import device_status
    from tests.test_gpu_indexer import AMB, TOL, _err
    B, S, S_kv, H, D, topk, recipe, seed, dense = case
    x = inputs.indexer_custom(B, S, S_kv, H, D, topk, recipe=recipe, seed=seed,
                              batched_layout=True)
    if dense:
        x["topk_indices"] = _dense_rows(B, S, S_kv, topk, seed)
    g = {k: v.cuda() for k, v in x.items()}
    dq = batched_indexer_bwd(g["index_q"], g["weights"], g["index_k"], g["topk_indices"],
                             g["grad_scores"])
    torch.cuda.synchronize()
    assert device_status() == 0
    ref, slack = oracle.indexer_bwd_batched(x["index_q"], x["weights"], x["index_k"],
                                            x["topk_indices"], x["grad_scores"], amb=AMB)
    e = _err(dq, ref, slack)
    assert np.isfinite(e) and e <= TOL, f"batched dq: rel err {e:.3e} > {TOL}"
