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
that most slot blocks are full."""
import numpy as np
import pytest
import torch

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
