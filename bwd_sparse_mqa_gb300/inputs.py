"""Seeded synthetic inputs for top-k sparse MQA (shared by the tests, the
benchmark and the smoke check; holds none of the method's arithmetic).

The workloads follow the shapes, dtypes and index structures of the sparse
MQA forward/backward interfaces on the DeepSeek-V4 kernel pages of NeMo
AutoModel (tilelang_sparse_mla_fwd / tilelang_sparse_mla_bwd): q [B,S,H,D],
kv [B,S_kv,D] and dO [B,S,H,D] bf16 drawn N(0,1), attn_sink [H] fp32 N(0,1),
topk_idxs [B,S,topk] int32.  The pages publish no dataset; every tensor here
is synthetic.

Index recipes (query position i = s, keys j in [0, S_kv)):
  causal_uniform      distinct j <= i, uniform; rows with fewer than topk
                      candidates take all of them and pad with -1
  causal_masked10     causal_uniform, then 10% of all slots replaced by -1 or
                      S_kv (fair coin), both outside [0, S_kv) and so masked
  causal_recent512    the whole window [i-511, i] (as far as it exists) plus
                      uniform distinct j <= i outside it
  hot4096_masked10    one seeded set of 4096 hot rows; every row draws topk
                      distinct rows from it with no causal limit, then 10% of
                      the slots are set to -1
  causal_window64     the window [i-63, i] always, plus uniform distinct
                      j <= i outside it
Within a row the used slots are in random order and pads (-1) come last,
except that the masked10 recipes scatter their masked slots at random.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

__all__ = ["SMQAConfig", "CONFIGS", "make_inputs", "make_indices", "by_name",
           "INDEXER_CONFIGS", "make_indexer_inputs", "indexer_custom"]


@dataclasses.dataclass(frozen=True)
class SMQAConfig:
    name: str
    B: int
    S: int
    S_kv: int
    H: int
    D: int
    topk: int
    recipe: str
    passes: str          # "fwd", "fwd+bwd" or "bwd"
    seed: int
    device: str = "cpu"  # where the seeded generator runs

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def describe(self) -> str:
        return (f"B={self.B} S={self.S} S_kv={self.S_kv} H={self.H} D={self.D} "
                f"topk={self.topk} idx={self.recipe}")


# The five workloads: a small one the oracle finishes on every token, a forward
# one with masked slots, the H=128 D=512 topk=2048 headline one, a dKV scatter
# stress one and a long-context one.
CONFIGS = [
    SMQAConfig("small_h16_d64_k32", 1, 128, 128, 16, 64, 32, "causal_uniform", "fwd+bwd", 0),
    SMQAConfig("fwd_h64_d512_k512", 2, 4096, 4096, 64, 512, 512, "causal_masked10", "fwd", 1,
               "cuda"),
    SMQAConfig("h128_d512_k2048_s8192", 1, 8192, 8192, 128, 512, 2048, "causal_recent512",
               "fwd+bwd", 2, "cuda"),
    SMQAConfig("hot4096_h128_d512_k2048", 1, 8192, 8192, 128, 512, 2048, "hot4096_masked10",
               "bwd", 3, "cuda"),
    SMQAConfig("long_h128_d512_k2048_s32768", 1, 32768, 32768, 128, 512, 2048,
               "causal_window64", "fwd+bwd", 4, "cuda"),
]


def by_name(name: str) -> SMQAConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def _shuffle_valid_first(idx: torch.Tensor, gen: torch.Generator) -> torch.Tensor:
    """Random order among slots >= 0, slots equal to -1 moved to the end."""
    keys = torch.rand(idx.shape, generator=gen, device=idx.device)
    keys = keys.masked_fill(idx < 0, 2.0)
    perm = torch.argsort(keys, dim=1)
    return torch.gather(idx, 1, perm)


def _causal_rows(S: int, S_kv: int, topk: int, window: int, gen: torch.Generator,
                 device) -> torch.Tensor:
    """Distinct causal indices: for query i take the `window` newest keys
    j in (i-window, i] first, then uniform distinct j <= i; pad with -1."""
    out = torch.empty((S, topk), dtype=torch.int32, device=device)
    chunk = max(1, min(S, (1 << 26) // max(S_kv, 1)))
    j = torch.arange(S_kv, device=device)
    for r0 in range(0, S, chunk):
        rows = torch.arange(r0, min(S, r0 + chunk), device=device)
        keys = torch.rand((rows.numel(), S_kv), generator=gen, device=device)
        causal = j[None, :] <= rows[:, None]
        if window > 0:
            recent = causal & (j[None, :] > rows[:, None] - window)
            keys = torch.where(recent, keys - 1.0, keys)
        keys = keys.masked_fill(~causal, 3.0)
        k_eff = min(topk, S_kv)
        vals, sel = torch.topk(keys, k_eff, dim=1, largest=False, sorted=True)
        sel = sel.to(torch.int32).masked_fill(vals >= 3.0, -1)
        if k_eff < topk:
            pad = torch.full((rows.numel(), topk - k_eff), -1, dtype=torch.int32, device=device)
            sel = torch.cat([sel, pad], dim=1)
        out[r0:r0 + rows.numel()] = _shuffle_valid_first(sel, gen)
    return out


def _mask_fraction(idx: torch.Tensor, frac: float, S_kv: int, gen: torch.Generator,
                   coin: bool) -> torch.Tensor:
    hit = torch.rand(idx.shape, generator=gen, device=idx.device) < frac
    if coin:
        heads = torch.rand(idx.shape, generator=gen, device=idx.device) < 0.5
        repl = torch.where(heads, torch.full_like(idx, -1), torch.full_like(idx, S_kv))
    else:
        repl = torch.full_like(idx, -1)
    return torch.where(hit, repl, idx)


def make_indices(recipe: str, B: int, S: int, S_kv: int, topk: int, gen: torch.Generator,
                 device) -> torch.Tensor:
    """int32 [B, S, topk] indices following one of the recipes above."""
    per_b = []
    for _ in range(B):
        if recipe == "causal_uniform":
            r = _causal_rows(S, S_kv, topk, 0, gen, device)
        elif recipe == "causal_masked10":
            r = _causal_rows(S, S_kv, topk, 0, gen, device)
            valid = r >= 0
            r = torch.where(valid, _mask_fraction(r, 0.10, S_kv, gen, coin=True), r)
        elif recipe == "causal_recent512":
            r = _causal_rows(S, S_kv, topk, 512, gen, device)
        elif recipe == "causal_window64":
            r = _causal_rows(S, S_kv, topk, 64, gen, device)
        elif recipe == "hot4096_masked10":
            n_hot = min(4096, S_kv)
            hot = torch.randperm(S_kv, generator=gen, device=device)[:n_hot].to(torch.int32)
            k_eff = min(topk, n_hot)
            r = torch.empty((S, topk), dtype=torch.int32, device=device)
            chunk = max(1, (1 << 24) // n_hot)
            for r0 in range(0, S, chunk):
                n = min(S, r0 + chunk) - r0
                keys = torch.rand((n, n_hot), generator=gen, device=device)
                sel = torch.topk(keys, k_eff, dim=1, largest=False).indices
                rows = hot[sel]
                if k_eff < topk:
                    rows = torch.cat([rows, torch.full((n, topk - k_eff), -1, dtype=torch.int32,
                                                       device=device)], dim=1)
                r[r0:r0 + n] = rows
            r = _mask_fraction(r, 0.10, S_kv, gen, coin=False)
        else:
            raise ValueError(f"unknown index recipe {recipe!r}")
        per_b.append(r)
    return torch.stack(per_b, 0).contiguous()


def make_inputs(cfg: SMQAConfig, device: Optional[str] = None, with_do: bool = True) -> dict:
    """Seeded q, kv, attn_sink, dO (bf16/fp32) and topk_idxs (int32), drawn
    in that order from one generator on ``device`` (default: the config's)."""
    dev = torch.device(device or cfg.device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    q = torch.randn((cfg.B, cfg.S, cfg.H, cfg.D), generator=gen, device=dev).to(torch.bfloat16)
    kv = torch.randn((cfg.B, cfg.S_kv, cfg.D), generator=gen, device=dev).to(torch.bfloat16)
    sink = torch.randn((cfg.H,), generator=gen, device=dev, dtype=torch.float32)
    dout = None
    if with_do:
        dout = torch.randn((cfg.B, cfg.S, cfg.H, cfg.D), generator=gen,
                           device=dev).to(torch.bfloat16)
    idx = make_indices(cfg.recipe, cfg.B, cfg.S, cfg.S_kv, cfg.topk, gen, dev)
    return {"q": q.contiguous(), "kv": kv.contiguous(), "attn_sink": sink.contiguous(),
            "do": None if dout is None else dout.contiguous(), "topk_idxs": idx}


def custom(B: int, S: int, S_kv: int, H: int, D: int, topk: int, recipe: str = "causal_uniform",
           seed: int = 0, device: str = "cpu") -> dict:
    """Inputs for an arbitrary shape (tests use this for edge cases)."""
    cfg = SMQAConfig("custom", B, S, S_kv, H, D, topk, recipe, "fwd+bwd", seed, device)
    return make_inputs(cfg)


# ---------------------------------------------------------------------------
# Lightning-indexer backward (tilelang_indexer_bwd page): index_q [S,H,D]
# bf16, weights [S,H] fp32, index_k [S_kv,D] bf16, topk_indices [S,topk]
# int32, grad_scores [S,topk] fp32 per batch element.  The page measures
# nothing; the workload uses the DeepSeek-V4 indexer's head count and width
# (64 heads of 128) with the attention workloads' sequence length and topk.
# ---------------------------------------------------------------------------
INDEXER_CONFIGS = [
    SMQAConfig("indexer_h64_d128_k2048_s8192", 1, 8192, 8192, 64, 128, 2048, "causal_uniform",
               "indexer_bwd", 5, "cuda"),
]


def indexer_by_name(name: str) -> SMQAConfig:
    for c in INDEXER_CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def make_indexer_inputs(cfg: SMQAConfig, device: Optional[str] = None,
                        batched_layout: bool = False) -> dict:
    """Seeded indexer inputs drawn in the order index_q, index_k, weights,
    grad_scores, topk_indices (all N(0,1) but the indices).  Per-element
    layouts ([B,S,H,D], [B,S_kv,D], [B,S,H]) unless ``batched_layout``, which
    gives the page's batched ones: index_q [S,B,H,D], weights [S,B,H],
    index_k [S_kv,B,D]; topk_indices and grad_scores are [B,S,topk] in both."""
    dev = torch.device(device or cfg.device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    q = torch.randn((cfg.B, cfg.S, cfg.H, cfg.D), generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn((cfg.B, cfg.S_kv, cfg.D), generator=gen, device=dev).to(torch.bfloat16)
    w = torch.randn((cfg.B, cfg.S, cfg.H), generator=gen, device=dev, dtype=torch.float32)
    g = torch.randn((cfg.B, cfg.S, cfg.topk), generator=gen, device=dev, dtype=torch.float32)
    idx = make_indices(cfg.recipe, cfg.B, cfg.S, cfg.S_kv, cfg.topk, gen, dev)
    if batched_layout:
        q = q.permute(1, 0, 2, 3)
        k = k.permute(1, 0, 2)
        w = w.permute(1, 0, 2)
    return {"index_q": q.contiguous(), "weights": w.contiguous(), "index_k": k.contiguous(),
            "topk_indices": idx.contiguous(), "grad_scores": g.contiguous()}


def indexer_custom(B: int, S: int, S_kv: int, H: int, D: int, topk: int,
                   recipe: str = "causal_uniform", seed: int = 0, device: str = "cpu",
                   batched_layout: bool = False) -> dict:
    cfg = SMQAConfig("indexer_custom", B, S, S_kv, H, D, topk, recipe, "indexer_bwd", seed, device)
    return make_indexer_inputs(cfg, batched_layout=batched_layout)
