"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerances (stated for this op, applied per tensor): max |gpu - ref| <=
2e-2 * max |ref| for O, dQ, dKV and dsink, and <= 1e-4 * max |ref| for the log2 LSE,
where ref is the fp64 oracle on the same bf16 inputs.  dsink_h is a sum over
tokens of -p_sink * Delta whose terms may cancel, and the GPU forms each Delta
from the bf16 O it is given (the backward interface takes o), so each term
carries O's rounding; where the oracle's per-token terms are at hand, the
dsink scale is therefore max_h sum_t |p_sink * Delta| rather than max |ref|
(the same whenever the terms share a sign).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bwd_sparse_mqa_gb300 import sparse_mqa_bwd_interface, sparse_mqa_fwd_interface
from bwd_sparse_mqa_gb300.api import device_status

TOL = {"o": 2e-2, "dq": 2e-2, "dkv": 2e-2, "dsink": 2e-2, "lse": 1e-4}


def rel_err(gpu, ref) -> float:
    a = gpu.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    denom = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(a - ref))) / denom


def assert_close(name, gpu, ref, tol=None, scale=None):
    e = rel_err(gpu, ref)
    if scale is not None:
        e *= max(float(np.max(np.abs(ref))), 1e-30) / max(scale, float(np.max(np.abs(ref))), 1e-30)
    t = TOL[name] if tol is None else tol
    assert np.isfinite(e) and e <= t, f"{name}: rel err {e:.3e} > {t:.1e}"
    return e


def dsink_scale(attn_sink, lse2_ref, delta_ref) -> float:
    """max over heads of sum over tokens |p_sink * Delta|, from the oracle's
    log2 LSE and Delta ([tokens, H] after flattening), p_sink =
    2^(sink_h log2(e) - lse2)."""
    sink = np.asarray(attn_sink.detach().cpu() if hasattr(attn_sink, "detach") else attn_sink,
                      dtype=np.float64)
    H = sink.shape[0]
    lse2 = np.asarray(lse2_ref, dtype=np.float64).reshape(-1, H)
    delta = np.asarray(delta_ref, dtype=np.float64).reshape(-1, H)
    p_sink = np.exp2(sink[None, :] / np.log(2.0) - lse2)
    return float(np.max(np.sum(np.abs(p_sink * delta), axis=0)))


def to_dev(x: dict, dev="cuda") -> dict:
    return {k: (None if v is None else v.to(dev)) for k, v in x.items()}


def sample_tokens(B: int, S: int, topk: int, n: int, seed: int, extra=()) -> np.ndarray:
    """Seeded token sample that always includes s = 0, topk-1, topk, S-1 of
    every batch element plus any `extra` flat ids."""
    rng = np.random.default_rng(seed)
    must = set()
    for b in range(B):
        for s in (0, topk - 1, topk, S - 1):
            if 0 <= s < S:
                must.add(b * S + s)
    must.update(int(e) for e in extra)
    rest = rng.choice(B * S, size=min(n, B * S), replace=False)
    out = sorted(must | set(int(r) for r in rest))
    return np.array(out, dtype=np.int64)


def run_fwd(g: dict, sm_scale=None, **kw):
    o, lse = sparse_mqa_fwd_interface(g["q"], g["kv"], g["attn_sink"], g["topk_idxs"],
                                      sm_scale=sm_scale, **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    return o, lse


def run_bwd(g: dict, o, lse, dout, sm_scale=None, **kw):
    out = sparse_mqa_bwd_interface(g["q"], g["kv"], g["attn_sink"], o, dout, g["topk_idxs"],
                                   lse, sm_scale=sm_scale, **kw)
    torch.cuda.synchronize()
    assert device_status() == 0
    return out


def check_full(x: dict, sm_scale=None, bwd=True):
    """Every token against the oracle (small shapes)."""
    g = to_dev(x)
    o, lse = run_fwd(g, sm_scale)
    o_ref, lse_ref = oracle.fwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], sm_scale)
    errs = {"o": assert_close("o", o, o_ref), "lse": assert_close("lse", lse, lse_ref)}
    if bwd:
        dq, dkv, dsink = run_bwd(g, o, lse, g["do"], sm_scale, return_dsink=True)
        dq_ref, dkv_ref, dsink_ref, delta_ref = oracle.bwd(x["q"], x["kv"], x["attn_sink"],
                                                           x["topk_idxs"], x["do"], sm_scale)
        errs["dq"] = assert_close("dq", dq, dq_ref)
        errs["dkv"] = assert_close("dkv", dkv, dkv_ref)
        errs["dsink"] = assert_close("dsink", dsink, dsink_ref,
                                     scale=dsink_scale(x["attn_sink"], lse_ref, delta_ref))
    return errs


def check_sampled(g: dict, tokens: np.ndarray, do_fwd=True, do_bwd=True):
    """Full-size GPU run, oracle on a token sample.  dKV and dsink use a second
    backward whose dO is zero outside the sample, so the sample alone feeds
    them (Delta, and with it each token's dsink term, is 0 elsewhere)."""
    B, S = g["q"].shape[:2]
    q_cpu = g["q"].cpu()
    kv_cpu = g["kv"].cpu()
    sink_cpu = g["attn_sink"].cpu()
    idx_cpu = g["topk_idxs"].cpu()
    errs = {}
    o, lse = run_fwd(g)
    if do_fwd:
        o_ref, lse_ref = oracle.fwd(q_cpu, kv_cpu, sink_cpu, idx_cpu, tokens=tokens)
        o_s = o.reshape(B * S, *o.shape[2:])[torch.as_tensor(tokens, device=o.device)]
        l_s = lse.reshape(B * S, -1)[torch.as_tensor(tokens, device=o.device)]
        errs["o"] = assert_close("o", o_s, o_ref)
        errs["lse"] = assert_close("lse", l_s, lse_ref)
    if do_bwd:
        dout = g["do"]
        keep = torch.zeros(B * S, dtype=torch.bool, device=dout.device)
        keep[torch.as_tensor(tokens, device=dout.device)] = True
        d_r = torch.where(keep.view(B, S, 1, 1), dout, torch.zeros_like(dout))
        dq, dkv, dsink = run_bwd(g, o, lse, d_r, return_dsink=True)
        do_cpu = dout.cpu()
        dq_ref, dkv_ref, dsink_ref, delta_ref = oracle.bwd(q_cpu, kv_cpu, sink_cpu, idx_cpu,
                                                           do_cpu, tokens=tokens)
        if not do_fwd:
            _, lse_ref = oracle.fwd(q_cpu, kv_cpu, sink_cpu, idx_cpu, tokens=tokens)
        dq_s = dq.reshape(B * S, *dq.shape[2:])[torch.as_tensor(tokens, device=dq.device)]
        errs["dq"] = assert_close("dq", dq_s, dq_ref)
        errs["dkv"] = assert_close("dkv", dkv, dkv_ref)
        errs["dsink"] = assert_close("dsink", dsink, dsink_ref,
                                     scale=dsink_scale(sink_cpu, lse_ref, delta_ref))
    return errs
