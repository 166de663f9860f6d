"""Checks that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an oracle library handle (the real one, or a
deliberately broken copy in the mutation test) and raises AssertionError if
the oracle disagrees with:
  - torch's own attention (scaled_dot_product_attention in fp64) and autograd
    on the dense problem the sparse one reduces to when the indices list every
    key row (the sink is an extra key column whose logit is sink_h and whose
    value row is zero);
  - central finite differences of L = sum(O * dO) in fp64;
  - closed forms (one valid slot; all slots masked);
  - invariants (slot order, masked slot == dropped slot, token-subset
    linearity of dKV, duplicated slot == duplicated key row);
  - brute force over every topk-subset of a tiny key set.
The definition being pinned is that of the sparse MQA forward/backward
interfaces on the DeepSeek-V4 kernel pages (tilelang_sparse_mla_fwd,
tilelang_sparse_mla_bwd): per-head sink in the softmax denominator, slots
outside [0, S_kv) masked, log2 LSE, gradients for q and the shared kv.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle

LN2 = math.log(2.0)


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def _perm_rows(S_kv, k, rng):
    return rng.permutation(S_kv)[:k]


def _dense_torch(q, kv, sink, idx, scale, need_grad=False, dout=None):
    """Reference built from torch primitives: per token, gather the listed
    valid key rows, append a zero key/value whose logit is forced to sink_h
    through an additive mask, and call scaled_dot_product_attention (fp64).
    Returns O [B,S,H,D], LSE2 [B,S,H] and, with need_grad, the gradients of
    sum(O*dO) w.r.t. q, kv and sink (torch autograd)."""
    B, S, H, D = q.shape
    S_kv = kv.shape[1]
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=need_grad)
    kvt = torch.tensor(kv, dtype=torch.float64, requires_grad=need_grad)
    st = torch.tensor(sink, dtype=torch.float64, requires_grad=need_grad)
    outs, lses = [], []
    for b in range(B):
        for s in range(S):
            rows = [int(r) for r in idx[b, s] if 0 <= r < S_kv]
            keys = kvt[b, rows] if rows else kvt.new_zeros((0, D))
            keys = torch.cat([keys, kvt.new_zeros((1, D))], 0)            # [n+1, D]
            n1 = keys.shape[0]
            qq = qt[b, s].unsqueeze(1).unsqueeze(0)                          # [1,H,1,D]
            kk = keys.unsqueeze(0).unsqueeze(0).expand(1, H, n1, D)
            mask = torch.cat([kvt.new_zeros((H, n1 - 1)), st.unsqueeze(1)], 1)
            mask = mask.unsqueeze(0).unsqueeze(2)                            # [1,H,1,n+1]
            o = F.scaled_dot_product_attention(qq, kk, kk, attn_mask=mask, scale=scale)
            outs.append(o[0, :, 0, :])
            logits = torch.cat([scale * (qt[b, s] @ keys[:-1].T), st.unsqueeze(1)], 1)
            lses.append(torch.logsumexp(logits, dim=1) / LN2)
    O = torch.stack(outs).reshape(B, S, H, D)
    L2 = torch.stack(lses).reshape(B, S, H)
    grads = None
    if need_grad:
        loss = (O * torch.tensor(dout, dtype=torch.float64)).sum()
        gq, gkv, gs = torch.autograd.grad(loss, [qt, kvt, st])
        grads = (gq.numpy(), gkv.numpy(), gs.numpy())
    return O.detach().numpy(), L2.detach().numpy(), grads


def _close(a, b, rtol=1e-9, atol=1e-11, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    if not np.allclose(a, b, rtol=rtol, atol=atol):
        err = np.max(np.abs(a - b))
        raise AssertionError(f"{what}: max abs err {err:.3e}")


def _tiny(rng, B=2, S=3, S_kv=5, H=2, D=4, topk=4, masked=True):
    q = _rand((B, S, H, D), rng)
    kv = _rand((B, S_kv, D), rng)
    sink = _rand((H,), rng)
    dout = _rand((B, S, H, D), rng)
    idx = np.stack([np.stack([_perm_rows(S_kv, topk, rng) for _ in range(S)]) for _ in range(B)])
    idx = idx.astype(np.int32)
    if masked:
        idx[0, 1, 0] = -1
        idx[B - 1, S - 1, topk - 1] = S_kv
    return q, kv, sink, idx, dout


def pin_dense_sdpa_fwd(lib):
    """All key rows listed, none masked: O and LSE2 equal torch's dense
    attention with the sink column."""
    rng = np.random.default_rng(11)
    B, S, S_kv, H, D = 2, 3, 6, 3, 5
    q, kv, sink = _rand((B, S, H, D), rng), _rand((B, S_kv, D), rng), _rand((H,), rng)
    idx = np.stack([np.stack([rng.permutation(S_kv) for _ in range(S)]) for _ in range(B)])
    idx = idx.astype(np.int32)
    for scale in (D ** -0.5, 0.37):
        o, l2 = oracle.fwd_f64(q, kv, sink, idx, sm_scale=scale, lib=lib)
        O, L2, _ = _dense_torch(q, kv, sink, idx, scale)
        _close(o.reshape(O.shape), O, what="dense O")
        _close(l2.reshape(L2.shape), L2, what="dense LSE2")


def pin_dense_autograd_bwd(lib):
    """dQ, dKV and dsink equal torch autograd through the dense reference,
    including masked slots and several tokens hitting the same rows."""
    rng = np.random.default_rng(12)
    q, kv, sink, idx, dout = _tiny(rng, B=2, S=4, S_kv=5, H=3, D=4, topk=4)
    scale = 0.45
    dq, dkv, dsink, _ = oracle.bwd_f64(q, kv, sink, idx, dout, sm_scale=scale, lib=lib)
    _, _, (gq, gkv, gs) = _dense_torch(q, kv, sink, idx, scale, need_grad=True, dout=dout)
    _close(dq.reshape(gq.shape), gq, what="dQ vs autograd")
    _close(dkv, gkv, what="dKV vs autograd")
    _close(dsink, gs, what="dsink vs autograd")


def pin_permutation(lib):
    """Reordering a token's slots changes nothing."""
    rng = np.random.default_rng(13)
    q, kv, sink, idx, dout = _tiny(rng)
    perm = idx.copy()
    for b in range(perm.shape[0]):
        for s in range(perm.shape[1]):
            perm[b, s] = perm[b, s][rng.permutation(perm.shape[2])]
    o1, l1 = oracle.fwd_f64(q, kv, sink, idx, lib=lib)
    o2, l2 = oracle.fwd_f64(q, kv, sink, perm, lib=lib)
    _close(o1, o2, what="perm O")
    _close(l1, l2, what="perm LSE")
    r1 = oracle.bwd_f64(q, kv, sink, idx, dout, lib=lib)
    r2 = oracle.bwd_f64(q, kv, sink, perm, dout, lib=lib)
    for a, b, n in zip(r1, r2, ("dQ", "dKV", "dsink", "Delta")):
        _close(a, b, what=f"perm {n}")


def pin_masked_equals_dropped(lib):
    """Slots with indices -1, -7, S_kv or S_kv+3 act as if absent: a row of
    topk=6 with four masked slots equals the same two valid slots at topk=2."""
    rng = np.random.default_rng(14)
    B, S, S_kv, H, D = 1, 2, 5, 2, 3
    q, kv, sink = _rand((B, S, H, D), rng), _rand((B, S_kv, D), rng), _rand((H,), rng)
    dout = _rand((B, S, H, D), rng)
    small = np.array([[[3, 1], [0, 4]]], np.int32)
    big = np.array([[[-1, 3, S_kv, -7, 1, S_kv + 3], [0, S_kv, -1, 4, -2, S_kv + 9]]], np.int32)
    a = oracle.fwd_f64(q, kv, sink, small, lib=lib)
    b = oracle.fwd_f64(q, kv, sink, big, lib=lib)
    _close(a[0], b[0], what="masked O")
    _close(a[1], b[1], what="masked LSE")
    ga = oracle.bwd_f64(q, kv, sink, small, dout, lib=lib)
    gb = oracle.bwd_f64(q, kv, sink, big, dout, lib=lib)
    for x, y, n in zip(ga, gb, ("dQ", "dKV", "dsink", "Delta")):
        _close(x, y, what=f"masked {n}")


def pin_all_masked(lib):
    """No valid slot: O = 0, LSE2 = sink_h / ln 2, dQ = 0, nothing reaches
    dKV, dsink = 0 (Delta = <dO, 0> = 0)."""
    rng = np.random.default_rng(15)
    B, S, S_kv, H, D = 1, 2, 4, 3, 5
    q, kv, sink = _rand((B, S, H, D), rng), _rand((B, S_kv, D), rng), _rand((H,), rng) * 3
    dout = _rand((B, S, H, D), rng)
    idx = np.array([[[-1, S_kv, -3], [2, -1, S_kv]]], np.int32)
    o, l2 = oracle.fwd_f64(q, kv, sink, idx, lib=lib)
    _close(o[0], np.zeros((H, D)), what="all-masked O")
    _close(l2[0], sink / LN2, what="all-masked LSE2")
    dq, dkv, dsink, delta = oracle.bwd_f64(q, kv, sink, idx, dout, tokens=[0], lib=lib)
    _close(dq, np.zeros_like(dq), what="all-masked dQ")
    _close(dkv, np.zeros_like(dkv), what="all-masked dKV")
    _close(dsink, np.zeros_like(dsink), what="all-masked dsink")
    _close(delta, np.zeros_like(delta), what="all-masked Delta")


def pin_single_slot_closed_form(lib):
    """One valid slot r: z = c<q,k_r>, O = k_r * sigmoid(z - sink) and
    LSE2 = log2(e^z + e^sink)."""
    rng = np.random.default_rng(16)
    B, S, S_kv, H, D = 1, 1, 4, 3, 6
    q, kv, sink = _rand((B, S, H, D), rng), _rand((B, S_kv, D), rng), _rand((H,), rng)
    r, scale = 2, 0.31
    idx = np.array([[[-1, r, S_kv]]], np.int32)
    o, l2 = oracle.fwd_f64(q, kv, sink, idx, sm_scale=scale, lib=lib)
    for h in range(H):
        z = scale * float(np.dot(q[0, 0, h], kv[0, r]))
        sig = 1.0 / (1.0 + math.exp(-(z - sink[h])))
        _close(o[0, h], kv[0, r] * sig, what="one-slot O")
        _close(l2[0, h], math.log2(math.exp(z) + math.exp(sink[h])), what="one-slot LSE2")


def pin_sink_limit(lib):
    """sink -> -1e4 removes the sink: plain softmax over the valid logits
    (torch.softmax) and LSE2 = log2 sum exp."""
    rng = np.random.default_rng(17)
    q, kv, _, idx, _ = _tiny(rng, B=1, S=3, S_kv=6, H=2, D=4, topk=5)
    sink = np.full((2,), -1e4)
    o, l2 = oracle.fwd_f64(q, kv, sink, idx, lib=lib)
    D = q.shape[3]
    for s in range(3):
        rows = [int(r) for r in idx[0, s] if 0 <= r < 6]
        K = torch.tensor(kv[0, rows])
        for h in range(2):
            z = (torch.tensor(q[0, s, h]) @ K.T) * D ** -0.5
            p = torch.softmax(z, 0)
            _close(o[s, h], (p @ K).numpy(), what="no-sink O")
            _close(l2[s, h], float(torch.logsumexp(z, 0)) / LN2, what="no-sink LSE2")


def pin_finite_differences(lib):
    """dQ, dKV and dsink equal central differences of L = sum(O * dO)."""
    rng = np.random.default_rng(18)
    q, kv, sink, idx, dout = _tiny(rng, B=2, S=3, S_kv=4, H=2, D=3, topk=3)
    scale = 0.52
    dq, dkv, dsink, _ = oracle.bwd_f64(q, kv, sink, idx, dout, sm_scale=scale, lib=lib)

    def loss(qq, kk, ss):
        o, _ = oracle.fwd_f64(qq, kk, ss, idx, sm_scale=scale, lib=lib)
        return float(np.sum(o.reshape(dout.shape) * dout))

    eps = 1e-6
    for arr, grad, name in ((q, dq.reshape(q.shape), "dQ"), (kv, dkv, "dKV"),
                            (sink, dsink, "dsink")):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[i] += eps
            minus[i] -= eps
            args_p = [q, kv, sink]
            args_m = [q, kv, sink]
            k = {"dQ": 0, "dKV": 1, "dsink": 2}[name]
            args_p[k], args_m[k] = plus, minus
            fd[i] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        _close(grad, fd, rtol=1e-6, atol=1e-8, what=f"{name} vs finite differences")


def pin_bruteforce_subsets(lib):
    """Every 3-subset of 6 key rows, in a random slot order, equals dense
    attention restricted to that subset (torch SDPA)."""
    rng = np.random.default_rng(19)
    B, S, S_kv, H, D = 1, 4, 6, 2, 3
    q, kv, sink = _rand((B, S, H, D), rng), _rand((B, S_kv, D), rng), _rand((H,), rng)
    for subset in itertools.combinations(range(S_kv), 3):
        idx = np.stack([rng.permutation(np.array(subset)) for _ in range(S)])[None].astype(np.int32)
        o, l2 = oracle.fwd_f64(q, kv, sink, idx, lib=lib)
        O, L2, _ = _dense_torch(q, kv, sink, idx, D ** -0.5)
        _close(o.reshape(O.shape), O, what=f"subset {subset} O")
        _close(l2.reshape(L2.shape), L2, what=f"subset {subset} LSE2")


def pin_token_subset_linearity(lib):
    """dKV over all tokens = sum of the per-token dKVs, and a run with dO
    zeroed outside a token sample gives the sample's dKV (the restricted-dO
    check used for full-size parity)."""
    rng = np.random.default_rng(20)
    q, kv, sink, idx, dout = _tiny(rng, B=2, S=4, S_kv=5, H=2, D=3, topk=3)
    _, dkv_all, dsink_all, _ = oracle.bwd_f64(q, kv, sink, idx, dout, lib=lib)
    acc = np.zeros_like(dkv_all)
    acc_s = np.zeros_like(dsink_all)
    for t in range(8):
        _, d1, s1, _ = oracle.bwd_f64(q, kv, sink, idx, dout, tokens=[t], lib=lib)
        acc += d1
        acc_s += s1
    _close(acc, dkv_all, what="dKV linearity")
    _close(acc_s, dsink_all, what="dsink linearity")
    sample = [1, 6]
    restricted = np.zeros_like(dout)
    for t in sample:
        restricted[t // 4, t % 4] = dout[t // 4, t % 4]
    _, dkv_r, _, _ = oracle.bwd_f64(q, kv, sink, idx, restricted, lib=lib)
    _, dkv_s, _, _ = oracle.bwd_f64(q, kv, sink, idx, dout, tokens=sample, lib=lib)
    _close(dkv_r, dkv_s, what="restricted dO")


def pin_duplicate_slot(lib):
    """A row listed twice counts twice: equals dense attention over a key
    list that holds that row twice; its dKV gets both slots' terms."""
    rng = np.random.default_rng(21)
    B, S, S_kv, H, D = 1, 1, 4, 2, 3
    q, kv, sink = _rand((B, S, H, D), rng), _rand((B, S_kv, D), rng), _rand((H,), rng)
    dout = _rand((B, S, H, D), rng)
    idx = np.array([[[2, 0, 2]]], np.int32)
    o, l2 = oracle.fwd_f64(q, kv, sink, idx, lib=lib)
    O, L2, grads = _dense_torch(q, kv, sink, idx, D ** -0.5, need_grad=True, dout=dout)
    _close(o.reshape(O.shape), O, what="dup O")
    _close(l2.reshape(L2.shape), L2, what="dup LSE2")
    dq, dkv, dsink, _ = oracle.bwd_f64(q, kv, sink, idx, dout, lib=lib)
    _close(dq.reshape(q.shape), grads[0], what="dup dQ")
    _close(dkv, grads[1], what="dup dKV")


def pin_bf16_entry_matches_f64(lib):
    """The bf16 entry points read bf16 bits exactly: on bf16-representable
    inputs they equal the fp64 entry points bit for bit."""
    rng = np.random.default_rng(22)
    q, kv, sink, idx, dout = _tiny(rng)
    tq = torch.tensor(q).to(torch.bfloat16)
    tkv = torch.tensor(kv).to(torch.bfloat16)
    tdo = torch.tensor(dout).to(torch.bfloat16)
    ts = torch.tensor(sink, dtype=torch.float32)
    o1, l1 = oracle.fwd(tq, tkv, ts, torch.tensor(idx), lib=lib)
    o2, l2 = oracle.fwd_f64(tq.double().numpy(), tkv.double().numpy(), ts.double().numpy(), idx,
                            lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2), "bf16 entry differs from fp64"
    g1 = oracle.bwd(tq, tkv, ts, torch.tensor(idx), tdo, lib=lib)
    g2 = oracle.bwd_f64(tq.double().numpy(), tkv.double().numpy(), ts.double().numpy(), idx,
                        tdo.double().numpy(), lib=lib)
    for a, b in zip(g1, g2):
        assert np.allclose(a, b, rtol=1e-14, atol=1e-15), "bf16 bwd entry differs from fp64"


def pin_linear_in_dout(lib):
    """The backward is linear in dO: scaling dO by a power of two scales dQ,
    dKV, dsink and Delta by that power (fp64 rounding commutes with it), so
    the oracle has no absolute floor or offset at small or large gradient
    magnitudes."""
    rng = np.random.default_rng(23)
    q, kv, sink, idx, dout = _tiny(rng, B=2, S=3, S_kv=6, H=3, D=5, topk=4)
    base = oracle.bwd_f64(q, kv, sink, idx, dout, lib=lib)
    for alpha in (2.0 ** -30, 2.0 ** -20, 2.0 ** 10):
        got = oracle.bwd_f64(q, kv, sink, idx, dout * alpha, lib=lib)
        # dQ and Delta are per-token sums in a fixed order: exact.  dKV and
        # dsink are summed over tokens with OpenMP atomics in a varying order,
        # so they agree to a few fp64 roundings.
        for name, a, b in zip(("dq", "delta"), (got[0], got[3]), (base[0], base[3])):
            assert np.array_equal(a, b * alpha), f"{name} not linear in dO at {alpha}"
        for name, a, b in zip(("dkv", "dsink"), got[1:3], base[1:3]):
            _close(a / alpha, b, rtol=1e-12, atol=1e-14 * float(np.max(np.abs(b))),
                   what=f"{name} linear in dO at {alpha}")
    # And it is really a function of dO: a different dO changes dQ.
    other = oracle.bwd_f64(q, kv, sink, idx, dout[::-1].copy(), lib=lib)
    assert not np.allclose(other[0], base[0]), "dQ does not depend on dO"


def pin_query_scale_equals_sm_scale(lib):
    """Scaling q by a power of two is the same as scaling sm_scale by it:
    the logits c*q.k are equal, so O and LSE agree exactly, dKV agrees
    exactly (c*g*(a q) = (a c)*g*q), and dQ(q, a c) = a dQ(a q, c)."""
    rng = np.random.default_rng(24)
    q, kv, sink, idx, dout = _tiny(rng, B=1, S=4, S_kv=6, H=2, D=4, topk=5)
    c, a = 0.37, 8.0
    o1, l1 = oracle.fwd_f64(q * a, kv, sink, idx, c, lib=lib)
    o2, l2 = oracle.fwd_f64(q, kv, sink, idx, c * a, lib=lib)
    _close(o1, o2, rtol=1e-13, atol=1e-15, what="O under q scaling")
    _close(l1, l2, rtol=1e-13, atol=1e-15, what="LSE under q scaling")
    dq1, dkv1, ds1, _ = oracle.bwd_f64(q * a, kv, sink, idx, dout, c, lib=lib)
    dq2, dkv2, ds2, _ = oracle.bwd_f64(q, kv, sink, idx, dout, c * a, lib=lib)
    _close(dq2, a * dq1, rtol=1e-12, atol=1e-14, what="dQ under q scaling")
    _close(dkv1, dkv2, rtol=1e-12, atol=1e-14, what="dKV under q scaling")
    _close(ds1, ds2, rtol=1e-12, atol=1e-14, what="dsink under q scaling")


# ---------------------------------------------------------------------------
# Lightning-indexer backward (tilelang_indexer_bwd page; the reading
# score[t,j] = sum_h w[t,h] ReLU(<q[t,h], k[idx[t,j]]>) is not given by the
# page, so these pins tie the oracle to that reading, not to the page).
# ---------------------------------------------------------------------------
def _tiny_indexer(rng, S=3, H=3, D=5, S_kv=6, topk=4):
    q = _rand((S, H, D), rng)
    w = _rand((S, H), rng)
    k = _rand((S_kv, D), rng)
    g = _rand((S, topk), rng)
    idx = np.stack([_perm_rows(S_kv, topk, rng) for _ in range(S)]).astype(np.int32)
    idx[0, 1] = -1          # masked by -1
    idx[S - 1, 0] = S_kv    # masked by S_kv
    idx[1, 2] = idx[1, 0]   # a row listed twice
    return q, w, k, idx, g


def pin_indexer_dense_autograd(lib):
    """dq equals torch autograd (fp64) of sum_{t,j} g[t,j] score[t,j], the
    score built from torch's matmul and relu over the listed rows."""
    rng = np.random.default_rng(30)
    q, w, k, idx, g = _tiny_indexer(rng)
    S, H, D = q.shape
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k, dtype=torch.float64)
    loss = qt.new_zeros(())
    for t in range(S):
        js = [j for j in range(idx.shape[1]) if 0 <= idx[t, j] < k.shape[0]]
        rows = kt[[int(idx[t, j]) for j in js]]
        logits = qt[t] @ rows.T                                     # [H, n]
        score = (torch.tensor(w[t])[:, None] * torch.relu(logits)).sum(0)
        loss = loss + (torch.tensor(g[t, js]) * score).sum()
    (gq,) = torch.autograd.grad(loss, [qt])
    dq, slack = oracle.indexer_bwd_f64(q, w, k, idx, g, lib=lib)
    _close(dq, gq.numpy(), what="indexer dq vs autograd")
    assert np.all(slack == 0.0), "slack without an ambiguity band"


def pin_indexer_finite_differences(lib):
    """Central differences of F(q) = sum g * score(q), with the oracle's own
    score function, match dq (no logit near the ReLU kink)."""
    rng = np.random.default_rng(31)
    q, w, k, idx, g = _tiny_indexer(rng, S=2, H=2, D=4, S_kv=5, topk=3)
    dq, _ = oracle.indexer_bwd_f64(q, w, k, idx, g, lib=lib)

    def F(qq):
        return float(np.sum(g * oracle.indexer_scores_f64(qq, w, k, idx, lib=lib)))

    logits = np.einsum("thd,rd->thr", q, k)
    assert np.min(np.abs(logits)) > 1e-4, "a logit sits on the kink; pick another seed"
    eps = 1e-6
    fd = np.zeros_like(q)
    for pos in np.ndindex(*q.shape):
        qp, qm = q.copy(), q.copy()
        qp[pos] += eps
        qm[pos] -= eps
        fd[pos] = (F(qp) - F(qm)) / (2 * eps)
    _close(dq, fd, rtol=1e-6, atol=1e-8, what="indexer dq vs finite differences")


def pin_indexer_closed_forms(lib):
    """All gates closed (every logit negative) gives dq = 0; all gates open
    (every logit positive) gives the plain weighted sum
    w[t,h] * sum_{valid j} g[t,j] k_j."""
    rng = np.random.default_rng(32)
    q, w, k, idx, g = _tiny_indexer(rng)
    qn, kp = -np.abs(q), np.abs(k)
    dq, _ = oracle.indexer_bwd_f64(qn, w, kp, idx, g, lib=lib)
    assert np.all(dq == 0.0), "closed gates must give dq = 0"
    qp = np.abs(q)
    dq, _ = oracle.indexer_bwd_f64(qp, w, kp, idx, g, lib=lib)
    want = np.zeros_like(q)
    for t in range(q.shape[0]):
        for j in range(idx.shape[1]):
            if 0 <= idx[t, j] < k.shape[0]:
                want[t] += np.outer(w[t], g[t, j] * kp[idx[t, j]])
    _close(dq, want, what="indexer all-open closed form")


def pin_indexer_invariants(lib):
    """Masked slots equal dropped slots; permuting the slots together with
    grad_scores changes nothing; dq is linear in grad_scores and in the
    weights (power-of-two scalings are exact)."""
    rng = np.random.default_rng(33)
    q, w, k, idx, g = _tiny_indexer(rng, S=2, H=2, D=3, S_kv=7, topk=5)
    idx[0] = [3, -1, 6, 7, 1]
    idx[1] = [2, 4, -5, 0, 5]
    base, _ = oracle.indexer_bwd_f64(q, w, k, idx, g, lib=lib)
    keep = [[0, 2, 4], [0, 1, 3, 4]]
    for t in range(2):
        sub_idx = idx[t:t + 1, keep[t]].copy()
        sub_g = g[t:t + 1, keep[t]].copy()
        d1, _ = oracle.indexer_bwd_f64(q[t:t + 1], w[t:t + 1], k, sub_idx, sub_g, lib=lib)
        _close(d1[0], base[t], what="indexer masked == dropped")
    perm = rng.permutation(idx.shape[1])
    d2, _ = oracle.indexer_bwd_f64(q, w, k, idx[:, perm].copy(), g[:, perm].copy(), lib=lib)
    _close(d2, base, what="indexer slot permutation")
    for a in (2.0 ** -20, 2.0 ** 7):
        d3, _ = oracle.indexer_bwd_f64(q, w, k, idx, g * a, lib=lib)
        assert np.array_equal(d3, base * a), "indexer dq not linear in grad_scores"
        d4, _ = oracle.indexer_bwd_f64(q, w * a, k, idx, g, lib=lib)
        assert np.array_equal(d4, base * a), "indexer dq not linear in weights"


def pin_indexer_ambiguity_slack(lib):
    """With an ambiguity band, every pair left out is accounted for: the
    plain dq lies within slack of the banded one, and some slack is used."""
    rng = np.random.default_rng(34)
    q, w, k, idx, g = _tiny_indexer(rng, S=4, H=3, D=6, S_kv=8, topk=6)
    plain, s0 = oracle.indexer_bwd_f64(q, w, k, idx, g, lib=lib)
    banded, s1 = oracle.indexer_bwd_f64(q, w, k, idx, g, amb=0.3, lib=lib)
    assert np.all(s0 == 0.0) and np.max(s1) > 0.0
    assert np.all(np.abs(plain - banded) <= s1 + 1e-12), "slack does not cover the band"


def pin_indexer_bf16_entry(lib):
    """The bf16 entry point reads the same values as the fp64 one."""
    rng = np.random.default_rng(35)
    q, w, k, idx, g = _tiny_indexer(rng)
    tq = torch.tensor(q).to(torch.bfloat16)
    tk = torch.tensor(k).to(torch.bfloat16)
    tw = torch.tensor(w, dtype=torch.float32)
    tg = torch.tensor(g, dtype=torch.float32)
    a, _ = oracle.indexer_bwd(tq, tw, tk, torch.tensor(idx), tg, lib=lib)
    b, _ = oracle.indexer_bwd_f64(tq.double().numpy(), tw.double().numpy(), tk.double().numpy(),
                                  idx, tg.double().numpy(), lib=lib)
    assert np.array_equal(a, b), "indexer bf16 entry differs from fp64"


ALL_PINS = [
    pin_dense_sdpa_fwd,
    pin_dense_autograd_bwd,
    pin_permutation,
    pin_masked_equals_dropped,
    pin_all_masked,
    pin_single_slot_closed_form,
    pin_sink_limit,
    pin_finite_differences,
    pin_bruteforce_subsets,
    pin_token_subset_linearity,
    pin_duplicate_slot,
    pin_bf16_entry_matches_f64,
    pin_linear_in_dout,
    pin_query_scale_equals_sm_scale,
    pin_indexer_dense_autograd,
    pin_indexer_finite_differences,
    pin_indexer_closed_forms,
    pin_indexer_invariants,
    pin_indexer_ambiguity_slack,
    pin_indexer_bf16_entry,
]
