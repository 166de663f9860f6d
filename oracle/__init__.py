"""fp64 CPU oracle for top-k sparse MQA with an attention sink, and for the
lightning-indexer backward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product package
``bwd_sparse_mqa_gb300`` never does, and this package never imports it.

The arithmetic lives in ``smqa_oracle.c`` (plain C, double precision, OpenMP
over tokens); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  Inputs are the raw bf16 bit patterns (uint16) of the same
tensors the CUDA path reads, so both sides see identical values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsmqa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.smqa_oracle_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P, i64, P, P]
    lib.smqa_oracle_fwd.restype = ctypes.c_int
    lib.smqa_oracle_bwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P, i64,
                                    P, P, P, P]
    lib.smqa_oracle_bwd.restype = ctypes.c_int
    lib.smqa_oracle_fwd_f64.argtypes = lib.smqa_oracle_fwd.argtypes
    lib.smqa_oracle_fwd_f64.restype = ctypes.c_int
    lib.smqa_oracle_bwd_f64.argtypes = lib.smqa_oracle_bwd.argtypes
    lib.smqa_oracle_bwd_f64.restype = ctypes.c_int
    lib.smqa_oracle_indexer_bwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, i64, f64,
                                            P, P]
    lib.smqa_oracle_indexer_bwd.restype = ctypes.c_int
    lib.smqa_oracle_indexer_bwd_f64.argtypes = lib.smqa_oracle_indexer_bwd.argtypes
    lib.smqa_oracle_indexer_bwd_f64.restype = ctypes.c_int
    lib.smqa_oracle_indexer_scores_f64.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P, i64, P]
    lib.smqa_oracle_indexer_scores_f64.restype = ctypes.c_int
    lib.smqa_oracle_num_threads.argtypes = []
    lib.smqa_oracle_num_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.  A ``path`` loads
    that exact file instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _u16(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bits."""
    if hasattr(a, "detach"):
        import torch
        t = a.detach().to("cpu").contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        raise TypeError(f"expected bf16 tensor, got {t.dtype}")
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bits, got {a.dtype}")
    return a


def _np(a, dtype) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").contiguous().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads(lib: ctypes.CDLL | None = None) -> int:
    return int((lib or load()).smqa_oracle_num_threads())


def fwd(q, kv, attn_sink, topk_idxs, sm_scale: float | None = None, tokens=None, lib=None):
    """O (fp64 [n,H,D]) and log2-LSE (fp64 [n,H]) for the selected flat tokens.

    q [B,S,H,D] bf16, kv [B,S_kv,D] bf16, attn_sink [H] fp32,
    topk_idxs [B,S,topk] int32; ``tokens`` = flat ids b*S+s (None = all).
    """
    q16, kv16 = _u16(q), _u16(kv)
    sink = _np(attn_sink, np.float32)
    idx = _np(topk_idxs, np.int32)
    B, S, H, D = q16.shape
    S_kv = kv16.shape[1]
    topk = idx.shape[2]
    scale = D ** -0.5 if sm_scale is None else float(sm_scale)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = B * S if tok is None else len(tok)
    o = np.empty((n, H, D), np.float64)
    lse2 = np.empty((n, H), np.float64)
    rc = (lib or load()).smqa_oracle_fwd(_ptr(q16), _ptr(kv16), _ptr(sink), _ptr(idx), B, S, S_kv,
                                         H, D, topk, scale, _ptr(tok), n, _ptr(o), _ptr(lse2))
    if rc != 0:
        raise ValueError("oracle fwd rejected its arguments")
    return o, lse2


def bwd(q, kv, attn_sink, topk_idxs, dout, sm_scale: float | None = None, tokens=None, lib=None):
    """dQ (fp64 [n,H,D]), dKV (fp64 [B,S_kv,D], from the selected tokens
    only), dsink (fp64 [H]) and Delta (fp64 [n,H])."""
    q16, kv16, do16 = _u16(q), _u16(kv), _u16(dout)
    sink = _np(attn_sink, np.float32)
    idx = _np(topk_idxs, np.int32)
    B, S, H, D = q16.shape
    S_kv = kv16.shape[1]
    topk = idx.shape[2]
    scale = D ** -0.5 if sm_scale is None else float(sm_scale)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = B * S if tok is None else len(tok)
    dq = np.empty((n, H, D), np.float64)
    dkv = np.zeros((B, S_kv, D), np.float64)
    dsink = np.zeros((H,), np.float64)
    delta = np.empty((n, H), np.float64)
    rc = (lib or load()).smqa_oracle_bwd(_ptr(q16), _ptr(kv16), _ptr(sink), _ptr(idx), _ptr(do16),
                                         B, S, S_kv, H, D, topk, scale, _ptr(tok), n, _ptr(dq),
                                         _ptr(dkv), _ptr(dsink), _ptr(delta))
    if rc != 0:
        raise ValueError("oracle bwd rejected its arguments")
    return dq, dkv, dsink, delta


def fwd_f64(q, kv, attn_sink, topk_idxs, sm_scale: float | None = None, tokens=None, lib=None):
    """The forward on fp64 numpy inputs (q [B,S,H,D], kv [B,S_kv,D], sink [H])."""
    q64, kv64 = _np(q, np.float64), _np(kv, np.float64)
    sink = _np(attn_sink, np.float64)
    idx = _np(topk_idxs, np.int32)
    B, S, H, D = q64.shape
    S_kv = kv64.shape[1]
    topk = idx.shape[2]
    scale = D ** -0.5 if sm_scale is None else float(sm_scale)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = B * S if tok is None else len(tok)
    o = np.empty((n, H, D), np.float64)
    lse2 = np.empty((n, H), np.float64)
    rc = (lib or load()).smqa_oracle_fwd_f64(_ptr(q64), _ptr(kv64), _ptr(sink), _ptr(idx), B, S,
                                             S_kv, H, D, topk, scale, _ptr(tok), n, _ptr(o),
                                             _ptr(lse2))
    if rc != 0:
        raise ValueError("oracle fwd rejected its arguments")
    return o, lse2


def bwd_f64(q, kv, attn_sink, topk_idxs, dout, sm_scale: float | None = None, tokens=None,
            lib=None):
    """The backward on fp64 numpy inputs; returns (dq, dkv, dsink, delta)."""
    q64, kv64, do64 = _np(q, np.float64), _np(kv, np.float64), _np(dout, np.float64)
    sink = _np(attn_sink, np.float64)
    idx = _np(topk_idxs, np.int32)
    B, S, H, D = q64.shape
    S_kv = kv64.shape[1]
    topk = idx.shape[2]
    scale = D ** -0.5 if sm_scale is None else float(sm_scale)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = B * S if tok is None else len(tok)
    dq = np.empty((n, H, D), np.float64)
    dkv = np.zeros((B, S_kv, D), np.float64)
    dsink = np.zeros((H,), np.float64)
    delta = np.empty((n, H), np.float64)
    rc = (lib or load()).smqa_oracle_bwd_f64(_ptr(q64), _ptr(kv64), _ptr(sink), _ptr(idx),
                                             _ptr(do64), B, S, S_kv, H, D, topk, scale, _ptr(tok),
                                             n, _ptr(dq), _ptr(dkv), _ptr(dsink), _ptr(delta))
    if rc != 0:
        raise ValueError("oracle bwd rejected its arguments")
    return dq, dkv, dsink, delta


# ---------------------------------------------------------------------------
# Lightning-indexer backward (tilelang_indexer_bwd page; reading in the C
# source: score[t,j] = sum_h w[t,h] ReLU(<q[t,h], k[idx[t,j]]>), dq only).
# ---------------------------------------------------------------------------
def _tok(tokens, n_all):
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    return tok, (n_all if tok is None else len(tok))


def indexer_bwd(index_q, weights, index_k, topk_indices, grad_scores, tokens=None,
                amb: float = 0.0, lib=None):
    """dq (fp64 [n,H,D]) and its slack (fp64 [n,H,D], see the C source) for
    one batch element: index_q [S,H,D] bf16, weights [S,H] fp32, index_k
    [S_kv,D] bf16, topk_indices [S,topk] int32, grad_scores [S,topk] fp32."""
    q16, k16 = _u16(index_q), _u16(index_k)
    w = _np(weights, np.float32)
    idx = _np(topk_indices, np.int32)
    g = _np(grad_scores, np.float32)
    S, H, D = q16.shape
    S_kv = k16.shape[0]
    topk = idx.shape[1]
    tok, n = _tok(tokens, S)
    dq = np.empty((n, H, D), np.float64)
    slack = np.empty((n, H, D), np.float64)
    rc = (lib or load()).smqa_oracle_indexer_bwd(_ptr(q16), _ptr(w), _ptr(k16), _ptr(idx),
                                                 _ptr(g), S, S_kv, H, D, topk, _ptr(tok), n,
                                                 float(amb), _ptr(dq), _ptr(slack))
    if rc != 0:
        raise ValueError("oracle indexer bwd rejected its arguments")
    return dq, slack


def indexer_bwd_f64(index_q, weights, index_k, topk_indices, grad_scores, tokens=None,
                    amb: float = 0.0, lib=None):
    """The indexer backward on fp64 numpy inputs; returns (dq, slack)."""
    q, w, k = _np(index_q, np.float64), _np(weights, np.float64), _np(index_k, np.float64)
    idx, g = _np(topk_indices, np.int32), _np(grad_scores, np.float64)
    S, H, D = q.shape
    S_kv, topk = k.shape[0], idx.shape[1]
    tok, n = _tok(tokens, S)
    dq = np.empty((n, H, D), np.float64)
    slack = np.empty((n, H, D), np.float64)
    rc = (lib or load()).smqa_oracle_indexer_bwd_f64(_ptr(q), _ptr(w), _ptr(k), _ptr(idx),
                                                     _ptr(g), S, S_kv, H, D, topk, _ptr(tok), n,
                                                     float(amb), _ptr(dq), _ptr(slack))
    if rc != 0:
        raise ValueError("oracle indexer bwd rejected its arguments")
    return dq, slack


def indexer_scores_f64(index_q, weights, index_k, topk_indices, tokens=None, lib=None):
    """score[t,j] (fp64 [n,topk]) of the reading, on fp64 numpy inputs."""
    q, w, k = _np(index_q, np.float64), _np(weights, np.float64), _np(index_k, np.float64)
    idx = _np(topk_indices, np.int32)
    S, H, D = q.shape
    S_kv, topk = k.shape[0], idx.shape[1]
    tok, n = _tok(tokens, S)
    out = np.empty((n, topk), np.float64)
    rc = (lib or load()).smqa_oracle_indexer_scores_f64(_ptr(q), _ptr(w), _ptr(k), _ptr(idx),
                                                        S, S_kv, H, D, topk, _ptr(tok), n,
                                                        _ptr(out))
    if rc != 0:
        raise ValueError("oracle indexer scores rejected its arguments")
    return out


def indexer_bwd_batched(index_q, weights, index_k, topk_indices, grad_scores, tokens=None,
                        amb: float = 0.0, lib=None):
    """The batched layouts of `batched_indexer_bwd`: index_q [S,B,H,D],
    weights [S,B,H], index_k [S_kv,B,D], topk_indices [B,S,topk],
    grad_scores [B,S,topk].  Runs the single-element oracle on each batch
    element (the page's function loops over the batch the same way) and
    returns dq and slack as fp64 [S,B,H,D] (tokens: per-element positions s,
    then [n,B,H,D])."""
    q = index_q.detach().cpu()
    S, B, H, D = q.shape
    n = S if tokens is None else len(tokens)
    dq = np.empty((n, B, H, D), np.float64)
    slack = np.empty((n, B, H, D), np.float64)
    for b in range(B):
        d1, s1 = indexer_bwd(q[:, b].contiguous(), weights.detach().cpu()[:, b].contiguous(),
                             index_k.detach().cpu()[:, b].contiguous(),
                             topk_indices.detach().cpu()[b].contiguous(),
                             grad_scores.detach().cpu()[b].contiguous(), tokens=tokens, amb=amb,
                             lib=lib)
        dq[:, b], slack[:, b] = d1, s1
    return dq, slack
