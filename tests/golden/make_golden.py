"""Writes tests/golden/tiny_oracle.json: a tiny, fully spelled-out case and the
fp64 oracle's outputs for it.

The sparse MQA pages (DeepSeek-V4 kernel API pages of NeMo AutoModel) print no
worked example, so no stored value here comes from the pages.  This fixture is
a regression anchor written ONLY by the oracle (this script imports nothing
else that computes): a later change to the oracle's arithmetic that moves these
numbers must say, in its commit message, which reading of the pages justifies
it.  Inputs are small exact binary fractions so that they are the same in
bf16, fp32 and fp64.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def case():
    # B=1, S=3, S_kv=4, H=2, D=4, topk=3; slots include -1 and S_kv (masked).
    q = np.array([[[[0.5, -1.0, 0.25, 2.0], [1.5, 0.0, -0.75, 0.5]],
                   [[-0.5, 0.75, 1.0, -1.25], [0.0, 2.0, 0.5, -0.5]],
                   [[1.0, 1.0, -1.0, 0.25], [-2.0, 0.5, 0.0, 1.0]]]])
    kv = np.array([[[1.0, 0.5, -0.5, 0.0], [-1.0, 0.25, 0.75, 1.5],
                    [0.5, -1.5, 1.0, 0.25], [2.0, 0.0, -0.25, -1.0]]])
    sink = np.array([0.5, -1.0])
    idx = np.array([[[0, -1, 2], [3, 1, 4], [2, 0, 1]]], dtype=np.int32)
    dout = np.array([[[[1.0, 0.0, -0.5, 0.25], [0.5, 1.0, 0.0, -1.0]],
                      [[-0.25, 0.5, 1.0, 0.0], [2.0, -1.0, 0.5, 0.5]],
                      [[0.0, 0.75, -1.0, 1.0], [1.0, 1.0, 1.0, -0.5]]]])
    return q, kv, sink, idx, dout


def main():
    q, kv, sink, idx, dout = case()
    scale = 0.5
    o, lse2 = oracle.fwd_f64(q, kv, sink, idx, sm_scale=scale)
    dq, dkv, dsink, delta = oracle.bwd_f64(q, kv, sink, idx, dout, sm_scale=scale)
    out = {
        "about": "tiny sparse MQA case; expected values written by oracle/ only "
                 "(tests/golden/make_golden.py); the pages print no worked example",
        "sm_scale": scale,
        "inputs": {"q": q.tolist(), "kv": kv.tolist(), "attn_sink": sink.tolist(),
                   "topk_idxs": idx.tolist(), "do": dout.tolist()},
        "expected": {"o": o.reshape(q.shape).tolist(), "lse2": lse2.reshape(1, 3, 2).tolist(),
                     "dq": dq.reshape(q.shape).tolist(), "dkv": dkv.tolist(),
                     "dsink": dsink.tolist(), "delta": delta.reshape(1, 3, 2).tolist()},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
