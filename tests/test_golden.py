"""The oracle against its stored regression fixture (tests/golden)."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_oracle_fixture():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        g = json.load(f)
    inp, exp = g["inputs"], g["expected"]
    q = np.array(inp["q"])
    kv = np.array(inp["kv"])
    sink = np.array(inp["attn_sink"])
    idx = np.array(inp["topk_idxs"], dtype=np.int32)
    dout = np.array(inp["do"])
    o, lse2 = oracle.fwd_f64(q, kv, sink, idx, sm_scale=g["sm_scale"])
    dq, dkv, dsink, delta = oracle.bwd_f64(q, kv, sink, idx, dout, sm_scale=g["sm_scale"])
    np.testing.assert_allclose(o.reshape(q.shape), exp["o"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2.reshape(1, 3, 2), exp["lse2"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dq.reshape(q.shape), exp["dq"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dkv, exp["dkv"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dsink, exp["dsink"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(delta.reshape(1, 3, 2), exp["delta"], rtol=1e-12, atol=1e-14)
    # The masked slots (-1 and S_kv=4) really are in the fixture.
    assert (idx < 0).any() and (idx >= kv.shape[1]).any()
