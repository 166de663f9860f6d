"""The failure path of the kernels' bounded waits, in the form this pool
allows: no fault, trap or endless loop.  The library's test hook
(smqa_debug_stall) makes one CTA stop after its first tensor-core
instruction and wait for a condition that never comes true; with a 50 ms
wait limit that wait runs out, the CTA records SMQA_ERR_DEVICE_TIMEOUT in the
device status word, drains its copies and MMAs, frees TMEM and exits, and its
peer CTA (D = 512) gives up waiting for the exchange.  The lightning-indexer
backward's kernel is driven through the same path.  The test checks that the call returns, that the
status is reported (also as an exception with check_status=True, and through
the autograd wrapper), that later launches skip their work while the word is
set, that clearing it works, and that afterwards, in the same process and
context, a normal call matches the fp64 oracle.  It runs in a child process
so that the wait limit and the status word never leak into other tests."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys
import torch
sys.path.insert(0, ROOT)
import oracle
from bwd_sparse_mqa_gb300 import (inputs, sparse_mqa, sparse_mqa_bwd_interface,
                                  sparse_mqa_fwd_interface, set_wait_limit_ns, device_status)
from bwd_sparse_mqa_gb300 import _lib
from tests import _parity as P

TIMEOUT = _lib.SMQA_ERR_DEVICE_TIMEOUT
lib = _lib.load()
for D in (512, 64):
    x = inputs.custom(1, 32, 300, 128, D, 256, recipe="causal_masked10", seed=60 + D)
    g = P.to_dev(x)
    assert device_status(clear=True) == 0
    default = set_wait_limit_ns(50_000_000)
    lib.smqa_debug_stall(0)
    try:
        # The call returns; the status word reports the timeout and stays set.
        o, lse = sparse_mqa_fwd_interface(g["q"], g["kv"], g["attn_sink"], g["topk_idxs"])
        assert device_status(clear=False) == TIMEOUT, "forward did not time out"
        assert device_status(clear=False) == TIMEOUT, "status word is not sticky"
        # While it is set, every call skips its work and check_status raises.
        try:
            sparse_mqa_fwd_interface(g["q"], g["kv"], g["attn_sink"], g["topk_idxs"],
                                     check_status=True)
            raise AssertionError("check_status did not raise")
        except _lib.SMQAError as e:
            assert e.status == TIMEOUT
        assert device_status(clear=True) == TIMEOUT
        assert device_status(clear=False) == 0
        # The backward's waits run out the same way.
        o2 = torch.zeros_like(g["q"])
        lse2 = torch.zeros(g["q"].shape[:3], dtype=torch.float32, device="cuda")
        try:
            sparse_mqa_bwd_interface(g["q"], g["kv"], g["attn_sink"], o2, g["do"],
                                     g["topk_idxs"], lse2, check_status=True)
            raise AssertionError("backward check_status did not raise")
        except _lib.SMQAError as e:
            assert e.status == TIMEOUT
        assert device_status(clear=True) == TIMEOUT
        # The autograd wrapper raises from its forward.
        q = g["q"].clone().requires_grad_(True)
        try:
            sparse_mqa(q, g["kv"], g["attn_sink"], g["topk_idxs"], check_status=True)
            raise AssertionError("autograd check_status did not raise")
        except _lib.SMQAError as e:
            assert e.status == TIMEOUT
        assert device_status(clear=True) == TIMEOUT
    finally:
        lib.smqa_debug_stall(-1)
        set_wait_limit_ns(0)
    assert set_wait_limit_ns(0) == default
    # Same process, same context: a normal call works and matches the oracle.
    errs = P.check_full(x)
    o, lse = sparse_mqa_fwd_interface(g["q"], g["kv"], g["attn_sink"], g["topk_idxs"],
                                      check_status=True)
    sparse_mqa_bwd_interface(g["q"], g["kv"], g["attn_sink"], o, g["do"], g["topk_idxs"], lse,
                             check_status=True)
    print("D", D, "after the timeout:", errs)

# The indexer backward's kernel takes the same path.
from bwd_sparse_mqa_gb300 import indexer_bwd_interface
import numpy as np
xi = inputs.indexer_custom(1, 24, 150, 64, 128, 100, recipe="causal_masked10", seed=61)
gi = {k: v[0].contiguous().cuda() for k, v in xi.items()}
set_wait_limit_ns(50_000_000)
lib.smqa_debug_stall(3)
try:
    indexer_bwd_interface(gi["index_q"], gi["weights"], gi["index_k"], gi["topk_indices"],
                          gi["grad_scores"])
    assert device_status(clear=False) == TIMEOUT, "indexer backward did not time out"
    assert device_status(clear=True) == TIMEOUT
finally:
    lib.smqa_debug_stall(-1)
    set_wait_limit_ns(0)
dq = indexer_bwd_interface(gi["index_q"], gi["weights"], gi["index_k"], gi["topk_indices"],
                           gi["grad_scores"])
assert device_status(clear=False) == 0
ref, slack = oracle.indexer_bwd(xi["index_q"][0], xi["weights"][0], xi["index_k"][0],
                                xi["topk_indices"][0], xi["grad_scores"][0], amb=2.0 ** -12)
got = dq.float().cpu().numpy().astype(np.float64)
e = float(np.max(np.maximum(np.abs(got - ref) - slack, 0.0)) / np.max(np.abs(ref)))
assert e <= 2e-2, e
print("indexer after the timeout:", e)
print("OK")
'''


@pytest.mark.gpu
def test_bounded_wait_timeout_is_reported_and_recovered():
    code = "ROOT = %r\n" % ROOT + SCRIPT
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    print(r.stdout[-3000:])
    print(r.stderr[-3000:])
    assert r.returncode == 0 and r.stdout.strip().endswith("OK")
