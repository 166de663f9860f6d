"""GPU (CUDA path through the C ABI) against the fp64 oracle, element by
element, on seeded inputs: small shapes on every token, the full-size
workloads on a token sample (see tests/_parity.py for the tolerances)."""
import numpy as np
import pytest
import torch

from bwd_sparse_mqa_gb300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu


def test_small_config_all_tokens():
    """B=1 S=128 H=16 D=64 topk=32, causal, short rows padded with -1."""
    errs = P.check_full(inputs.make_inputs(inputs.CONFIGS[0]))
    print(errs)


@pytest.mark.parametrize("H", [128, 64, 16])
def test_d512_several_blocks_ragged_tail(H):
    """D=512 (CTA-pair path); topk=200 = 3 full 64-slot blocks + a tail of 8
    (6 full 32-slot backward blocks + 8); 10% masked slots; B=2."""
    x = inputs.custom(2, 48, 300, H, 512, 200, recipe="causal_masked10", seed=7)
    print(P.check_full(x))


def test_d64_h128_masked():
    x = inputs.custom(2, 40, 90, 128, 64, 70, recipe="causal_masked10", seed=8)
    print(P.check_full(x))


def test_explicit_sm_scale_and_topk_one():
    x = inputs.custom(1, 20, 20, 32, 512, 1, seed=9)
    print(P.check_full(x, sm_scale=0.11))


def test_all_masked_rows_and_duplicates():
    x = inputs.custom(1, 16, 64, 64, 512, 96, seed=10)
    idx = x["topk_idxs"]
    idx[0, 3] = -1                      # a row with every slot masked
    idx[0, 5, :] = 64                   # masked by S_kv
    idx[0, 9, :10] = 7                  # one row listed ten times
    errs = P.check_full(x)
    print(errs)
    g = P.to_dev(x)
    o, lse = P.run_fwd(g)
    assert torch.all(o[0, 3] == 0) and torch.all(o[0, 5] == 0)
    sink2 = g["attn_sink"] / np.log(2.0)
    assert torch.allclose(lse[0, 3], sink2, rtol=1e-5, atol=1e-6)


def test_masked_tails_and_gaps():
    """Both kernels stop after the last slot block holding a valid slot;
    rows whose valid slots end early, sit only at the end, or straddle a
    fully masked block must still match the oracle."""
    x = inputs.custom(1, 24, 300, 128, 512, 256, seed=12)
    idx = x["topk_idxs"]
    idx[0, 0, 1:] = -1                  # only slot 0 valid: one block
    idx[0, 1, 64:128] = -1              # a fully masked 64-slot block, valid slots after it
    idx[0, 2, :255] = 300               # only the last slot valid
    idx[0, 3, 130:] = -1                # tail ends inside a block
    idx[0, 4, 64:] = -1                 # exactly one full 64-slot block
    idx[0, 5, 32:] = -1                 # exactly one full 32-slot block
    print(P.check_full(x))


def test_return_dkv_fp32_and_reference_rounding():
    # D = 64 (no exchange): the two exp2-argument orders agree to about one
    # fp32 rounding of the logit.
    x64 = inputs.custom(1, 24, 100, 64, 64, 80, recipe="causal_masked10", seed=12)
    g64 = P.to_dev(x64)
    o, lse = P.run_fwd(g64)
    o2, lse2 = P.run_fwd(g64, reference_rounding=True)
    assert P.rel_err(o2, o.double().cpu().numpy()) < 1e-2
    assert P.rel_err(lse2, lse.double().cpu().numpy()) < 1e-5
    # D = 512: each order goes through the pair's block-floating-point
    # exchange in its own scaling, so they agree to the LSE tolerance; each
    # is checked against the oracle.
    x = inputs.custom(1, 24, 100, 128, 512, 80, recipe="causal_masked10", seed=11)
    g = P.to_dev(x)
    o, lse = P.run_fwd(g)
    o2, lse2 = P.run_fwd(g, reference_rounding=True)
    assert P.rel_err(o2, o.double().cpu().numpy()) < 1e-2
    assert P.rel_err(lse2, lse.double().cpu().numpy()) < P.TOL["lse"]
    o_ref, lse_ref = P.oracle.fwd(x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], None)
    P.assert_close("o", o2, o_ref)
    P.assert_close("lse", lse2, lse_ref)
    dq, dkv = P.run_bwd(g, o, lse, g["do"])
    dq32, dkv32 = P.run_bwd(g, o, lse, g["do"], return_dkv_accum_dtype=True)
    assert dkv32.dtype == torch.float32 and dkv.dtype == torch.bfloat16
    assert torch.equal(dq32, dq)
    assert P.rel_err(dkv, dkv32.double().cpu().numpy()) < 8e-3


@pytest.mark.parametrize("D", [64, 512])
@pytest.mark.parametrize("H", [1, 48, 100])
def test_head_counts_off_the_tile(H, D):
    """Head counts that are not a multiple of 16 (the MMA tile is 128 head
    rows; rows H..127 are zero-filled and never stored), every token."""
    x = inputs.custom(2, 40, 200, H, D, 150, recipe="causal_masked10", seed=40 + H)
    print(P.check_full(x))


@pytest.mark.parametrize("D", [64, 512])
def test_topk_4096(D):
    """topk = 4096 (64 slot blocks per token, twice the largest workload's),
    each row a permutation of the same 4096 rows of S_kv = 5000 with 10% of
    the slots masked, every token."""
    x = inputs.custom(1, 12, 5000, 64, D, 4096, recipe="hot4096_masked10", seed=50)
    print(P.check_full(x))


@pytest.mark.parametrize("ci", [1, 2, 3, 4])
def test_full_size_workloads_sampled(ci):
    """The full-size workloads (fwd h64/d512/k512; h128/d512/k2048 recent;
    hot-4096 scatter stress; 32k long context), run whole on the GPU in the
    benchmark's launch configuration and checked on a seeded sample of 256
    tokens (plus s = 0, topk-1, topk and S-1 of every batch element)."""
    cfg = inputs.CONFIGS[ci]
    x = inputs.make_inputs(cfg, device="cuda")
    tokens = P.sample_tokens(cfg.B, cfg.S, cfg.topk, 256, seed=100 + ci)
    errs = P.check_sampled(x, tokens, do_fwd=cfg.passes != "bwd",
                           do_bwd=cfg.passes != "fwd")
    print(cfg.name, errs)
