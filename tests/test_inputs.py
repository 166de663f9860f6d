"""The seeded input recipes have the structure they claim (CPU, small sizes)."""
import torch

from bwd_sparse_mqa_gb300 import inputs


def _rows_ok(idx, S_kv, causal=True):
    for s in range(idx.shape[0]):
        row = idx[s].tolist()
        valid = [r for r in row if 0 <= r < S_kv]
        assert len(valid) == len(set(valid)), "duplicate index in a row"
        if causal:
            assert all(r <= s for r in valid), "non-causal index"


def test_determinism():
    a = inputs.custom(1, 32, 32, 4, 16, 8, seed=5)
    b = inputs.custom(1, 32, 32, 4, 16, 8, seed=5)
    for k in a:
        assert torch.equal(a[k], b[k])


def test_small_config_shapes_and_causality():
    cfg = inputs.CONFIGS[0]
    x = inputs.make_inputs(cfg)
    assert x["q"].shape == (1, 128, 16, 64) and x["q"].dtype == torch.bfloat16
    assert x["kv"].shape == (1, 128, 64) and x["kv"].dtype == torch.bfloat16
    assert x["attn_sink"].dtype == torch.float32 and x["attn_sink"].shape == (16,)
    idx = x["topk_idxs"]
    assert idx.dtype == torch.int32 and idx.shape == (1, 128, 32)
    _rows_ok(idx[0], 128)
    # rows with fewer than topk candidates take all of them and pad at the end
    for s in range(31):
        row = idx[0, s].tolist()
        assert sorted(row[: s + 1]) == list(range(s + 1))
        assert all(r == -1 for r in row[s + 1:])
    assert (idx[0, 40:] >= 0).all()


def test_recent_window_recipe():
    g = torch.Generator().manual_seed(0)
    idx = inputs.make_indices("causal_recent512", 1, 1200, 1200, 600, g, "cpu")[0]
    _rows_ok(idx, 1200)
    i = 1100
    row = set(idx[i].tolist())
    assert set(range(i - 511, i + 1)) <= row


def test_window64_recipe():
    g = torch.Generator().manual_seed(0)
    idx = inputs.make_indices("causal_window64", 1, 300, 300, 100, g, "cpu")[0]
    _rows_ok(idx, 300)
    for i in (64, 150, 299):
        assert set(range(i - 63, i + 1)) <= set(idx[i].tolist())


def test_masked10_recipe():
    g = torch.Generator().manual_seed(1)
    idx = inputs.make_indices("causal_masked10", 1, 400, 400, 64, g, "cpu")[0]
    tail = idx[100:]
    frac = ((tail < 0) | (tail >= 400)).float().mean().item()
    assert 0.07 < frac < 0.13
    assert (tail == 400).any() and (tail == -1).any()
    _rows_ok(idx, 400)


def test_hot_rows_recipe():
    g = torch.Generator().manual_seed(2)
    idx = inputs.make_indices("hot4096_masked10", 1, 64, 8192, 256, g, "cpu")[0]
    valid = idx[(idx >= 0)]
    assert len(set(valid.tolist())) <= 4096
    frac = (idx < 0).float().mean().item()
    assert 0.06 < frac < 0.14
    _rows_ok(idx, 8192, causal=False)
