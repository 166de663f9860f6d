"""Canary guard words: every buffer a kernel writes (outputs, workspaces,
the exchange pools, the dKV accumulator) is placed between two guard zones
filled with a known byte pattern, and after the calls every guard byte must
be unchanged.  A write past either end of a buffer -- an indexing slip the
sanitizer would report, which this GPU pool does not run -- shows up here
as a changed guard, on the host, without faulting anything.  The cases run
ragged shapes (a partial last slot block, H off the 16-row grid, masked and
out-of-range indices) on both the CTA-pair (D = 512) and the single-CTA
(D = 64) paths, the deterministic backward and the indexer backward."""
import pytest
import torch

from bwd_sparse_mqa_gb300 import _lib, inputs
from bwd_sparse_mqa_gb300.api import device_status

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side
PATTERN = 0xA5


class Guarded:
    """A device byte buffer of `nbytes` between two guard zones; `view`
    returns the interior as a tensor of the given dtype and shape."""

    def __init__(self, nbytes: int):
        self.n = (nbytes + 255) // 256 * 256
        self.raw = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")

    def ptr(self):
        return self.raw.data_ptr() + GUARD

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype)[:_numel(shape)].view(shape)

    def intact(self) -> bool:
        return bool(torch.all(self.raw[:GUARD] == PATTERN)) and \
            bool(torch.all(self.raw[GUARD + self.n:] == PATTERN))


def _numel(shape):
    n = 1
    for s in shape:
        n *= s
    return n


def _p(x):
    import ctypes
    return ctypes.c_void_p(x if isinstance(x, int) else x.data_ptr())


@pytest.mark.parametrize("D,H,deterministic", [(512, 48, False), (512, 128, True),
                                               (64, 100, False), (64, 16, True)])
def test_attention_writes_stay_in_bounds(D, H, deterministic):
    import ctypes
    x = inputs.custom(2, 37, 150, H, D, 133, recipe="causal_masked10", seed=80 + H)
    g = {k: v.cuda() for k, v in x.items()}
    B, S, _, _ = g["q"].shape
    S_kv = g["kv"].shape[1]
    shp = _lib.Shape(B, S, S_kv, H, D, 133)
    lib = _lib.load()
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    o = Guarded(B * S * H * D * 2)
    lse = Guarded(B * S * H * 4)
    fws = Guarded(max(int(lib.smqa_fwd_workspace_bytes(shp)), 256))
    assert lib.smqa_fwd(_p(g["q"]), _p(g["kv"]), _p(g["attn_sink"]), _p(g["topk_idxs"]), shp,
                        0.0, _p(o.ptr()), _p(lse.ptr()), _p(fws.ptr()), fws.n, 0, sp) == 0
    flags = _lib.FLAG_DETERMINISTIC_DKV if deterministic else 0
    dq = Guarded(B * S * H * D * 2)
    dkv = Guarded(B * S_kv * D * 2)
    dsink = Guarded(H * 4)
    bws = Guarded(int(lib.smqa_bwd_workspace_bytes(shp, flags)))
    assert lib.smqa_bwd(_p(g["q"]), _p(g["kv"]), _p(g["attn_sink"]), _p(o.ptr()), _p(g["do"]),
                        _p(g["topk_idxs"]), _p(lse.ptr()), shp, 0.0, _p(dq.ptr()),
                        _p(dkv.ptr()), _p(dsink.ptr()), _p(bws.ptr()), bws.n, flags, sp) == 0
    torch.cuda.synchronize()
    assert device_status() == 0
    for name, buf in (("o", o), ("lse", lse), ("fwd workspace", fws), ("dq", dq), ("dkv", dkv),
                      ("dsink", dsink), ("bwd workspace", bws)):
        assert buf.intact(), f"{name}: a guard byte changed (out-of-bounds write)"
    # The interiors were written (the guard check is not vacuous).
    assert not torch.all(o.view(torch.uint8, (B * S * H * D * 2,)) == PATTERN)
    assert not torch.all(dq.view(torch.uint8, (B * S * H * D * 2,)) == PATTERN)


@pytest.mark.parametrize("D,H", [(128, 64), (64, 37)])
def test_indexer_writes_stay_in_bounds(D, H):
    import ctypes
    x = inputs.indexer_custom(1, 29, 170, H, D, 117, recipe="causal_masked10", seed=90 + H)
    g = {k: v[0].contiguous().cuda() for k, v in x.items()}
    S = g["index_q"].shape[0]
    shp = _lib.Shape(1, S, g["index_k"].shape[0], H, D, 117)
    lib = _lib.load()
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dq = Guarded(S * H * D * 2)
    assert lib.smqa_indexer_bwd(_p(g["index_q"]), _p(g["weights"]), _p(g["index_k"]),
                                _p(g["topk_indices"]), _p(g["grad_scores"]), shp,
                                _p(dq.ptr()), sp) == 0
    torch.cuda.synchronize()
    assert device_status() == 0
    assert dq.intact(), "indexer dq: a guard byte changed (out-of-bounds write)"
    assert not torch.all(dq.view(torch.uint8, (S * H * D * 2,)) == PATTERN)
