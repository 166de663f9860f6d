"""The C-ABI library: it loads, exports every symbol include/sparse_mqa.h
declares, and rejects bad arguments on the host before touching a GPU
(these calls return before any CUDA call, so they run without a device)."""
import ctypes
import os
import re

import pytest

from bwd_sparse_mqa_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "sparse_mqa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smqa_\w+)\s*\(", text)))


def test_exports_match_header(lib):
    declared = _header_functions()
    assert declared, "no declarations parsed"
    assert sorted(_lib.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), f"{name} not exported"


def test_version_and_strings(lib):
    assert lib.smqa_abi_version() == 6
    assert lib.smqa_status_string(0) == b"SMQA_OK"
    assert lib.smqa_status_string(4) == b"SMQA_ERR_DEVICE_TIMEOUT"
    assert lib.smqa_status_string(99) == b"SMQA_ERR_UNKNOWN"


def test_wait_limit_setter(lib):
    """smqa_set_wait_limit_ns returns the limit in force before the call and
    0 restores the default (4 s unless SMQA_WAIT_LIMIT_NS is set).  Host
    state only: nothing is launched."""
    default = lib.smqa_set_wait_limit_ns(0)
    assert default > 0
    assert lib.smqa_set_wait_limit_ns(12345) == default
    assert lib.smqa_set_wait_limit_ns(0) == 12345
    assert lib.smqa_set_wait_limit_ns(0) == default


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_fwd_rejects_bad_shapes(lib):
    p = _fake()
    bad = [(_lib.Shape(0, 1, 1, 1, 64, 1), _lib.SMQA_ERR_INVALID_ARG),
           (_lib.Shape(1, 1, 1, 1, 64, 0), _lib.SMQA_ERR_INVALID_ARG),
           (_lib.Shape(1, 1, 1, 129, 64, 1), _lib.SMQA_ERR_UNSUPPORTED),
           (_lib.Shape(1, 1, 1, 16, 128, 1), _lib.SMQA_ERR_UNSUPPORTED),
           (_lib.Shape(1, 1, 1 << 23, 16, 512, 1), _lib.SMQA_ERR_UNSUPPORTED)]
    for shp, want in bad:
        assert lib.smqa_fwd(p, p, p, p, shp, 0.0, p, p, None, 0, 0, None) == want


def test_fwd_rejects_null_misaligned_and_flags(lib):
    shp = _lib.Shape(1, 4, 4, 16, 64, 4)
    p = _fake()
    assert lib.smqa_fwd(None, p, p, p, shp, 0.0, p, p, None, 0, 0, None) == \
        _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_fwd(_fake(0x10008), p, p, p, shp, 0.0, p, p, None, 0, 0, None) == \
        _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_fwd(p, p, p, p, shp, 0.0, p, p, None, 0, 8, None) == _lib.SMQA_ERR_INVALID_ARG
    assert b"misaligned" in lib.smqa_last_error()


def test_bwd_workspace_and_checks(lib):
    shp = _lib.Shape(2, 8, 16, 16, 64, 4)
    ws = lib.smqa_bwd_workspace_bytes(shp, 0)
    ws32 = lib.smqa_bwd_workspace_bytes(shp, _lib.FLAG_RETURN_DKV_FP32)
    acc = 2 * 16 * 64 * 4
    delta = 2 * 8 * 16 * 4
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert ws == r(acc) + r(delta)
    assert ws32 == r(delta)
    assert lib.smqa_bwd_workspace_bytes(_lib.Shape(1, 1, 1, 1, 100, 1), 0) == 0
    p = _fake()
    args = [p] * 7 + [shp, 0.0, p, p, None, p]
    assert lib.smqa_bwd(*args, ws - 1, 0, None) == _lib.SMQA_ERR_UNSUPPORTED
    assert lib.smqa_bwd(*args, ws, 8, None) == _lib.SMQA_ERR_INVALID_ARG
    args_null = [p] * 6 + [None, shp, 0.0, p, p, None, p]
    assert lib.smqa_bwd(*args_null, ws, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    # dsink is optional but, when given, must be 4-byte aligned.
    args_bad_dsink = [p] * 7 + [shp, 0.0, p, p, _fake(0x10002), p]
    assert lib.smqa_bwd(*args_bad_dsink, ws, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_bwd_sink_grad(p, p, None, shp, p, None) == _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_bwd_sink_grad(p, p, p, _lib.Shape(1, 1, 1, 129, 64, 1), p, None) == \
        _lib.SMQA_ERR_UNSUPPORTED


def test_bwd_deterministic_flag_workspace_and_checks(lib):
    """SMQA_FLAG_DETERMINISTIC_DKV: the fixed-point accumulator (8 bytes per
    dkv element), a 256-byte block of per-call statistics and a 4-byte
    reference count per kv row, always in the workspace (also with the fp32
    output); unknown flags are rejected."""
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    shp = _lib.Shape(2, 8, 16, 16, 64, 4)
    acc8, stats, counts, delta = 2 * 16 * 64 * 8, 256, 2 * 16 * 4, 2 * 8 * 16 * 4
    det = _lib.FLAG_DETERMINISTIC_DKV
    want = r(acc8) + stats + r(counts) + r(delta)
    assert lib.smqa_bwd_workspace_bytes(shp, det) == want
    assert lib.smqa_bwd_workspace_bytes(shp, det | _lib.FLAG_RETURN_DKV_FP32) == want
    p = _fake()
    args = [p] * 7 + [shp, 0.0, p, p, None, p]
    need = lib.smqa_bwd_workspace_bytes(shp, det)
    assert lib.smqa_bwd(*args, need - 1, det, None) == _lib.SMQA_ERR_UNSUPPORTED
    assert lib.smqa_bwd(*args, need, 8, None) == _lib.SMQA_ERR_INVALID_ARG


def test_bwd_exchange_pool_size_and_checks(lib):
    """D = 512: the workspace carries the CTA-pair exchange pool (4 KB of slot
    flags + 96 slots of two receivers x two block parities x 33 KB of
    block-floating-point partial S and dP); D = 64 needs none.  smqa_bwd_main rejects a
    pool that is too small, or missing, before any GPU work."""
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    s512 = _lib.Shape(1, 8, 16, 16, 512, 4)
    ex = lib.smqa_bwd_exchange_bytes(s512)
    assert ex == 4096 + 96 * 2 * 2 * (32768 + 1024)
    acc, delta = 16 * 512 * 4, 8 * 16 * 4
    assert lib.smqa_bwd_workspace_bytes(s512, 0) == r(acc) + r(delta) + r(ex)
    assert lib.smqa_bwd_exchange_bytes(_lib.Shape(1, 8, 16, 16, 64, 4)) == 0
    assert lib.smqa_bwd_exchange_bytes(_lib.Shape(1, 8, 16, 16, 100, 4)) == 0
    p = _fake()
    args = [p] * 7 + [s512, 0.0, p, p]
    assert lib.smqa_bwd_main(*args, p, ex - 1, None) == _lib.SMQA_ERR_UNSUPPORTED
    assert b"exchange pool too small" in lib.smqa_last_error()
    assert lib.smqa_bwd_main(*args, None, ex, None) == _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_bwd_main(*args, _fake(0x10010), ex, None) == _lib.SMQA_ERR_INVALID_ARG


def test_fwd_exchange_pool_size_and_checks(lib):
    """D = 512: the forward's CTA pairs trade block-floating-point partial
    scores through an exchange pool (4 KB of slot flags + 96 slots of two
    receivers x six buffers x 16.5 KB); D = 64 needs none.  smqa_fwd
    rejects a pool that is too small, missing or misaligned before any GPU
    work, and the static-scratch entry rejects bad shapes the same way."""
    s512 = _lib.Shape(1, 8, 16, 16, 512, 4)
    ex = lib.smqa_fwd_workspace_bytes(s512)
    assert ex == 4096 + 96 * 2 * 6 * (16384 + 512)
    assert ex <= _lib.STATIC_SCRATCH_BYTES
    assert lib.smqa_fwd_workspace_bytes(_lib.Shape(1, 8, 16, 16, 64, 4)) == 0
    assert lib.smqa_fwd_workspace_bytes(_lib.Shape(1, 8, 16, 16, 100, 4)) == 0
    p = _fake()
    args = [p] * 4 + [s512, 0.0, p, p]
    assert lib.smqa_fwd(*args, p, ex - 1, 0, None) == _lib.SMQA_ERR_UNSUPPORTED
    assert b"workspace too small" in lib.smqa_last_error()
    assert lib.smqa_fwd(*args, None, ex, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_fwd(*args, _fake(0x10010), ex, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    bad = _lib.Shape(1, 8, 16, 129, 512, 4)
    assert lib.smqa_fwd_static_scratch(p, p, p, p, bad, 0.0, p, p, 0, None) == \
        _lib.SMQA_ERR_UNSUPPORTED


def _r256(x):
    return (x + 255) // 256 * 256


def test_host_entry_workspace_sizes_and_checks(lib):
    """smqa_fwd_host / smqa_fwd_bwd_host: the workspace holds a device copy of
    every input and output (each region 256-byte aligned) plus the exchange
    pools; bad arguments are rejected before any CUDA call."""
    B, S, S_kv, H, D, K = 2, 300, 200, 16, 512, 64
    shp = _lib.Shape(B, S, S_kv, H, D, K)
    rows, kvel = B * S * H, B * S_kv * D
    fwd = (_r256(kvel * 2) + _r256(H * 4) + 2 * _r256(rows * D * 2) + _r256(B * S * K * 4) +
           _r256(rows * 4) + _r256(lib.smqa_fwd_workspace_bytes(shp)))
    assert lib.smqa_fwd_host_workspace_bytes(shp) == fwd
    bwd_tail = (2 * _r256(rows * D * 2) + _r256(rows * 4) + _r256(H * 4) +
                _r256(lib.smqa_bwd_exchange_bytes(shp)))
    assert lib.smqa_fwd_bwd_host_workspace_bytes(shp, 0) == \
        fwd + bwd_tail + _r256(kvel * 4) + _r256(kvel * 2)
    # fp32 dkv: the accumulator is the result; deterministic: 8-byte
    # accumulator, 256 bytes of statistics and a count per kv row
    assert lib.smqa_fwd_bwd_host_workspace_bytes(shp, _lib.FLAG_RETURN_DKV_FP32) == \
        fwd + bwd_tail + _r256(kvel * 4)
    assert lib.smqa_fwd_bwd_host_workspace_bytes(shp, _lib.FLAG_DETERMINISTIC_DKV) == \
        fwd + bwd_tail + _r256(kvel * 8) + 256 + _r256(B * S_kv * 4) + _r256(kvel * 2)
    assert lib.smqa_fwd_host_workspace_bytes(_lib.Shape(1, 8, 16, 129, 512, 4)) == 0
    assert lib.smqa_fwd_bwd_host_workspace_bytes(_lib.Shape(1, 8, 16, 16, 100, 4), 0) == 0

    p = _fake()
    need = lib.smqa_fwd_bwd_host_workspace_bytes(shp, 0)
    args = [p] * 5 + [shp, 0.0] + [p] * 5
    assert lib.smqa_fwd_bwd_host(*args, p, need - 1, 0, None) == _lib.SMQA_ERR_UNSUPPORTED
    assert b"workspace too small" in lib.smqa_last_error()
    assert lib.smqa_fwd_bwd_host(*args, _fake(0x10010), need, 0, None) == \
        _lib.SMQA_ERR_INVALID_ARG
    assert lib.smqa_fwd_bwd_host(*args, p, need, 8, None) == _lib.SMQA_ERR_INVALID_ARG
    no_dout = [p] * 4 + [None, shp, 0.0] + [p] * 5
    assert lib.smqa_fwd_bwd_host(*no_dout, p, need, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    no_dkv = [p] * 5 + [shp, 0.0] + [p] * 3 + [None, p]
    assert lib.smqa_fwd_bwd_host(*no_dkv, p, need, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    fneed = lib.smqa_fwd_host_workspace_bytes(shp)
    fargs = [p] * 4 + [shp, 0.0, p, p]
    assert lib.smqa_fwd_host(*fargs, p, fneed - 1, 0, None) == _lib.SMQA_ERR_UNSUPPORTED
    assert lib.smqa_fwd_host(*fargs, None, fneed, 0, None) == _lib.SMQA_ERR_INVALID_ARG
    # the backward's flags are not forward flags
    assert lib.smqa_fwd_host(*fargs, p, fneed, _lib.FLAG_RETURN_DKV_FP32, None) == \
        _lib.SMQA_ERR_INVALID_ARG
    bad = _lib.Shape(1, 8, 16, 16, 100, 4)
    assert lib.smqa_fwd_host(p, p, p, p, bad, 0.0, p, p, p, fneed, 0, None) == \
        _lib.SMQA_ERR_UNSUPPORTED


def test_host_interface_rejects_device_tensors():
    import torch
    from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_bwd_host, sparse_mqa_fwd_host
    q = torch.zeros(1, 4, 16, 64, dtype=torch.bfloat16)
    kv = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    sink = torch.zeros(16)
    idx = torch.zeros(1, 4, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CPU tensor"):
        sparse_mqa_fwd_host(q.to("meta"), kv, sink, idx)
    with pytest.raises(TypeError, match="int32"):
        sparse_mqa_fwd_host(q, kv, sink, idx.long())
    with pytest.raises(ValueError, match="shape"):
        sparse_mqa_fwd_bwd_host(q, kv, sink, idx, q[:, :2].contiguous())


def test_python_interface_rejects_cpu_tensors():
    import torch
    from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_interface
    q = torch.zeros(1, 4, 16, 64, dtype=torch.bfloat16)
    kv = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    sink = torch.zeros(16)
    idx = torch.zeros(1, 4, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        sparse_mqa_fwd_interface(q, kv, sink, idx)


def test_autograd_wrapper_rejects_cpu_tensors():
    import torch
    from bwd_sparse_mqa_gb300 import sparse_mqa
    q = torch.zeros(1, 4, 16, 64, dtype=torch.bfloat16, requires_grad=True)
    kv = torch.zeros(1, 4, 64, dtype=torch.bfloat16, requires_grad=True)
    sink = torch.zeros(16, requires_grad=True)
    idx = torch.zeros(1, 4, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        sparse_mqa(q, kv, sink, idx)


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "bwd_sparse_mqa_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "smqa_oracle" not in text, f


@pytest.mark.parametrize("B,S", [(1, 1), (1, 255), (1, 256), (1, 1100), (1, 8192), (2, 600),
                                 (3, 100), (7, 300), (64, 128), (1000, 3), (4, 32768),
                                 (5, 257)])
def test_host_chunk_plan_partitions_the_tokens(lib, B, S):
    """The host entry's chunk plan covers every (b, s) exactly once, in
    order, with contiguous tokens per chunk, at least 256 tokens per chunk
    (except the last piece of a batch element's positions, a last group of
    whole batch elements, or a smaller problem), pieces of S in whole waves
    of 76 tokens (D = 512 on 152 SMs, no device here) but the last one, and
    at most about 24 chunks."""
    shp = _lib.Shape(B, S, 64, 16, 512, 8)
    n = lib.smqa_host_chunk_plan(shp, None, 0)
    assert n >= 1
    buf = (ctypes.c_int32 * (4 * n))()
    assert lib.smqa_host_chunk_plan(shp, buf, n) == n
    plan = [tuple(buf[4 * c:4 * c + 4]) for c in range(n)]
    flat = []
    for b0, nb, s0, ns in plan:
        assert nb >= 1 and ns >= 1 and b0 + nb <= B and s0 + ns <= S
        if nb > 1:
            assert s0 == 0 and ns == S
        flat.extend(range(b0 * S + s0, b0 * S + s0 + nb * ns))
        last_piece = nb == 1 and s0 + ns == S
        assert nb * ns >= min(256, B * S) or last_piece or (b0 + nb == B and s0 == 0 and ns == S)
        if nb == 1 and not last_piece:
            assert ns % 76 == 0
    assert flat == list(range(B * S))
    assert n <= 25
    assert lib.smqa_host_chunk_plan(_lib.Shape(B, S, 64, 16, 100, 8), None, 0) == 0
