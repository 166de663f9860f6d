#!/usr/bin/env python
"""Benchmark: top-k sparse MQA forward + backward on GB300.

One step = the whole hot path over one batch of a workload: forward (O,
log2 LSE), then the backward's preprocess (Delta and zeroing of the fp32 dKV
accumulator), main kernel (dQ, dKV scatter) and postprocess (dKV to bf16);
forward-only workloads stop after the forward, and the dKV-scatter stress
workload times the backward alone (its O and LSE come from one forward run
before the timed region).  The default workload is B=1, S=S_kv=8192, H=128,
D=512, topk=2048 with causal indices biased to the newest 512 keys; every
workload is synthetic and seeded (bwd_sparse_mqa_gb300/inputs.py).

Metric: TFLOP/s of the step, FLOPs counted on valid slots only
(4*H*D per valid slot forward, 10*H*D backward).  `value` times the kernels
on device-resident inputs; `e2e` times the host-buffer entry points
(smqa_fwd_host / smqa_fwd_bwd_host: page-locked inputs in, results out,
copies overlapped with the kernels in token chunks).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all]
                    [--impl reference]

Prints one JSON line per workload (rank 0).  Under torchrun every rank runs
its own replica (the op shards by tokens with no data-path collective) and
the timed region is bracketed by barriers; value = all ranks' FLOPs / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bwd_sparse_mqa_gb300 import _lib, inputs  # noqa: E402
from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_bwd_host, sparse_mqa_fwd_host  # noqa: E402

WORKLOAD = "h128_d512_k2048_s8192"
METRIC = "sparse MQA fwd/bwd TFLOP/s + % BF16 roofline, 1×GB300, H=128 D=512 topk=2048"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, vendor figure (context for the slower-of fraction)
L2_BYTES = 129 * 2 ** 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_bwd_main_h128_d512_k2048.json")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    """Hash of the backward main kernel's source: its layout and body in
    smqa_bwd.cu (from `struct BwdLayout` to its launcher) and the PTX helpers
    it includes.  Other kernels in the file do not change it."""
    csrc = os.path.join(ROOT, "bwd_sparse_mqa_gb300", "csrc")
    with open(os.path.join(csrc, "smqa_bwd.cu")) as fh:
        text = fh.read()
    start = text.index("struct BwdLayout")
    end = text.index("static cudaError_t launch_bwd_impl", start)
    h = hashlib.sha256(text[start:end].encode())
    with open(os.path.join(csrc, "smqa_ptx.cuh"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the backward main kernel from the committed
    ncu summary, or None if the kernel source changed since it was taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}



def flops_of(idx: torch.Tensor, S_kv: int, H: int, D: int):
    nv = int(((idx >= 0) & (idx < S_kv)).sum().item())
    return 4.0 * H * D * nv, 10.0 * H * D * nv, nv


def passes_of(cfg):
    """(forward in the step, backward in the step) for a workload."""
    return cfg.passes in ("fwd", "fwd+bwd"), cfg.passes in ("fwd+bwd", "bwd")


def algorithmic_bytes(cfg, n_valid):
    """Bytes the forward and the backward must move (valid slots): gathered
    kv rows, the dense per-token tensors, and for the backward the fp32 dKV
    reductions and the per-call accumulator zero / read / cast."""
    B, S, S_kv, H, D, K = cfg.B, cfg.S, cfg.S_kv, cfg.H, cfg.D, cfg.topk
    T = B * S
    fwd = 2 * D * n_valid + 4 * H * D * T + 4 * K * T + 4 * H * T
    bwd = 6 * D * n_valid + 8 * H * D * T + 4 * K * T + 8 * H * T + 10 * B * S_kv * D
    return fwd, bwd


def cpu_baseline(x: dict, cfg, workload: str, target_s: float = 15.0, max_tokens: int = 512):
    """The fp64 oracle as it stands, on the host cores, over a seeded token
    sample of the workload (its passes) sized to ~target_s seconds."""
    import numpy as np

    import oracle
    has_fwd, has_bwd = passes_of(cfg)
    q, kv, sink, idx = x["q"].cpu(), x["kv"].cpu(), x["attn_sink"].cpu(), x["topk_idxs"].cpu()
    dout = x["do"].cpu() if has_bwd else None
    rng = np.random.default_rng(1234)
    T = cfg.B * cfg.S

    def run(n):
        toks = np.sort(rng.choice(T, size=min(n, T), replace=False))
        sel = idx.reshape(T, -1)[torch.as_tensor(toks)]
        nv = int(((sel >= 0) & (sel < cfg.S_kv)).sum())
        t0 = time.perf_counter()
        if has_fwd:
            oracle.fwd(q, kv, sink, idx, tokens=toks)
        if has_bwd:
            oracle.bwd(q, kv, sink, idx, dout, tokens=toks)
        return time.perf_counter() - t0, nv, len(toks)

    probe_n = 4
    dt, _, _ = run(probe_n)
    n = int(max(probe_n, min(max_tokens, probe_n * target_s / max(dt, 1e-3))))
    dt, nv, n = run(n)
    fl = ((4.0 if has_fwd else 0.0) + (10.0 if has_bwd else 0.0)) * cfg.H * cfg.D * nv
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} seeded tokens of {workload} ({cfg.passes}, fp64, {nv} valid slots), "
                      f"{dt:.1f} s"}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (x itself without a process group); the
    tensor lives on `device` (the GPU for NCCL, the CPU for gloo)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank_step: float, steps: int, max_ms: float) -> float:
    """Weak scaling: every rank processes the same units each step, so the
    job's rate is all ranks' units over the slowest rank's time (per second)."""
    return world * units_per_rank_step * steps / (max_ms * 1e-3)


def reference_arm(args, rank: int):
    """--impl reference: the fp64 oracle timed on the host cores, each step a
    bounded token sample of the same workload."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    cfg, workload = workload_cfg(args.workload if args.workload != "all" else WORKLOAD, args.seq)
    has_fwd, has_bwd = passes_of(cfg)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = inputs.make_inputs(cfg, device=dev)
    q, kv, sink, idx = x["q"].cpu(), x["kv"].cpu(), x["attn_sink"].cpu(), x["topk_idxs"].cpu()
    dout = x["do"].cpu() if has_bwd else None
    T = cfg.B * cfg.S
    per_step = min(T, int(os.environ.get("SMQA_REF_TOKENS_PER_STEP", "8")))
    rng = np.random.default_rng(99)
    per_slot = ((4.0 if has_fwd else 0.0) + (10.0 if has_bwd else 0.0)) * cfg.H * cfg.D

    def step():
        toks = np.sort(rng.choice(T, size=per_step, replace=False))
        sel = idx.reshape(T, -1)[torch.as_tensor(toks)]
        nv = int(((sel >= 0) & (sel < cfg.S_kv)).sum())
        if has_fwd:
            oracle.fwd(q, kv, sink, idx, tokens=toks)
        if has_bwd:
            oracle.bwd(q, kv, sink, idx, dout, tokens=toks)
        return per_slot * nv

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    total = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    v = total / dt / 1e12
    line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload, "B": cfg.B, "S": cfg.S, "S_kv": cfg.S_kv,
                       "H": cfg.H, "D": cfg.D, "topk": cfg.topk, "passes": cfg.passes,
                       "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{per_step} seeded tokens per step ({cfg.passes}, "
                                       f"fp64)"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_cfg(name: str, seq=None, tokens=None):
    cfg = inputs.by_name(name)
    workload = name
    if seq:
        import dataclasses
        cfg = dataclasses.replace(cfg, S=seq, S_kv=seq)
        workload = f"{name} with S=S_kv={seq} (profiling size)"
    if tokens:
        workload = f"{workload}, query positions {tokens[0]}-{tokens[1] - 1} (profiling slice)"
    return cfg, workload


def parse_tokens(text):
    """'A:B' -> (A, B): the query positions [A, B) of every batch element."""
    if not text:
        return None
    a, b = (int(v) for v in text.split(":"))
    if not 0 <= a < b:
        raise ValueError("--tokens wants A:B with 0 <= A < B")
    return a, b


def run_workload(args, name, dist, world, rank, local, dev):
    """Times one workload and returns its JSON line (rank 0) or None."""
    tok = parse_tokens(args.tokens)
    cfg, workload = workload_cfg(name, args.seq, tok)
    has_fwd, has_bwd = passes_of(cfg)
    x = inputs.make_inputs(cfg, device=str(dev))
    if tok is not None:
        # Profiling: only the query positions [A, B) of the workload (their
        # index rows still name keys anywhere in [0, S_kv)).
        import dataclasses
        a, b = tok[0], min(tok[1], cfg.S)
        for k in ("q", "do", "topk_idxs"):
            x[k] = x[k][:, a:b].contiguous()
        cfg = dataclasses.replace(cfg, S=b - a)
        torch.cuda.empty_cache()
    q, kv, sink, idx, dout = x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], x["do"]
    B, S, S_kv, H, D, K = cfg.B, cfg.S, cfg.S_kv, cfg.H, cfg.D, cfg.topk
    f_fwd, f_bwd, n_valid = flops_of(idx, S_kv, H, D)
    f_step = (f_fwd if has_fwd else 0.0) + (f_bwd if has_bwd else 0.0)
    lib = _lib.load()
    shp = _lib.Shape(B, S, S_kv, H, D, K)
    o = torch.empty_like(q)
    lse = torch.empty((B, S, H), dtype=torch.float32, device=dev)
    # One exchange pool serves the forward and the backward main kernel (they
    # run one after the other on the stream).
    exch_bytes = max(int(lib.smqa_fwd_workspace_bytes(shp)), int(lib.smqa_bwd_exchange_bytes(shp)))
    exch = torch.empty((max(exch_bytes, 256),), dtype=torch.uint8, device=dev)
    if has_bwd:
        dq = torch.empty_like(q)
        dkv = torch.empty((B, S_kv, D), dtype=torch.bfloat16, device=dev)
        acc = torch.empty((B, S_kv, D), dtype=torch.float32, device=dev)
        delta = torch.empty((B, S, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    scale = D ** -0.5

    def fwd():
        _lib.check("smqa_fwd", lib.smqa_fwd(P(q), P(kv), P(sink), P(idx), shp, scale, P(o), P(lse),
                                            P(exch), exch_bytes, 0, sp))

    kernels = []  # (name, launch) in step order
    if has_fwd:
        kernels.append(("fwd", fwd))
    if has_bwd:
        kernels += [
            ("bwd_pre", lambda: _lib.check("pre", lib.smqa_bwd_preprocess(
                P(o), P(dout), shp, P(delta), P(acc), sp))),
            ("bwd_main", lambda: _lib.check("main", lib.smqa_bwd_main(
                P(q), P(kv), P(sink), P(dout), P(idx), P(lse), P(delta), shp, scale, P(dq),
                P(acc), P(exch), exch_bytes, sp))),
            ("bwd_post", lambda: _lib.check("post", lib.smqa_bwd_postprocess(
                P(acc), shp, P(dkv), sp))),
        ]
    if not has_fwd:
        fwd()  # O and LSE for a backward-only step, outside the timed region

    # Inputs smaller than L2 are flushed between timed steps (a 512 MiB
    # write, outside the per-step events); larger ones stream from HBM anyway.
    in_bytes = sum(t.numel() * t.element_size() for t in (q, kv, idx) if t is not None)
    if has_bwd:
        in_bytes += dout.numel() * dout.element_size()
    flush = torch.empty((512 << 20,), dtype=torch.uint8, device=dev) if in_bytes < 2 * L2_BYTES \
        else None

    def step(ev=None):
        for k, (_, launch) in enumerate(kernels):
            if ev is not None:
                ev[k].record(stream)
            launch()
        if ev is not None:
            ev[len(kernels)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if lib.smqa_device_status(1) != 0:
        raise RuntimeError("device timeout during warm-up")

    nk = len(kernels)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier(device_ids=[local])
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i & 255)
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier(device_ids=[local])
    torch.cuda.synchronize(dev)
    if lib.smqa_device_status(1) != 0:
        raise RuntimeError("device timeout during the timed region")
    # With the flush, the step time is the sum of the steps' own spans.
    elapsed_ms = (sum(e[0].elapsed_time(e[nk]) for e in evs) if flush is not None
                  else start.elapsed_time(end))
    kms = {nm: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in evs)
           for k, (nm, _) in enumerate(kernels)}
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    ms_step = elapsed_ms / args.steps
    value = whole_job_rate(world, f_step, args.steps, elapsed_ms) / 1e12

    t_sink = t_det = None
    if has_bwd and not args.no_extras:
        t_sink, t_det = time_extras(lib, shp, q, kv, sink, o, dout, idx, lse, delta, dq, dkv,
                                    scale, stream, sp, dev)

    # End to end through the public API: page-locked host inputs -> device,
    # the kernels, results -> page-locked host, every step.
    host = {k: v.cpu().pin_memory() for k, v in (("q", q), ("kv", kv), ("sink", sink),
                                                 ("idx", idx))}
    if has_bwd:
        host["do"] = dout.cpu().pin_memory()
    outs = {"o": torch.empty_like(host["q"]).pin_memory(),
            "lse": torch.empty((B, S, H), dtype=torch.float32).pin_memory()}
    if has_bwd:
        outs["dq"] = torch.empty_like(host["q"]).pin_memory()
        outs["dkv"] = torch.empty((B, S_kv, D), dtype=torch.bfloat16).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    if has_bwd:
        ws = torch.empty((int(lib.smqa_fwd_bwd_host_workspace_bytes(shp, 0)),),
                         dtype=torch.uint8, device=dev)
        f_e2e = f_fwd + f_bwd

        def e2e_step():
            sparse_mqa_fwd_bwd_host(host["q"], host["kv"], host["sink"], host["idx"], host["do"],
                                    device=dev, workspace=ws, out=outs, synchronize=False)
    else:
        ws = torch.empty((max(int(lib.smqa_fwd_host_workspace_bytes(shp)), 256),),
                         dtype=torch.uint8, device=dev)
        f_e2e = f_fwd

        def e2e_step():
            sparse_mqa_fwd_host(host["q"], host["kv"], host["sink"], host["idx"], device=dev,
                                workspace=ws, out=outs, synchronize=False)

    e2e_value, e2e_windows = None, []
    if args.e2e_steps > 0:
        e2e_step()
        torch.cuda.synchronize(dev)
        for _ in range(args.e2e_windows):
            if dist is not None:
                dist.barrier(device_ids=[local])
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.e2e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_windows.append(max_over_ranks(e0.elapsed_time(e1), dist, dev))
        e2e_ms = statistics.median(e2e_windows)
        e2e_value = whole_job_rate(world, f_e2e, args.e2e_steps, e2e_ms) / 1e12
        if lib.smqa_device_status(1) != 0:
            raise RuntimeError("device timeout in the end-to-end leg")

    if rank != 0:
        return None
    pk, src = peaks()
    peak_tf = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")))
    hbm = float(pk.get("hbm_gbs"))
    T = B * S
    fwd_bytes, bwd_bytes = algorithmic_bytes(cfg, n_valid)

    def slower_of(flops, nbytes, ms):
        return {"measured_hbm": max(flops / (peak_tf * 1e12), nbytes / (hbm * 1e9)) / (ms * 1e-3),
                "nominal_8tbs": max(flops / (peak_tf * 1e12),
                                    nbytes / (NOMINAL_HBM_GBS * 1e9)) / (ms * 1e-3)}

    dom = "bwd_main" if has_bwd else "fwd"
    f_dom = f_bwd if has_bwd else f_fwd
    ach = f_dom / (kms[dom] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload, "B": B, "S": S, "S_kv": S_kv, "H": H, "D": D,
                   "topk": K, "index_recipe": cfg.recipe, "passes": cfg.passes,
                   "valid_slots": n_valid,
                   "l2": ("inputs smaller than L2: a 512 MiB write between timed steps, "
                          "outside the step spans") if flush is not None else
                         "inputs larger than L2 (q, dO, o, dq stream from HBM); kv stays "
                         "L2-resident by design",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor",
                     "kernel": "smqa_bwd_kernel (bwd main)" if has_bwd else "smqa_fwd_kernel",
                     "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s", "frac": ach / peak_tf,
                     "peak_source": f"{src} bf16 sustained (kernel timed inside a long step)",
                     "traffic": recorded_traffic() if (has_bwd and name == WORKLOAD and
                                                       not args.seq and not tok) else None},
        "kernels_ms": kms,
        "tokens_per_s": whole_job_rate(world, T, args.steps, elapsed_ms),
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "windows_ms": [round(w, 3) for w in e2e_windows],
                "window": f"median of {len(e2e_windows)} windows of `steps` steps",
                "entry": "smqa_fwd_bwd_host" if has_bwd else "smqa_fwd_host",
                "flops": "fwd+bwd" if has_bwd else "fwd"},
        "gpu_launches": nk * args.steps,
        "clocks": clk.summary(),
    }
    if has_fwd:
        t = kms["fwd"]
        line["fwd"] = {"tflops": f_fwd / (t * 1e-3) / 1e12, "ms": t,
                       "frac_tensor": f_fwd / (t * 1e-3) / 1e12 / peak_tf,
                       "frac_roofline_slower_of": slower_of(f_fwd, fwd_bytes, t)}
    if has_bwd:
        t = kms["bwd_pre"] + kms["bwd_main"] + kms["bwd_post"]
        line["bwd"] = {"tflops": f_bwd / (t * 1e-3) / 1e12, "ms": t,
                       "frac_tensor": f_bwd / (t * 1e-3) / 1e12 / peak_tf,
                       "frac_roofline_slower_of": slower_of(f_bwd, bwd_bytes, t)}
        line["bwd_deterministic"] = None if t_det is None else {
            "ms": t_det, "vs_atomic_bwd": t_det / t,
            "note": "smqa_bwd with SMQA_FLAG_DETERMINISTIC_DKV, timed alone (5 calls), "
                    "not in the step"}
        line["sink_grad"] = None if t_sink is None else {
            "ms": t_sink, "bytes": 8 * T * H + 8 * H,
            "gbs": (8 * T * H + 8 * H) / (t_sink * 1e-3) / 1e9,
            "note": "dsink kernel timed alone (20 launches), not in the step"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, cfg, workload)
    return line


def run_indexer_workload(args, name, dist, world, rank, local, dev):
    """The lightning-indexer backward (its own kernel; not part of the
    attention step): one launch per step over the whole workload."""
    cfg = inputs.indexer_by_name(name)
    x = inputs.make_indexer_inputs(cfg, device=str(dev))
    q, w, k, idx, g = (x["index_q"][0], x["weights"][0], x["index_k"][0], x["topk_indices"][0],
                       x["grad_scores"][0])
    S, S_kv, H, D, K = cfg.S, cfg.S_kv, cfg.H, cfg.D, cfg.topk
    n_valid = int(((idx >= 0) & (idx < S_kv)).sum().item())
    flops = 4.0 * H * D * n_valid          # L = q.k^T and dq += G.k, valid slots
    nbytes = 2 * D * n_valid + 4 * H * D * S + 8 * K * S + 4 * H * S
    lib = _lib.load()
    shp = _lib.Shape(1, S, S_kv, H, D, K)
    dq = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def launch():
        _lib.check("indexer", lib.smqa_indexer_bwd(P(q), P(w), P(k), P(idx), P(g), shp, P(dq), sp))

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier(device_ids=[local])
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            evs[i][0].record(stream)
            launch()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier(device_ids=[local])
    if lib.smqa_device_status(1) != 0:
        raise RuntimeError("device timeout in the indexer backward")
    elapsed_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs), dist, dev)
    t = elapsed_ms / args.steps
    value = whole_job_rate(world, flops, args.steps, elapsed_ms) / 1e12

    # End to end: page-locked host inputs -> device, the call, dq -> host.
    host = {kk: v.cpu().pin_memory() for kk, v in (("q", q), ("w", w), ("k", k), ("idx", idx),
                                                   ("g", g))}
    dev_in = {kk: torch.empty_like(v, device=dev) for kk, v in host.items()}
    out = torch.empty_like(host["q"]).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out.numel() * out.element_size()

    def e2e_step():
        for kk in host:
            dev_in[kk].copy_(host[kk], non_blocking=True)
        dd = dev_in
        _lib.check("indexer", lib.smqa_indexer_bwd(P(dd["q"]), P(dd["w"]), P(dd["k"]),
                                                   P(dd["idx"]), P(dd["g"]), shp, P(dq), sp))
        out.copy_(dq, non_blocking=True)

    e2e_windows = []
    if args.e2e_steps > 0:
        e2e_step()
        torch.cuda.synchronize(dev)
        for _ in range(args.e2e_windows):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.e2e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_windows.append(max_over_ranks(e0.elapsed_time(e1), dist, dev))
    e2e_value = (whole_job_rate(world, flops, args.e2e_steps, statistics.median(e2e_windows))
                 / 1e12 if e2e_windows else None)
    if rank != 0:
        return None
    pk, src = peaks()
    peak_tf = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")))
    hbm = float(pk.get("hbm_gbs"))
    ach = flops / (t * 1e-3) / 1e12
    line = {
        "metric": "lightning-indexer backward TFLOP/s + % BF16 roofline, 1\u00d7GB300",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": 1, "S": S, "S_kv": S_kv, "H": H, "D": D, "topk": K,
                   "index_recipe": cfg.recipe, "valid_slots": n_valid,
                   "l2": "inputs larger than L2 (index_q, dq 128 MiB each, the index rows and "
                         "grad_scores 64 MiB each); index_k 2 MiB stays L2-resident",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "smqa_indexer_bwd_kernel", "achieved": ach,
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": ach / peak_tf,
                     "peak_source": f"{src} bf16 sustained",
                     "note": "H=64 fills half of the 128-row MMA tile; FLOPs count the 64 "
                             "heads only", "traffic": None,
                     "frac_slower_of_measured_hbm":
                         max(flops / (peak_tf * 1e12), nbytes / (hbm * 1e9)) / (t * 1e-3)},
        "kernels_ms": {"indexer_bwd": t},
        "tokens_per_s": whole_job_rate(world, S, args.steps, elapsed_ms),
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "windows_ms": [round(v, 3) for v in e2e_windows],
                "window": f"median of {len(e2e_windows)} windows of `steps` steps",
                "entry": "smqa_indexer_bwd with torch copies from / to page-locked memory"},
        "gpu_launches": args.steps, "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import numpy as np

        import oracle
        rng = np.random.default_rng(4321)
        xc = {kk: v.cpu() for kk, v in (("q", q), ("w", w), ("k", k), ("idx", idx), ("g", g))}

        def run(n):
            toks = np.sort(rng.choice(S, size=n, replace=False))
            nv = int(((xc["idx"][torch.as_tensor(toks)] >= 0) &
                      (xc["idx"][torch.as_tensor(toks)] < S_kv)).sum())
            t0 = time.perf_counter()
            oracle.indexer_bwd(xc["q"], xc["w"], xc["k"], xc["idx"], xc["g"], tokens=toks)
            return time.perf_counter() - t0, nv

        dt, _ = run(8)
        n = int(max(8, min(2048, 8 * 15.0 / max(dt, 1e-3))))
        dt, nv = run(n)
        line["cpu_baseline"] = {"value": 4.0 * H * D * nv / dt / 1e12, "unit": "TFLOP/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{n} seeded tokens of {name} (fp64), {dt:.1f} s"}
    return line


def time_extras(lib, shp, q, kv, sink, o, dout, idx, lse, delta, dq, dkv, scale, stream, sp,
                dev):
    """The optional backward paths outside the step, each timed alone: the
    sink gradient kernel and the deterministic-dKV backward."""
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dsink = torch.empty((shp.H,), dtype=torch.float32, device=dev)

    def sink_grad():
        _lib.check("sink", lib.smqa_bwd_sink_grad(P(sink), P(lse), P(delta), shp, P(dsink), sp))

    for _ in range(3):
        sink_grad()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(20):
        sink_grad()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    t_sink = s0.elapsed_time(s1) / 20

    det = _lib.FLAG_DETERMINISTIC_DKV
    det_ws = torch.empty((int(lib.smqa_bwd_workspace_bytes(shp, det)),), dtype=torch.uint8,
                         device=dev)

    def det_bwd():
        _lib.check("det", lib.smqa_bwd(P(q), P(kv), P(sink), P(o), P(dout), P(idx), P(lse),
                                       shp, scale, P(dq), P(dkv), None, P(det_ws),
                                       det_ws.numel(), det, sp))

    for _ in range(2):
        det_bwd()
    s0.record(stream)
    for _ in range(5):
        det_bwd()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    t_det = s0.elapsed_time(s1) / 5
    if lib.smqa_device_status(1) != 0:
        raise RuntimeError("device timeout in the deterministic backward")
    return t_sink, t_det


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[c.name for c in inputs.CONFIGS] +
                    [c.name for c in inputs.INDEXER_CONFIGS] + ["all"],
                    help="the workload to time (default: the H=128 D=512 topk=2048 one); "
                         "'all' prints one line per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-windows", type=int, default=7)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the timings of the optional paths outside the step "
                         "(deterministic-dKV backward, sink gradient)")
    ap.add_argument("--seq", type=int, default=None,
                    help="profiling only: override S = S_kv (the bench line then names the "
                         "smaller workload)")
    ap.add_argument("--tokens", default=None,
                    help="profiling only: A:B times the query positions [A, B) of the "
                         "workload (e.g. 7168:8192, full-length index rows)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.e2e_windows < 5:
        ap.error("--e2e-windows must be >= 5")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")
    if args.impl == "reference":
        reference_arm(args, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    names = ([c.name for c in inputs.CONFIGS] + [c.name for c in inputs.INDEXER_CONFIGS]
             if args.workload == "all" else [args.workload])
    indexer_names = {c.name for c in inputs.INDEXER_CONFIGS}
    for name in names:
        run = run_indexer_workload if name in indexer_names else run_workload
        line = run(args, name, dist, world, rank, local, dev)
        if line is not None:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
