#!/usr/bin/env python
"""Benchmark: top-k sparse MQA forward + backward on GB300.

One step = the whole hot path over one batch: forward (O, log2 LSE), then the
backward's preprocess (Delta and zeroing of the fp32 dKV accumulator), main
kernel (dQ, dKV scatter) and postprocess (dKV to bf16).  Workload: B=1,
S=S_kv=8192, H=128, D=512, topk=2048, indices causal and biased to the
newest 512 keys (the H=128 D=512 topk=2048 configuration).  Inputs are
synthetic and seeded; q, o, dO and dq are 1 GiB each (larger than L2), kv
(8 MiB) stays L2-resident as it would in the real workload.

Metric: TFLOP/s of the step, FLOPs counted on valid slots only
(4*H*D per valid slot forward, 10*H*D backward).  `value` times the kernels
on device-resident inputs; `e2e` times the host-buffer entry point
(smqa_fwd_bwd_host: page-locked inputs in, results out, copies overlapped
with the kernels in token chunks).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
(the op shards by tokens with no data-path collective) and the timed region
is bracketed by barriers; value = all ranks' FLOPs / the slowest rank's time.
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
from bwd_sparse_mqa_gb300 import sparse_mqa_fwd_bwd_host  # noqa: E402

WORKLOAD = "h128_d512_k2048_s8192"
METRIC = "sparse MQA fwd/bwd TFLOP/s + % BF16 roofline, 1×GB300, H=128 D=512 topk=2048"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
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


def cpu_baseline(x: dict, cfg, target_s: float = 15.0, max_tokens: int = 512):
    """The fp64 oracle as it stands, on the host cores, fwd+bwd over a seeded
    token sample of the workload sized to ~target_s seconds."""
    import numpy as np

    import oracle
    q, kv, sink, idx, dout = (x["q"].cpu(), x["kv"].cpu(), x["attn_sink"].cpu(),
                              x["topk_idxs"].cpu(), x["do"].cpu())
    rng = np.random.default_rng(1234)
    T = cfg.B * cfg.S

    def run(n):
        toks = np.sort(rng.choice(T, size=n, replace=False))
        sel = idx.reshape(T, -1)[torch.as_tensor(toks)]
        nv = int(((sel >= 0) & (sel < cfg.S_kv)).sum())
        t0 = time.perf_counter()
        oracle.fwd(q, kv, sink, idx, tokens=toks)
        oracle.bwd(q, kv, sink, idx, dout, tokens=toks)
        return time.perf_counter() - t0, nv

    probe_n = 4
    dt, _ = run(probe_n)
    n = int(max(probe_n, min(max_tokens, probe_n * target_s / max(dt, 1e-3))))
    dt, nv = run(n)
    fl = 14.0 * cfg.H * cfg.D * nv
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} seeded tokens of {WORKLOAD} (fwd+bwd, fp64, {nv} valid slots), "
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
    cfg = inputs.by_name(WORKLOAD)
    workload = WORKLOAD
    if args.seq:
        import dataclasses
        cfg = dataclasses.replace(cfg, S=args.seq, S_kv=args.seq)
        workload = f"{WORKLOAD} with S=S_kv={args.seq} (profiling size)"
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = inputs.make_inputs(cfg, device=dev)
    q, kv, sink, idx, dout = (x["q"].cpu(), x["kv"].cpu(), x["attn_sink"].cpu(),
                              x["topk_idxs"].cpu(), x["do"].cpu())
    T = cfg.B * cfg.S
    per_step = int(os.environ.get("SMQA_REF_TOKENS_PER_STEP", "8"))
    rng = np.random.default_rng(99)

    def step():
        toks = np.sort(rng.choice(T, size=per_step, replace=False))
        sel = idx.reshape(T, -1)[torch.as_tensor(toks)]
        nv = int(((sel >= 0) & (sel < cfg.S_kv)).sum())
        oracle.fwd(q, kv, sink, idx, tokens=toks)
        oracle.bwd(q, kv, sink, idx, dout, tokens=toks)
        return 14.0 * cfg.H * cfg.D * nv

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
                       "H": cfg.H, "D": cfg.D, "topk": cfg.topk,
                       "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{per_step} seeded tokens per step (fwd+bwd, fp64)"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the timings of the optional paths outside the step "
                         "(deterministic-dKV backward, sink gradient)")
    ap.add_argument("--seq", type=int, default=None,
                    help="profiling only: override S = S_kv (the bench line then names the "
                         "smaller workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

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
    cfg = inputs.by_name(WORKLOAD)
    workload = WORKLOAD
    if args.seq:
        import dataclasses
        cfg = dataclasses.replace(cfg, S=args.seq, S_kv=args.seq)
        workload = f"{WORKLOAD} with S=S_kv={args.seq} (profiling size)"
    x = inputs.make_inputs(cfg, device=str(dev))
    q, kv, sink, idx, dout = x["q"], x["kv"], x["attn_sink"], x["topk_idxs"], x["do"]
    B, S, S_kv, H, D, K = cfg.B, cfg.S, cfg.S_kv, cfg.H, cfg.D, cfg.topk
    f_fwd, f_bwd, n_valid = flops_of(idx, S_kv, H, D)
    lib = _lib.load()
    shp = _lib.Shape(B, S, S_kv, H, D, K)
    o = torch.empty_like(q)
    lse = torch.empty((B, S, H), dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dkv = torch.empty((B, S_kv, D), dtype=torch.bfloat16, device=dev)
    acc = torch.empty((B, S_kv, D), dtype=torch.float32, device=dev)
    delta = torch.empty((B, S, H), dtype=torch.float32, device=dev)
    # One exchange pool serves the forward and the backward main kernel (they
    # run one after the other on the stream).
    exch_bytes = max(int(lib.smqa_fwd_workspace_bytes(shp)), int(lib.smqa_bwd_exchange_bytes(shp)))
    exch = torch.empty((max(exch_bytes, 256),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    scale = D ** -0.5

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        _lib.check("smqa_fwd", lib.smqa_fwd(P(q), P(kv), P(sink), P(idx), shp, scale, P(o), P(lse),
                                            P(exch), exch_bytes, 0, sp))
        if ev is not None:
            ev[1].record(stream)
        _lib.check("pre", lib.smqa_bwd_preprocess(P(o), P(dout), shp, P(delta), P(acc), sp))
        if ev is not None:
            ev[2].record(stream)
        _lib.check("main", lib.smqa_bwd_main(P(q), P(kv), P(sink), P(dout), P(idx), P(lse),
                                             P(delta), shp, scale, P(dq), P(acc), P(exch),
                                             exch_bytes, sp))
        if ev is not None:
            ev[3].record(stream)
        _lib.check("post", lib.smqa_bwd_postprocess(P(acc), shp, P(dkv), sp))
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if lib.smqa_device_status(1) != 0:
        raise RuntimeError("device timeout during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier(device_ids=[local])
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier(device_ids=[local])
    torch.cuda.synchronize(dev)
    elapsed_ms = start.elapsed_time(end)
    if lib.smqa_device_status(1) != 0:
        raise RuntimeError("device timeout during the timed region")
    t_fwd = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    t_pre = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    t_main = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    t_post = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    ms_step = elapsed_ms / args.steps
    value = whole_job_rate(world, f_fwd + f_bwd, args.steps, elapsed_ms) / 1e12

    def time_extras():
        """The optional paths outside the step, each timed alone."""
        # The sink gradient (an optional backward output the pages do not return,
        # so not part of the step): its own kernel, timed alone on the step's
        # Delta and LSE.
        dsink = torch.empty((H,), dtype=torch.float32, device=dev)

        def sink_grad():
            _lib.check("sink", lib.smqa_bwd_sink_grad(P(sink), P(lse), P(delta), shp, P(dsink),
                                                      sp))

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

        # The deterministic-dKV backward (fixed-point integer accumulation; an
        # option, not part of the step): the whole smqa_bwd call, timed alone.
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

    t_sink = t_det = None
    if not args.no_extras:
        t_sink, t_det = time_extras()

    # end to end through the public API: pinned host inputs -> device, fwd,
    # bwd, results -> pinned host, every step
    host = {k: v.cpu().pin_memory() for k, v in (("q", q), ("kv", kv), ("sink", sink),
                                                 ("idx", idx), ("do", dout))}
    outs = {"o": torch.empty_like(host["q"]).pin_memory(),
            "lse": torch.empty((B, S, H), dtype=torch.float32).pin_memory(),
            "dq": torch.empty_like(host["q"]).pin_memory(),
            "dkv": torch.empty((B, S_kv, D), dtype=torch.bfloat16).pin_memory()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    ws = torch.empty((int(lib.smqa_fwd_bwd_host_workspace_bytes(shp, 0)),), dtype=torch.uint8,
                     device=dev)

    def e2e_step():
        # one call: chunked host->device copies, forward, backward and
        # device->host copies, overlapped on the library's streams
        sparse_mqa_fwd_bwd_host(host["q"], host["kv"], host["sink"], host["idx"], host["do"],
                                device=dev, workspace=ws, out=outs, synchronize=False)

    # Two timed windows of e2e_steps steps each; the faster one is reported and
    # both are listed: a window now and then runs ~2.5x longer (seen with every
    # chunk plan, in whole windows), which the host-side copies point to.
    e2e_value = None
    e2e_windows = []
    if args.e2e_steps > 0:
        e2e_step()
        torch.cuda.synchronize(dev)
        for _ in range(2):
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
        e2e_ms = min(e2e_windows)
        e2e_value = whole_job_rate(world, f_fwd + f_bwd, args.e2e_steps, e2e_ms) / 1e12

    if rank == 0:
        pk, src = peaks()
        peak_tf = float(pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")))
        hbm = float(pk.get("hbm_gbs"))
        ach_main = f_bwd / (t_main * 1e-3) / 1e12
        ach_fwd = f_fwd / (t_fwd * 1e-3) / 1e12
        T = B * S
        # bytes per the op's algorithmic accounting (valid slots)
        fwd_bytes = 2 * D * n_valid + 4 * H * D * T + 4 * K * T + 4 * H * T
        bwd_bytes = 6 * D * n_valid + 8 * H * D * T + 4 * K * T + 8 * H * T + 10 * B * S_kv * D
        bwd_ms = t_pre + t_main + t_post
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload, "B": B, "S": S, "S_kv": S_kv, "H": H, "D": D,
                       "topk": K, "index_recipe": cfg.recipe, "valid_slots": n_valid,
                       "l2": "inputs larger than L2 (q, o, dO, dq 1 GiB each); kv 8 MiB stays "
                             "L2-resident by design",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "kernel": "smqa_bwd_kernel<256,2> (bwd main)",
                         "achieved": ach_main, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": ach_main / peak_tf, "peak_source":
                         f"{src} bf16 sustained (kernel timed inside a long step)",
                         "traffic": recorded_traffic()},
            "kernels_ms": {"fwd": t_fwd, "bwd_pre": t_pre, "bwd_main": t_main,
                           "bwd_post": t_post},
            "fwd": {"tflops": ach_fwd, "ms": t_fwd, "frac_tensor": ach_fwd / peak_tf,
                    "frac_roofline_slower_of":
                        max(f_fwd / (peak_tf * 1e12), fwd_bytes / (hbm * 1e9)) / (t_fwd * 1e-3)},
            "bwd": {"tflops": f_bwd / (bwd_ms * 1e-3) / 1e12, "ms": bwd_ms,
                    "frac_tensor": f_bwd / (bwd_ms * 1e-3) / 1e12 / peak_tf,
                    "frac_roofline_slower_of":
                        max(f_bwd / (peak_tf * 1e12), bwd_bytes / (hbm * 1e9)) / (bwd_ms * 1e-3)},
            "tokens_per_s": whole_job_rate(world, T, args.steps, elapsed_ms),
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                    "windows_ms": [round(w, 3) for w in e2e_windows],
                    "window": "faster of two windows of `steps` steps"},
            "gpu_launches": 4 * args.steps,
            "bwd_deterministic": None if t_det is None else {
                "ms": t_det, "vs_atomic_bwd": t_det / bwd_ms,
                "note": "smqa_bwd with SMQA_FLAG_DETERMINISTIC_DKV, timed alone (5 calls), "
                        "not in the step"},
            "sink_grad": None if t_sink is None else {
                "ms": t_sink, "bytes": 8 * T * H + 8 * H,
                "gbs": (8 * T * H + 8 * H) / (t_sink * 1e-3) / 1e9,
                "note": "dsink kernel timed alone (20 launches), not in the step"},
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(x, cfg)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
