"""Benchmark of the fused attention forward on GB300.

One step = one attn_fwd call over the whole workload (default: the causal
b=1, h=32, s=16384, d=128 bf16 problem with Q, K ~ N(0, 9)).  Prints one JSON
line (rank 0).  Work is counted as 4*b*h*sq*sk*d FLOPs, half of it when
causal; `value` is whole-job TFLOPS over all ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
problem of the same shape (the forward has no exchange step), so scaling is
weak; the only collectives are the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS on 1 GB300 (d=128, bf16, causal) and % of dense tensor peak"
METRIC_BWD = "attention bwd TFLOPS on 1 GB300 (d=128, bf16, causal) and % of dense tensor peak"
L2_BYTES = 129e6


def shard_heads(bh: int, world: int, rank: int):
    """Contiguous [start, end) range of the b*h heads owned by `rank` when one
    problem is split across ranks (heads are independent: no exchange)."""
    base, rem = divmod(bh, world)
    start = rank * base + min(rank, rem)
    return start, start + base + (1 if rank < rem else 0)


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's time (the job finishes when the last rank does)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(bf16=float(d["bf16_tflops"]), bf16_sustained=float(d["bf16_tflops_sustained"]),
                    hbm=float(d["hbm_gbs"]), source="measured")
    return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, source="fallback")


# Device sources of each kernel family: the counters in profiles/ are tied
# to these (host-side API code does not change what a kernel reads/writes).
KERNEL_SOURCES = {
    "attn_fwd_kernel": ["ptx.cuh", "attn_fwd_kernel.cuh", "launch.h", "inst_d64.cu", "inst_d128_noncausal.cu",
                        "inst_d128_causal.cu", "inst_fp8.cu"],
    "attn_bwd_kernel": ["ptx.cuh", "attn_bwd_kernel.cuh", "attn_bwd_launch.h", "attn_bwd_inst.cu"],
}


def kernel_source_hash(kernel: str = "attn_fwd_kernel"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_14_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "attn_fwd_kernel"):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    or None when no summary exists or the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(w, q, k, v, target_s: float = 12.0, want_rows: bool = False):
    """The fp64 oracle, as it stands, on the host cores: a bounded sample of
    query rows of the first head, sized to ~target_s seconds.  Returns
    (TFLOPS, description, cores, seconds), and with want_rows also the
    sampled rows and the oracle's O and LSE for them."""
    import numpy as np
    import oracle

    qh, kh, vh = (t[0, 0].double().numpy() for t in (q, k, v))
    cores = oracle.num_threads()

    def visible(rows):
        if not w.causal:
            return np.full(len(rows), w.sk, dtype=np.float64)
        return np.clip(np.asarray(rows) + 1 + (w.sk - w.sq), 0, w.sk).astype(np.float64)

    last = {}

    def run(rows):
        t0 = time.perf_counter()
        last["o"], last["lse"] = oracle.attn_head_rows(qh, kh, vh, rows, w.causal, w.scale)
        return time.perf_counter() - t0

    rng = np.random.default_rng(w.seed)
    probe = np.sort(rng.choice(w.sq, size=min(w.sq, 4 * cores), replace=False))
    dt = run(probe)
    rate = 4.0 * w.d * visible(probe).sum() / max(dt, 1e-6)  # flop/s of the oracle
    per_row = 4.0 * w.d * visible(np.arange(w.sq)).mean()
    n = int(min(w.sq, max(len(probe), target_s * rate / per_row)))
    rows = np.sort(rng.choice(w.sq, size=n, replace=False))
    dt = run(rows)
    flops = 4.0 * w.d * visible(rows).sum()
    desc = (f"{n} seeded query rows of head (0,0) of {w.name}, each against all its visible keys "
            f"({flops / 1e9:.1f} GFLOP counted as 4*d per visible key)")
    if want_rows:
        return flops / dt / 1e12, desc, cores, dt, (rows, last["o"], last["lse"])
    return flops / dt / 1e12, desc, cores, dt


def bench_reference(args, w):
    """The oracle arm: each step is one bounded sample (fp64, host cores)."""
    from attention_forward_14_gb300 import workloads as W
    q, k, v = W.inputs(w)
    per = max(1.0, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(w, q, k, v, target_s=per / 4)
    vals, descs, times = [], [], []
    cores = None
    for _ in range(args.steps):
        tf, desc, cores, dt = cpu_baseline(w, q, k, v, target_s=per)
        vals.append(tf)
        descs.append(desc)
        times.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "b": w.b, "h": w.h, "sq": w.sq, "sk": w.sk, "d": w.d,
                   "causal": w.causal, "input_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": descs[-1]},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_varlen(args, w):
    """Packed variable-length workload: one step = one attn_fwd_varlen call."""
    import torch
    import attention_forward_14_gb300 as af
    from attention_forward_14_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v, cu_q, cu_k, _ = W.varlen_inputs(w)
    lens = w.lengths()
    qd, kd, vd, cqd, ckd = q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.h, q.shape[0]), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        af.attn_fwd_varlen(qd, kd, vd, cqd, ckd, max(lens), max(lens), causal=w.causal, scale=w.scale, o=o, lse=lse,
                           stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    peaks = load_peaks()
    value = w.flops() / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "sequences": w.n, "lengths": lens, "total_tokens": int(q.shape[0]), "h": w.h,
                   "d": w.d, "causal": w.causal, "flops_per_step": w.flops()},
        "pct_of_peak": 100.0 * value / peaks["bf16"],
        "roofline": {"bound": "tensor", "achieved": value, "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": value / peaks["bf16"], "traffic": profiled_traffic(w.name),
                     "peak_kind": f"{peaks['source']} bf16 dense burst (cuBLAS)", "kernel": "attn_fwd_kernel",
                     "algorithmic_bytes": w.bytes()},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_kvcache(kw, q, kc, vc, kn, vn, lens, heads: int = 8):
    """The fp64 KV-cache oracle, as it stands, on the host cores: all
    sequences of the decode step, `heads` of their heads, the caches cut to
    the longest valid length.  Returns (TFLOPS, description, cores, seconds)."""
    import oracle

    hs = slice(0, min(heads, kw.h))
    need = min(kw.cap, max(min(max(int(x), 0), kw.cap) + kw.s_new for x in lens.tolist()))
    args = [t[:, hs].double().numpy() for t in (q, kc[:, :, :need], vc[:, :, :need], kn, vn)]
    t0 = time.perf_counter()
    oracle.attn_fwd_kvcache(args[0], args[1], args[2], lens.tolist(), args[3], args[4], kw.causal, kw.scale)
    dt = time.perf_counter() - t0
    flops = kw.flops() * (hs.stop / kw.h)
    desc = (f"heads 0..{hs.stop - 1} of all {kw.b} sequences of {kw.name} (cache write and attention, caches "
            f"cut to {need} slots; {flops / 1e9:.2f} GFLOP counted as 4*d per visible key)")
    return flops / dt / 1e12, desc, oracle.num_threads(), dt


def bench_kvcache(args, kw):
    """KV-cache decode workload: one step = one attn_fwd_kvcache call (the
    cache write, the split-KV forward and the combine)."""
    import torch
    import attention_forward_14_gb300 as af
    from attention_forward_14_gb300 import binding
    from attention_forward_14_gb300 import workloads as W

    q, kc, vc, kn, vn, lens = W.kvcache_inputs(kw)
    table = None
    if kw.page_size:
        _, kc_pool, vc_pool, _, _, _, table = W.kvcache_paged_inputs(kw)
    if args.impl == "reference":
        per = max(1.0, 120.0 / max(1, args.steps + args.warmup))
        vals, times, desc, cores = [], [], "", None
        for i in range(args.warmup + args.steps):
            tf, desc, cores, dt = cpu_baseline_kvcache(kw, q, kc, vc, kn, vn, lens)
            if i >= args.warmup:
                vals.append(tf)
                times.append(dt)
        value = statistics.median(vals)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": kw.name, "b": kw.b, "h": kw.h, "cap": kw.cap, "lengths": kw.lengths(),
                       "s_new": kw.s_new, "d": kw.d, "causal": kw.causal},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if kw.page_size:  # the device holds the pools; the dense caches serve the CPU leg only
        kcd, vcd, tabd = kc_pool.to(dev), vc_pool.to(dev), table.to(dev)
        qd, knd, vnd, lensd = (t.to(dev) for t in (q, kn, vn, lens))
    else:
        qd, kcd, vcd, knd, vnd, lensd = (t.to(dev) for t in (q, kc, vc, kn, vn, lens))
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    splits = args.num_splits or binding.splitkv_default_splits(kw.b, kw.h, kw.sq, kw.cap, kw.d, kw.causal)
    ws = torch.empty(max(16, binding.splitkv_workspace_bytes(kw.b, kw.h, kw.sq, kw.d, splits)), dtype=torch.uint8,
                     device=dev)

    def step():
        if kw.page_size:
            af.attn_fwd_kvcache_paged(qd, kcd, vcd, lensd, tabd, knd, vnd, causal=kw.causal, scale=kw.scale,
                                      num_splits=splits, o=o, lse=lse, workspace=ws, stream=stream)
        else:
            af.attn_fwd_kvcache(qd, kcd, vcd, lensd, knd, vnd, causal=kw.causal, scale=kw.scale, num_splits=splits,
                                o=o, lse=lse, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # end to end: per step the new tokens (q, k_new, v_new) and the lengths
    # go host -> device from pinned memory, O and LSE come back; the cache is
    # the resident state of the decoder and stays on the device.
    qh, knh, vnh, lh = (t.pin_memory() for t in (q, kn, vn, lens))
    oh = torch.empty_like(qh).pin_memory()
    lseh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()

    def e2e_step():
        for src, dst in ((qh, qd), (knh, knd), (vnh, vnd), (lh, lensd)):
            dst.copy_(src, non_blocking=True)
        step()
        oh.copy_(o, non_blocking=True)
        lseh.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = x0.elapsed_time(x1) / args.e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (qh, knh, vnh, lh))
    d2h = oh.numel() * oh.element_size() + lseh.numel() * 4

    peaks = load_peaks()
    value = kw.flops() / (ms * 1e-3) / 1e12
    achieved = kw.bytes() / (kern_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": kw.dtype,
        "data": "synthetic",
        "config": {"workload": kw.name, "b": kw.b, "h": kw.h, "cap": kw.cap, "lengths": kw.lengths(),
                   "s_new": kw.s_new, "d": kw.d, "causal": kw.causal, "flops_per_step": kw.flops(),
                   "page_size": kw.page_size or None,
                   "l2": f"cache {2 * kc.numel() * 2 / 1e9:.1f} GB > L2, valid K/V {kw.bytes() / 1e9:.2f} GB/step, "
                         "no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm"], "traffic": profiled_traffic(kw.name),
                     "peak_kind": f"{peaks['source']} HBM copy",
                     "kernel": "attn_kvcache_append_kernel + attn_fwd_kernel + attn_splitkv_combine_kernel "
                               "(one step)",
                     "algorithmic_bytes": kw.bytes(), "num_splits": splits},
        "e2e": {"value": kw.flops() / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * (2 + (1 if splits > 1 else 0)),
        "clocks": sampler.summary(),
    }
    if not args.no_cpu_baseline:
        tf, desc, cores, dt = cpu_baseline_kvcache(kw, q, kc, vc, kn, vn, lens)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc,
                                "seconds": dt}
    print(json.dumps(line), flush=True)


def bench_bwd(args, bw):
    """Backward workload: one step = one attn_bwd call (prep, main and dQ
    convert kernels) on the forward's outputs, inputs resident in HBM."""
    import torch
    import attention_forward_14_gb300 as af
    from attention_forward_14_gb300 import workloads as W

    if int(os.environ.get("WORLD_SIZE", "1")) != 1:
        raise SystemExit("the backward workloads run on one GPU")
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = bw.w
    q, k, v = W.inputs(w)
    do = W.draw_grad(w.b, w.h, w.sq, w.d, w.dtype, bw.grad_seed)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = af.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(af.bwd_workspace_bytes(w.b, w.h, w.sq, w.d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        af.attn_bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                    stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A problem whose bytes are within twice L2 (with the fp32 dQ accumulator
    # it would largely stay there between steps): a 256 MB write before each
    # timed step, and the step's time from its own event pair.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if bw.bytes() < 2 * L2_BYTES else None
    t0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms = step_ms if flush is not None else t0.elapsed_time(t1) / args.steps
    value = bw.flops() / (ms * 1e-3) / 1e12
    achieved = bw.flops() / (step_ms * 1e-3) / 1e12

    # end to end: H2D of q, k, v, o, dO, lse from pinned memory, the
    # backward, D2H of dq, dk, dv, every step
    hs = [t.cpu().pin_memory() for t in (qd, kd, vd, o, dod, lse)]
    outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
    devs = (qd, kd, vd, o, dod, lse)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        for dst, src in zip(devs, hs):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(outs, (dq, dk, dv)):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    peaks = load_peaks()
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": bw.name, "pass": "backward", "b": w.b, "h": w.h, "sq": w.sq, "sk": w.sk, "d": w.d,
                   "causal": w.causal, "qk_std": w.qk_std, "flops_per_step": bw.flops(),
                   "flops_rule": "2.5 x forward (five products: S, dP, dV, dK, dQ)",
                   "l2": f"{bw.bytes() / 1e6:.0f} MB of inputs and outputs > 2 x L2, no flush" if flush is None else
                   f"{bw.bytes() / 1e6:.0f} MB of inputs and outputs within 2 x L2 {L2_BYTES / 1e6:.0f} MB: "
                   "256 MB flush before each timed step, time from each step's own events"},
        "pct_of_peak": 100.0 * value / peaks["bf16"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16"], "traffic": profiled_traffic(bw.name, "attn_bwd_kernel"),
                     "peak_kind": f"{peaks['source']} bf16 dense burst (cuBLAS)",
                     "kernel": "attn_bwd_kernel (+ prep and dQ convert, timed together)",
                     "algorithmic_bytes": bw.bytes()},
        "e2e": {"value": bw.flops() / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hs),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs), "ms_per_step": e2e_ms},
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        n = min(2048, w.sq, w.sk)
        sub = [t[:1, :1, :n].double().numpy() for t in (q, k, v, do)]
        t_start = time.perf_counter()
        oracle.attn_bwd(*sub, w.causal, w.scale)
        dt = time.perf_counter() - t_start
        f = 2.5 * 4.0 * n * n * w.d * (0.5 if w.causal else 1.0)
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(),
                                "kind": "oracle", "sample": f"backward of the first {n} queries and keys of head 0 "
                                f"(a self-contained block of the same problem), fp64", "seconds": dt}
    print(json.dumps(line), flush=True)


def bench_bwd_varlen(args, bw):
    """Packed backward workload: one step = one attn_bwd_varlen call (prep,
    main and dQ convert kernels) on the packed forward's outputs."""
    import torch
    import attention_forward_14_gb300 as af
    from attention_forward_14_gb300 import workloads as W

    if int(os.environ.get("WORLD_SIZE", "1")) != 1:
        raise SystemExit("the backward workloads run on one GPU")
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = bw.w
    lens = w.lengths()
    q, k, v, cu_q, cu_k, _ = W.varlen_inputs(w)
    do = W.bwd_varlen_grad(bw)
    qd, kd, vd, dod, cqd, ckd = (t.to(dev) for t in (q, k, v, do, cu_q, cu_k))
    mx = max(lens)
    o, lse = af.attn_fwd_varlen(qd, kd, vd, cqd, ckd, mx, mx, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    stream = torch.cuda.current_stream(dev)
    from attention_forward_14_gb300 import binding
    need = int(binding.load().attn_bwd_varlen_workspace_bytes(len(lens), w.h, q.shape[0], mx, w.d))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    def step():
        af.attn_bwd_varlen(qd, kd, vd, o, dod, lse, cqd, ckd, mx, mx, causal=w.causal, scale=w.scale, dq=dq, dk=dk,
                           dv=dv, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A problem whose bytes are within twice L2 (with the fp32 dQ accumulator
    # it would largely stay there between steps): a 256 MB write before each
    # timed step, and the step's time from its own event pair.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if bw.bytes() < 2 * L2_BYTES else None
    t0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms = step_ms if flush is not None else t0.elapsed_time(t1) / args.steps
    value = bw.flops() / (ms * 1e-3) / 1e12
    achieved = bw.flops() / (step_ms * 1e-3) / 1e12

    # end to end: H2D of q, k, v, o, dO, lse and the offsets from pinned
    # memory, the backward, D2H of dq, dk, dv, every step
    devs = (qd, kd, vd, o, dod, lse, cqd, ckd)
    hs = [t.cpu().pin_memory() for t in devs]
    outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        for dst, src in zip(devs, hs):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(outs, (dq, dk, dv)):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    peaks = load_peaks()
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": bw.name, "pass": "backward", "sequences": w.n, "lengths": lens,
                   "total_tokens": int(q.shape[0]), "h": w.h, "d": w.d, "causal": w.causal,
                   "flops_per_step": bw.flops(), "flops_rule": "2.5 x forward (five products: S, dP, dV, dK, dQ)",
                   "l2": "inputs larger than L2, no flush"},
        "pct_of_peak": 100.0 * value / peaks["bf16"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16"], "traffic": profiled_traffic(bw.name, "attn_bwd_kernel"),
                     "peak_kind": f"{peaks['source']} bf16 dense burst (cuBLAS)",
                     "kernel": "attn_bwd_kernel (+ prep and dQ convert, timed together)",
                     "algorithmic_bytes": bw.bytes()},
        "e2e": {"value": bw.flops() / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hs),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs), "ms_per_step": e2e_ms},
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)


def _finish_fp8(args, w, world, rank, dist, dev, q, k, v, qd, kd, vd, o, lse, stream, t_all0, t_all1, total_ms,
                launch_ms, sampler, step, l2_note):
    """e4m3 line: roofline against the 8-bit tensor peak (measured bf16 peak
    x the nominal fp8/bf16 ratio 2); e2e = H2D of q, k, v (pinned), the
    forward, D2H of O and LSE, each step."""
    import torch
    ms = total_ms / args.steps
    value = world * w.flops() / (ms * 1e-3) / 1e12
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        step()
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dist, dev)
    if rank == 0:
        peaks = load_peaks()
        peak8 = 2.0 * peaks["bf16"]
        kern_ms = statistics.mean(launch_ms)
        achieved = w.flops() / (kern_ms * 1e-3) / 1e12
        # arithmetic intensity under the ridge of the measured peaks: memory is the roof
        below_ridge = w.flops() / w.bytes() < peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": w.name, "b": w.b, "h": w.h, "sq": w.sq, "sk": w.sk, "d": w.d, "causal": w.causal,
                       "flops_per_step": w.flops(), "output": "bf16", "l2": l2_note},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak8, "unit": "TFLOP/s",
                         "frac": achieved / peak8, "traffic": profiled_traffic(w.name),
                         "peak_kind": f"{peaks['source']} bf16 burst x 2 (nominal fp8/bf16 ratio)",
                         "kernel": f"attn_fwd_kernel<{w.d}, e4m3>", "algorithmic_bytes": w.bytes()},
            "e2e": {"value": world * w.flops() / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                    "h2d_bytes_per_step": q.numel() + k.numel() + v.numel(),
                    "d2h_bytes_per_step": 2 * o.numel() + 4 * lse.numel(),
                    "ms_per_step": e2e_ms},
            "gpu_launches": args.steps,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-splits", type=int, default=0, help="KV-cache workloads: split count (0 = default)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from attention_forward_14_gb300 import workloads as W
    name = args.workload or W.HEADLINE
    if name in W.VARLEN:
        return bench_varlen(args, W.VARLEN[name])
    if name in W.BWD_VARLEN:
        if args.impl == "reference":
            raise SystemExit("the reference arm times the forward oracle only")
        return bench_bwd_varlen(args, W.BWD_VARLEN[name])
    if name in W.KVCACHE:
        return bench_kvcache(args, W.KVCACHE[name])
    if name in W.BWD:
        if args.impl == "reference":
            raise SystemExit("the reference arm times the forward oracle only")
        return bench_bwd(args, W.BWD[name])
    w = W.WORKLOADS[name]

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            bench_reference(args, w)
        return

    import torch
    import attention_forward_14_gb300 as af

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    q, k, v = W.inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    in_bytes = 3 * q.numel() * q.element_size() if w.sq == w.sk else (q.numel() + 2 * k.numel()) * q.element_size()

    if w.splitkv:
        from attention_forward_14_gb300 import binding
        splits = binding.splitkv_default_splits(w.b, w.h, w.sq, w.sk, w.d, w.causal)
        ws = torch.empty(max(16, binding.splitkv_workspace_bytes(w.b, w.h, w.sq, w.d, splits)),
                         dtype=torch.uint8, device=dev)

        def step():
            af.attn_fwd_splitkv(qd, kd, vd, causal=w.causal, scale=w.scale, num_splits=splits, o=o, lse=lse,
                                workspace=ws, stream=stream)
    elif w.dtype == "e4m3":
        splits = 1
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)

        def step():
            af.attn_fwd_fp8(qd, kd, vd, causal=w.causal, scale=w.scale, o=o, lse=lse, stream=stream)
    else:
        splits = 1

        def step():
            af.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, o=o, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    # Inputs that fit in L2 would be read from it on every step: then a
    # 256 MB write evicts them before each timed step, and the step's time is
    # its own event pair's (the flush is outside the pairs).
    out_bytes = o.numel() * o.element_size() + lse.numel() * 4
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes + out_bytes < L2_BYTES else None
    t_all0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    sampler.stop()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(launch_ms) if flush is not None else t_all0.elapsed_time(t_all1), dist, dev)
    ms = total_ms / args.steps
    value = world * w.flops() / (ms * 1e-3) / 1e12

    # end to end through the host-buffer entry point: H2D of Q, K, V from
    # pinned memory, the forward, D2H of O and LSE, every step.
    if w.dtype == "e4m3":  # the host-buffer entry point takes 16-bit inputs; time the same calls with copies
        l2_note = (f"inputs {in_bytes / 1e6:.0f} MB > L2 {L2_BYTES / 1e6:.0f} MB, no flush" if flush is None else
                   f"inputs {in_bytes / 1e6:.0f} MB fit in L2: 256 MB flush before each timed step, "
                   "time from each step's own events")
        return _finish_fp8(args, w, world, rank, dist, dev, q, k, v, qd, kd, vd, o, lse, stream, t_all0, t_all1,
                           total_ms, launch_ms, sampler, step, l2_note)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    for _ in range(2):
        af.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, o, lse, causal=w.causal, scale=w.scale, stream=stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        af.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, o, lse, causal=w.causal, scale=w.scale, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dist, dev)
    e2e_value = world * w.flops() / (e2e_ms * 1e-3) / 1e12
    # this machine's host link, for reading the end-to-end figure: one pinned
    # copy of the step's inputs to the device, alone
    e0.record(stream)
    for dst, src in ((qd, qh), (kd, kh), (vd, vh)):
        dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = in_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9

    if rank == 0:
        peaks = load_peaks()
        kern_ms = statistics.mean(launch_ms)
        achieved = w.flops() / (kern_ms * 1e-3) / 1e12
        # arithmetic intensity under the ridge of the measured peaks: memory is the roof
        below_ridge = w.flops() / w.bytes() < peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp16", "data": "synthetic",
            "config": {"workload": w.name, "b": w.b, "h": w.h, "sq": w.sq, "sk": w.sk, "d": w.d,
                       "causal": w.causal, "qk_std": w.qk_std, "flops_per_step": w.flops(),
                       "l2": f"inputs {in_bytes / 1e6:.0f} MB > L2 {L2_BYTES / 1e6:.0f} MB, no flush"
                       if flush is None else
                       f"inputs {in_bytes / 1e6:.0f} MB fit in L2: 256 MB flush before each timed step, "
                       "time from each step's own events"},
            "pct_of_peak": 100.0 * value / world / peaks["bf16"],
            "pct_of_sustained_peak": 100.0 * value / world / peaks["bf16_sustained"],
            # algorithmic bytes / launch time: the figure that matters below the ridge (small problems)
            "algorithmic_gbs": w.bytes() / (kern_ms * 1e-3) / 1e9,
            "pct_of_hbm": 100.0 * w.bytes() / (kern_ms * 1e-3) / 1e9 / peaks["hbm"],
            "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                          "frac": achieved / peaks["bf16"], "traffic": profiled_traffic(w.name),
                          "peak_kind": f"{peaks['source']} bf16 dense burst (cuBLAS)",
                          "kernel": "attn_fwd_kernel", "algorithmic_bytes": w.bytes()}
                         if not w.splitkv and not below_ridge else
                         {"bound": "hbm", "achieved": w.bytes() / (kern_ms * 1e-3) / 1e9, "peak": peaks["hbm"],
                          "unit": "GB/s", "frac": w.bytes() / (kern_ms * 1e-3) / 1e9 / peaks["hbm"],
                          "traffic": profiled_traffic(w.name), "peak_kind": f"{peaks['source']} HBM copy",
                          "kernel": "attn_fwd_kernel + attn_splitkv_combine_kernel (one step)" if w.splitkv
                          else "attn_fwd_kernel (below the ridge point: the HBM roof applies)",
                          "algorithmic_bytes": w.bytes(), "num_splits": splits}),
            "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": in_bytes,
                    "d2h_bytes_per_step": q.numel() * q.element_size() + lse.numel() * 4,
                    "ms_per_step": e2e_ms, "host_to_device_gbs": h2d_gbs,
                    "h2d_floor_ms": in_bytes / (h2d_gbs * 1e9) * 1e3},
            "gpu_launches": args.steps * (2 if splits > 1 else 1),
            "clocks": sampler.summary(),
        }
        if not args.no_cpu_baseline and world == 1:
            tf, desc, cores, dt, (rows, o_ref, lse_ref) = cpu_baseline(w, q, k, v, want_rows=True)
            line["cpu_baseline"] = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                                    "sample": desc, "seconds": dt,
                                    "extrapolated_full_seconds": w.flops() / (tf * 1e12)}
            # the same rows of the kernel's last output, against the oracle's
            import numpy as np
            idx = torch.as_tensor(rows, dtype=torch.long, device=dev)
            o_k = o[0, 0].index_select(0, idx).double().cpu().numpy()
            l_k = lse[0, 0].index_select(0, idx).double().cpu().numpy()
            fin = np.isfinite(lse_ref)
            line["accuracy"] = {
                "rows": int(len(rows)), "head": "(0, 0)", "against": "fp64 oracle (the cpu_baseline sample)",
                "o_max_abs": float(np.abs(o_k - o_ref).max()),
                "o_rel_l2": float(np.linalg.norm(o_k - o_ref) / max(np.linalg.norm(o_ref), 1e-300)),
                "lse_max_abs": float(np.abs(l_k[fin] - lse_ref[fin]).max()) if fin.any() else 0.0,
                "finite": bool(np.isfinite(o_k).all() and np.isfinite(l_k[fin]).all()),
            }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
