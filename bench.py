#!/usr/bin/env python
"""GLA forward + backward throughput on GB300 (one JSON line on stdout).

Workload: GLA, B=4 H=16 T=2048 K=V=128, bf16 q/k/v/do, fp32 gates, chunk 64,
no initial or final state (seeded synthetic inputs, see
chunked_gated_linear_chunk_gb300/inputs.py).  One step = gla_fwd + gla_bwd
over that batch.  Inputs are resident in HBM; L2 is flushed (a write of
twice the L2 size, then a read of it, so no dirty line of the flush is left
for the timed kernels to write back) before every timed step, outside the
timed interval.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl glacore|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(weak scaling, no collective on the data path); the step time is the max
over ranks and `value` counts the tokens of all ranks.

`--impl reference` times the fp64 CPU oracle on the host cores instead
(rank 0 only): each step is a bounded sample of the workload (one batch row,
all heads), reported in the same unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GLA fwd+bwd tokens/s & TFLOP/s (B4 H16 T2048 d128 bf16), % roofline, 1 GB300"
UNIT = "tokens/s"
WORKLOAD_INDEX = 2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def shape_of(w, n_docs=None, sms=None):
    from chunked_gated_linear_chunk_gb300 import roofline as rf

    nd = n_docs if n_docs is not None else w.B
    # the piece split applies to uniform rows (one document per row)
    plen = rf.piece_len(w.B, w.T, nd, w.H, sms, w.chunk) if sms and nd == w.B else 0
    return rf.Shape(B=w.B, T=w.T, H=w.H, Hqk=w.Hqk, K=w.K, V=w.V, elem=2 if w.dtype == "bf16" else 4,
                    gate="channel" if w.kind == "gla" else "head", n_docs=nd,
                    initial_state=w.initial_state, final_state=w.final_state, dht=w.final_state, chunk=w.chunk,
                    plen=plen)


def job_throughput(ms_local, tokens_per_rank_step, world, device=None):
    """Whole-job throughput: the slowest rank's step time (max over the
    ranks of the current process group) and the tokens of all ranks."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_rank_step / (ms / 1e3)


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.device_index = device_index

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            sel = []
            try:
                import torch

                uuid = torch.cuda.get_device_properties(self.device_index).uuid
                sel = ["-i", "GPU-" + str(uuid)]
            except Exception:
                sel = []
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50", *sel],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self, t_start=None):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        # samples after the first 0.3 s warm-up of the sampler cover the timed loop
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ----------------------------------------------------------- CPU oracle ----
def oracle_sample(d, rows, threads=None, heads=None, tokens=None):
    """Times the oracle fwd+bwd on batch rows `rows`, value heads `heads`
    (default all) and the first `tokens` tokens of each row (default all),
    every document of them; returns (seconds, token count scaled to all
    heads, threads the oracle used, description).  Heads are independent
    recurrences except where q / k are shared (SSD: one group), so a head
    subset of a grouped problem keeps whole groups."""
    import oracle

    H = d["v"].shape[2]
    Hqk = d["q"].shape[2]
    heads = list(range(H)) if heads is None else list(heads)
    grp = H // Hqk
    if grp > 1:  # whole q / k groups
        ng = max(1, len(heads) // grp)
        heads = list(range(ng * grp))
    hq = sorted({h // grp for h in heads})
    T = d["q"].shape[1] if tokens is None else min(tokens, d["q"].shape[1])
    r = slice(rows[0], rows[-1] + 1)
    hs = slice(heads[0], heads[-1] + 1)
    qs = slice(hq[0], hq[-1] + 1)
    seg = None
    n_docs = len(rows)
    if d["segment_ids"] is not None:
        seg = d["segment_ids"][r, :T]
        n_docs = oracle.count_docs(seg, seg.shape[0], T)
    st = lambda t: None if t is None else t[:n_docs, hs]  # the sample's documents come first
    if d["segment_ids"] is None:
        st = lambda t: None if t is None else t[r, hs]
    q, k = d["q"][r, :T, qs], d["k"][r, :T, qs]
    v, do = d["v"][r, :T, hs], d["do"][r, :T, hs]
    g = d["g"][r, :T, hs]
    used = max(1, min(threads or os.cpu_count() or 1, n_docs * len(hq)))
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, g, d["scale"], seg, st(d["h0"]), threads=threads)
    oracle.bwd(q, k, v, g, do, d["scale"], seg, st(d["h0"]), st(d["dht"]), threads=threads)
    secs = time.perf_counter() - t0
    ntok = q.shape[0] * q.shape[1]
    what = f"{q.shape[0]} x {q.shape[1]} tokens, heads {heads[0]}..{heads[-1]} of {H}"
    return secs, ntok * len(heads) / H, used, what


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from chunked_gated_linear_chunk_gb300 import inputs

    d = inputs.make(w)
    cores = os.cpu_count() or 1
    threads = min(cores, w.H)
    for _ in range(args.warmup):
        oracle_sample(d, [0], threads)
    samples = [oracle_sample(d, [0], threads) for _ in range(args.steps)]
    times = [smp[0] for smp in samples]
    threads = samples[0][2]
    ms = 1e3 * statistics.mean(times)
    tokens = w.T  # one batch row, all heads
    value = tokens / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V, "chunk": w.chunk,
                   "sample": "one batch row (T tokens, all heads) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"fp64 token-by-token oracle fwd+bwd on batch row 0 ({w.T} tokens x {w.H} heads) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- GPU arm ----
def flush_l2(buf, i):
    """Flushes L2 before a timed step: writes `buf` (twice the L2 size), then
    reads it back, so that the dirty lines of the write are written back to
    HBM here rather than during the timed kernels.  A short spin on the GPU
    follows, so that the host has enqueued the step's launches before the
    start event is reached: the events then time the kernels, not the
    Python call that launches the first of them."""
    import torch

    buf.fill_(i & 0xFF)
    buf.view(torch.int32).max()
    torch.cuda._sleep(400_000)  # about 0.2 ms at the GB300's 2 GHz SM clock


def measure_device(w, dev, steps, warmup, world=1, rank_sync=False):
    """Times `steps` fwd+bwd steps of workload w with inputs resident in HBM
    (L2 flushed by a write of twice its size before each step, outside the
    event pair).  Returns the per-step and per-kernel CUDA-event times and the
    roofline figures of the step and of its dominant kernel."""
    import torch

    import chunked_gated_linear_chunk_gb300 as glc
    from chunked_gated_linear_chunk_gb300 import inputs
    from chunked_gated_linear_chunk_gb300 import roofline as rf

    d = inputs.make(w)
    x = inputs.to_device(d, dev)
    scale, n_seqs = d["scale"], d["n_seqs"]
    fwd_fn = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd_fn = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    o = torch.empty_like(x["v"])
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    dg = torch.empty_like(x["g"])
    st_shape = (n_seqs, w.H, w.K, w.V)
    ht = torch.empty(st_shape, dtype=torch.float32, device=dev) if w.final_state else None
    dh0 = torch.empty(st_shape, dtype=torch.float32, device=dev) if x["h0"] is not None else None
    # size the workspaces through the ABI
    p, _ = glc._problem(x["q"], x["k"], x["v"], x["g"], scale, x["segment_ids"], x["h0"], w.chunk, n_seqs,
                        w.kind == "ssd")
    nf, nb = glc.workspace_size(p, w.kind + "_fwd"), glc.workspace_size(p, w.kind + "_bwd")
    fws = torch.empty(max(nf, 256), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def fwd_call():
        fwd_fn(x["q"], x["k"], x["v"], x["g"], scale, x["segment_ids"], x["h0"], w.final_state, w.chunk, n_seqs,
               out=o, final_out=ht, workspace=fws)

    def bwd_call():
        bwd_fn(x["q"], x["k"], x["v"], x["g"], x["do"], scale, x["segment_ids"], x["h0"], x["dht"], w.chunk,
               n_seqs, outs=(dq, dk, dv, dg, dh0), workspace=bws)

    for _ in range(warmup):
        flush_l2(flush, 1)
        fwd_call()
        bwd_call()
    torch.cuda.synchronize()
    glc.get_device_error()

    K = steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    tfs = [glc.LaunchTimer(16) for _ in range(K)]
    tbs = [glc.LaunchTimer(16) for _ in range(K)]
    if rank_sync:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for i in range(K):
            flush_l2(flush, i)
            starts[i].record()
            with tfs[i]:
                fwd_call()
            with tbs[i]:
                bwd_call()
            ends[i].record()
        torch.cuda.synchronize()
    if rank_sync:
        torch.distributed.barrier()
    glc.get_device_error()
    clocks = clk.summary()

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # per-kernel durations from the library's launch events
    per_kernel = {}
    launches = 0
    fwd_ms, bwd_ms = [], []
    for i in range(K):
        prev = starts[i]
        for lab, ev in zip(tfs[i].labels, tfs[i].events):
            per_kernel.setdefault(lab, []).append(prev.elapsed_time(ev))
            prev = ev
        fwd_ms.append(starts[i].elapsed_time(prev))
        fprev = prev
        for lab, ev in zip(tbs[i].labels, tbs[i].events):
            per_kernel.setdefault(lab, []).append(prev.elapsed_time(ev))
            prev = ev
        bwd_ms.append(fprev.elapsed_time(prev))
        launches += len(tfs[i].labels) + len(tbs[i].labels)

    peaks, peak_kind = load_peaks()
    shp = shape_of(w, n_seqs, torch.cuda.get_device_properties(dev).multi_processor_count)
    flops = rf.fwd_flops(shp) + rf.bwd_flops(shp)
    nbytes = rf.fwd_bytes(shp) + rf.bwd_bytes(shp)
    t_roof = rf.roofline_time_s(flops, nbytes, peaks["bf16_tflops"], peaks["hbm_gbs"])
    # a kernel launched several times per step (the fp32 path's state and
    # gradient passes are one launch each) is summed per step
    kern_us = {k: 1e3 * sum(v) / K for k, v in per_kernel.items()}
    dom = max(kern_us, key=kern_us.get)
    dom_bytes = rf.kernel_bytes(shp, dom)
    achieved = dom_bytes / (kern_us[dom] * 1e-6) / 1e9 if dom_bytes else None
    return {
        "d": d, "n_seqs": n_seqs, "nf": nf, "nb": nb, "fwd_fn": fwd_fn, "bwd_fn": bwd_fn,
        "ms_local": statistics.mean(step_ms), "step_ms": step_ms, "fwd_ms": statistics.mean(fwd_ms),
        "bwd_ms": statistics.mean(bwd_ms), "kernels_us": kern_us, "launches": launches, "clocks": clocks,
        "flops": flops, "bytes": nbytes, "t_roof": t_roof, "peaks": peaks, "peak_kind": peak_kind,
        "dom": dom, "dom_bytes": dom_bytes, "achieved": achieved,
    }


def roofline_entry(m, traffic=None):
    peaks = m["peaks"]
    return {"bound": "hbm", "kernel": m["dom"], "achieved": m["achieved"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": (m["achieved"] / peaks["hbm_gbs"]) if m["achieved"] else None, "traffic": traffic,
            "algorithmic_bytes_per_launch": m["dom_bytes"], "peak_kind": m["peak_kind"]}


def cpu_baseline_of(w, d, sample=(None, None, None)):
    """The oracle (fp64 token by token, as it stands) on the host cores over a
    bounded sample of workload w: `sample` = (batch rows, heads, tokens per
    row), None for all.  Returns the cpu_baseline object."""
    threads = os.cpu_count() or 1
    nrows, nheads, ntok = sample
    rows = list(range(w.B if nrows is None else min(nrows, w.B)))
    heads = list(range(w.H if nheads is None else min(nheads, w.H)))
    secs, tokens, used, what = oracle_sample(d, rows, threads, heads, ntok)
    return {"value": tokens / secs, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"fp64 token-by-token oracle fwd+bwd on {what}, {secs:.1f} s on {used} threads "
                      f"(tokens/s counted over all {w.H} heads)"}


# bounded CPU samples of the workloads: (batch rows, heads, tokens per row) of
# the oracle run, every document of them (a few seconds each on the host cores)
CPU_SAMPLE = {1: (None, None, None), 2: (None, None, None), 3: (1, None, 1024), 4: (None, 8, 8192),
              5: (None, 8, 8192)}


# the operations around the recurrence, at the sizes of the pages' layer:
# the output norm and gate on the bench workload's o (B4 T2048 H16 V128),
# the short convolution at the FLAT blog's benchmark shape (B8 S4096,
# 2048 channels, 4 taps, bias, SiLU)
FUSIONS = {
    "norm_gate_bf16_B4_T2048_H16_V128": dict(kind="norm_gate", shape=(4, 2048, 16, 128)),
    "short_conv_bf16_B8_T4096_D2048_K4_silu": dict(kind="short_conv", shape=(8, 4096, 2048, 4)),
}


def measure_fusion(name, spec, dev, steps, cpu):
    """Times the forward and the backward of one fused operation (L2 flushed
    before each, outside the event pairs) and reports GB/s against the
    measured copy bandwidth; the oracle (numpy fp64, one host thread) runs a
    bounded slice of the same inputs."""
    import torch

    import chunked_gated_linear_chunk_gb300 as glc

    peaks, peak_kind = load_peaks()
    g = torch.Generator("cpu")
    g.manual_seed(77)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    if spec["kind"] == "norm_gate":
        B, T, H, V = spec["shape"]
        o = torch.randn(B, T, H, V, generator=g).to(torch.bfloat16)
        z = (2.0 * torch.randn(B, T, H, V, generator=g)).to(torch.bfloat16)
        dy = torch.randn(B, T, H, V, generator=g).to(torch.bfloat16)
        wt = 1.0 + 0.5 * torch.randn(V, generator=g)
        od, zd, dyd, wd = (t.to(dev) for t in (o, z, dy, wt))
        y = torch.empty_like(od)
        outs = (torch.empty_like(od), torch.empty_like(od), torch.empty(V, device=dev))
        ws = torch.empty(max(256, int(glc.load().norm_gate_bwd_workspace_size(B * T * H, V))), dtype=torch.uint8,
                         device=dev)
        fwd = lambda: glc.norm_gate_fwd(od, zd, wd, 1e-5, out=y)
        bwd = lambda: glc.norm_gate_bwd(od, zd, wd, dyd, 1e-5, outs=outs, workspace=ws)
        n = B * T * H * V
        fbytes, bbytes = 3 * 2 * n, 5 * 2 * n
        units = B * T

        def oracle_slice():
            from oracle import fusions as F

            sl = slice(0, T // 16)
            F.norm_gate_fwd(o[:, sl], z[:, sl], wt, 1e-5)
            F.norm_gate_bwd(o[:, sl], z[:, sl], wt, dy[:, sl], 1e-5)
            return B * (T // 16)
    else:
        B, T, D, Kc = spec["shape"]
        x = torch.randn(B, T, D, generator=g).to(torch.bfloat16)
        dy = torch.randn(B, T, D, generator=g).to(torch.bfloat16)
        wt = 0.5 * torch.randn(Kc, D, generator=g)
        bt = 0.1 * torch.randn(D, generator=g)
        xd, dyd, wd, bd = (t.to(dev) for t in (x, dy, wt, bt))
        y = torch.empty_like(xd)
        outs = (torch.empty_like(xd), torch.empty(Kc, D, device=dev), torch.empty(D, device=dev))
        ws = torch.empty(max(256, int(glc.load().short_conv_bwd_workspace_size(B, T, D, Kc))), dtype=torch.uint8,
                         device=dev)
        fwd = lambda: glc.short_conv_fwd(xd, wd, bd, None, True, out=y)
        bwd = lambda: glc.short_conv_bwd(xd, wd, bd, dyd, None, True, outs=outs, workspace=ws)
        n = B * T * D
        fbytes, bbytes = 2 * 2 * n, 3 * 2 * n
        units = B * T

        def oracle_slice():
            from oracle import fusions as F

            sl = slice(0, T // 64)
            F.short_conv_fwd(x[:1, sl], wt, bt)
            F.short_conv_bwd(x[:1, sl], wt, bt, dy[:1, sl])
            return T // 64

    def timed(fn):
        for _ in range(3):
            flush_l2(flush, 1)
            fn()
        ts = []
        for i in range(steps):
            flush_l2(flush, i)
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b_.record()
            ts.append((a, b_))
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in ts) * 1e3  # us

    fus, bus = timed(fwd), timed(bwd)
    glc.get_device_error()
    hbm = peaks["hbm_gbs"]
    entry = {
        "fwd_us": fus, "bwd_us": bus, "tokens_per_s": units / ((fus + bus) * 1e-6),
        "fwd_roofline": {"bound": "hbm", "achieved": fbytes / (fus * 1e-6) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": fbytes / (fus * 1e-6) / 1e9 / hbm, "algorithmic_bytes_per_launch": fbytes,
                         "peak_kind": peak_kind},
        "bwd_roofline": {"bound": "hbm", "achieved": bbytes / (bus * 1e-6) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": bbytes / (bus * 1e-6) / 1e9 / hbm, "algorithmic_bytes_per_launch": bbytes,
                         "peak_kind": peak_kind},
        "dtype": "bf16",
    }
    if cpu:
        t0 = time.perf_counter()
        tok = oracle_slice()
        secs = time.perf_counter() - t0
        entry["cpu_baseline"] = {"value": tok / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                                 "sample": f"numpy fp64 oracle fwd+bwd on {tok} tokens of the shape, {secs:.2f} s"}
    return entry


def run_glacore(args, w):
    import torch

    import chunked_gated_linear_chunk_gb300 as glc
    from chunked_gated_linear_chunk_gb300 import inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    glc.load()
    m = measure_device(w, dev, args.steps, args.warmup, world, rank_sync=world > 1)
    d, n_seqs = m["d"], m["n_seqs"]
    ms, value = job_throughput(m["ms_local"], w.B * w.T, world, dev)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            tinfo = json.load(open(tpath)).get(m["dom"])
            if tinfo and tinfo.get("source_sha") == kernel_source_sha():
                traffic = tinfo.get("dram_bytes_per_launch")
        except (OSError, ValueError):
            traffic = None

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, d, dev, world, m["fwd_fn"], m["bwd_fn"], d["scale"], n_seqs, m["nf"], m["nb"])

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_of(w, d, CPU_SAMPLE[w.index])
    # every workload of the build on this GPU (rank 0, one GPU): the headline
    # one from the run above, the others timed here with fewer steps
    workloads = None
    if world == 1 and not args.no_workloads:
        workloads = {}
        for wi, wk in sorted(inputs.WORKLOADS.items()):
            mk = m if wk.name == w.name else measure_device(wk, dev, min(args.steps, 20), 3)
            tk = wk.B * wk.T / (mk["ms_local"] * 1e-3)
            entry = {
                "ms_per_step": mk["ms_local"], "tokens_per_s": tk, "tflops": mk["flops"] / (mk["ms_local"] * 1e-3) / 1e12,
                "steps": len(mk["step_ms"]),
                "step_roofline": {"roofline_us": mk["t_roof"] * 1e6, "measured_us": mk["ms_local"] * 1e3,
                                  "frac": mk["t_roof"] / (mk["ms_local"] * 1e-3), "peak": mk["peak_kind"]},
                "fwd_ms": mk["fwd_ms"], "bwd_ms": mk["bwd_ms"], "kernels_us": mk["kernels_us"],
                "roofline": roofline_entry(mk), "dtype": "bf16" if wk.dtype == "bf16" else "f32",
            }
            if not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu if wk.name == w.name else cpu_baseline_of(wk, mk["d"], CPU_SAMPLE[wi])
            workloads[wk.name] = entry
            if mk is not m:
                del mk
                torch.cuda.empty_cache()
    fusions = None
    if world == 1 and not args.no_workloads:
        fusions = {name: measure_fusion(name, spec, dev, min(args.steps, 20), not args.no_cpu_baseline)
                   for name, spec in FUSIONS.items()}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V, "chunk": w.chunk,
                   "l2": "flushed before every timed step (write of 2x L2, then read back; outside the timed events)", "parallelism": f"replicas x{world}"},
        "tflops": m["flops"] / (ms * 1e-3) / 1e12,
        "step_roofline": {"roofline_us": m["t_roof"] * 1e6, "measured_us": ms * 1e3, "frac": m["t_roof"] / (ms * 1e-3),
                          "peak": m["peak_kind"]},
        "fwd_ms": m["fwd_ms"], "bwd_ms": m["bwd_ms"],
        "kernels_us": m["kernels_us"],
        "roofline": roofline_entry(m, traffic),
        "gpu_launches": m["launches"],
        "clocks": m["clocks"],
        "e2e": e2e,
        "cpu_baseline": cpu,
        "workloads": workloads,
        "fusions": fusions,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_fusions_only(args):
    import torch

    import chunked_gated_linear_chunk_gb300 as glc

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    glc.load()
    out = {name: measure_fusion(name, spec, dev, args.steps, not args.no_cpu_baseline)
           for name, spec in FUSIONS.items()}
    print(json.dumps({"fusions": out}), flush=True)
    return 0


def run_e2e(args, w, d, dev, world, fwd_fn, bwd_fn, scale, n_seqs, nf, nb):
    """End to end through the public API from pinned host buffers: every step
    copies its inputs host -> device, runs the forward and backward, and
    copies all its outputs back.  The steps are pipelined the way a streaming
    consumer would run them: two device buffer sets, copies in on one stream,
    compute on the current stream, copies out on a third, so step i's copies
    overlap steps i - 1 and i + 1's compute.  Time = first copy in to last
    copy out, over K steps (pipeline fill and drain included)."""
    import torch

    names_in = [n for n in ("q", "k", "v", "g", "do", "segment_ids", "h0", "dht") if d.get(n) is not None]
    host_in = {n: d[n].pin_memory() for n in names_in}
    st_shape = (n_seqs, w.H, w.K, w.V)

    def make_set():
        xi = {n: torch.empty(host_in[n].shape, dtype=host_in[n].dtype, device=dev) for n in names_in}
        for n in ("segment_ids", "h0", "dht"):
            xi.setdefault(n, None)
        o = torch.empty_like(xi["v"])
        dq, dk, dv = torch.empty_like(xi["q"]), torch.empty_like(xi["k"]), torch.empty_like(xi["v"])
        dg = torch.empty_like(xi["g"])
        ht = torch.empty(st_shape, dtype=torch.float32, device=dev) if w.final_state else None
        dh0 = torch.empty(st_shape, dtype=torch.float32, device=dev) if xi["h0"] is not None else None
        return xi, (o, ht, dq, dk, dv, dg, dh0)

    sets = [make_set() for _ in range(2)]
    outs0 = [t for t in sets[0][1] if t is not None]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs0]
    fws = torch.empty(max(nf, 256), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    s_c = torch.cuda.current_stream(dev)
    # each direction's copies may be split over NCP streams (more streams measured no faster)
    NCP = 1
    s_in = [torch.cuda.Stream(dev) for _ in range(NCP)]
    s_out = [torch.cuda.Stream(dev) for _ in range(NCP)]

    def split_copy(pairs, streams, wait_ev, rec_ev):
        # pairs: (dst, src) tensors; every tensor is cut into len(streams) contiguous parts
        for k, sk in enumerate(streams):
            with torch.cuda.stream(sk):
                if wait_ev is not None:
                    sk.wait_event(wait_ev)
                for dst, src in pairs:
                    n = dst.numel()
                    a, b = n * k // len(streams), n * (k + 1) // len(streams)
                    if b > a:
                        dst.view(-1)[a:b].copy_(src.view(-1)[a:b], non_blocking=True)
                rec_ev[k].record(sk)

    def compute(xi, outs):
        o, ht, dq, dk, dv, dg, dh0 = outs
        fwd_fn(xi["q"], xi["k"], xi["v"], xi["g"], scale, xi["segment_ids"], xi["h0"], w.final_state, w.chunk,
               n_seqs, out=o, final_out=ht, workspace=fws)
        bwd_fn(xi["q"], xi["k"], xi["v"], xi["g"], xi["do"], scale, xi["segment_ids"], xi["h0"], xi["dht"],
               w.chunk, n_seqs, outs=(dq, dk, dv, dg, dh0), workspace=bws)

    def run(n):
        done = [torch.cuda.Event() for _ in range(n)]
        read = [[torch.cuda.Event() for _ in range(NCP)] for _ in range(n)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        start.record(s_c)
        for sk in s_in:
            sk.wait_event(start)
        for i in range(n):
            xi, outs = sets[i % 2]
            ready = [torch.cuda.Event() for _ in range(NCP)]
            # the compute of step i - 2 has read this input set
            split_copy([(xi[nme], host_in[nme]) for nme in names_in], s_in, done[i - 2] if i >= 2 else None, ready)
            for ev in ready:
                s_c.wait_event(ev)
            if i >= 2:
                for ev in read[i - 2]:
                    s_c.wait_event(ev)  # step i - 2's outputs have been copied out
            compute(xi, outs)
            done[i].record(s_c)
            split_copy(list(zip(host_out, [t for t in outs if t is not None])), s_out, done[i], read[i])
        for ev in read[n - 1]:
            s_c.wait_event(ev)
        end.record(s_c)
        torch.cuda.synchronize(dev)
        return start.elapsed_time(end)

    run(3)
    K = max(3, min(args.steps, 50))
    total_ms = run(K)
    ms, value = job_throughput(total_ms / K, w.B * w.T, world, dev)
    h2d = sum(host_in[n].numel() * host_in[n].element_size() for n in names_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": K, "pipelined": "copies in / compute / copies out on three streams, "
                                                        "two device buffer sets"}


def kernel_source_sha():
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_gated_linear_chunk_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# ncu kernel names -> the library's launch labels (template argument: mode)
NCU_LABELS = (("gla_fwd_kernel", "gla_fwd_kernel"), ("piece_state_kernel", "piece_state_kernel"),
              ("gla_bwd_rev_kernel", "gla_bwd_rev_kernel"), ("gla_bwd_dq_kernel", "gla_bwd_dq_kernel"),
              ("ssd_fwd_kernel", "ssd_fwd_kernel"), ("ssd_bwd_a_kernel", "ssd_bwd_a_kernel"),
              ("ssd_bwd_b_kernel", "ssd_bwd_b_kernel"))


def ingest_traffic(csv_path):
    """Writes profiles/traffic.json (DRAM bytes per launch, per kernel label)
    from an ncu --csv capture with dram__bytes_read.sum / dram__bytes_write.sum,
    stamped with the hash of the kernel sources it was taken on."""
    import csv

    rows = list(csv.reader(l for l in open(csv_path) if l.startswith('"')))
    hdr, data = rows[0], rows[1:]
    ix = {k: hdr.index(k) for k in ("Kernel Name", "Metric Name", "Metric Value", "ID", "Metric Unit")}
    scale_of = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1024.0, "MB": 1024.0 ** 2,
                "GB": 1024.0 ** 3}
    per = {}
    for r in data:
        name = r[ix["Kernel Name"]].replace("(bool)", "").replace("(int)", "").replace(" ", "")
        lab = next((l for key, l in NCU_LABELS if key in name), None)
        if lab is None or r[ix["Metric Name"]] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        val = float(r[ix["Metric Value"]].replace(",", "")) * scale_of.get(r[ix["Metric Unit"]], 1.0)
        per.setdefault(lab, {}).setdefault(r[ix["ID"]], 0.0)
        per[lab][r[ix["ID"]]] += val
    out = {}
    for lab, launches in per.items():
        vals = list(launches.values())
        out[lab] = {"dram_bytes_per_launch": statistics.mean(vals), "launches": len(vals),
                    "source_sha": kernel_source_sha()}
    path = os.path.join(ROOT, "profiles", "traffic.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
    print(json.dumps(out))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="glacore", choices=["glacore", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload entries (all five workloads, timed after the headline one)")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX, choices=[1, 2, 3, 4, 5],
                    help="synthetic workload (default 2: GLA B4 H16 T2048 d128 bf16, the headline)")
    ap.add_argument("--fusions-only", action="store_true",
                    help="time only the two fused operations around the recurrence (one JSON line)")
    ap.add_argument("--ingest-traffic", metavar="NCU_CSV",
                    help="write profiles/traffic.json from an ncu DRAM-bytes capture and exit")
    args = ap.parse_args(argv)
    if args.ingest_traffic:
        return ingest_traffic(args.ingest_traffic)
    if args.warmup < 3:
        args.warmup = 3
    from chunked_gated_linear_chunk_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    if args.fusions_only:
        return run_fusions_only(args)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_glacore(args, w)


if __name__ == "__main__":
    sys.exit(main())
