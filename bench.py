"""Benchmark: fused attention forward + backward on the long-context causal workload
(B=1, H=32, N=8192, d=128, bf16 inputs, fp32 LSE), one step = fa_fwd + fa_bwd over one batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fa|reference] [--workload c4]

Prints ONE JSON line (rank 0). ``value`` is whole-job attention TFLOP/s (forward 4 B H N^2 d,
backward 2.5x, halved for causal) with inputs resident in HBM; ``e2e`` is the same metric with
pinned-host inputs copied in and results copied out inside the timed region. Multi-GPU runs
(torchrun) are weak-scaled replicas: every rank runs its own batch; there is no collective on the
data path (only the max-over-ranks timing reduction).

``--impl reference`` times the fp64 CPU oracle (the only reference this method has) on a bounded
sample of the same workload: one head per step.
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_io_aware_38_gb300 import roofline as rl  # noqa: E402
from exact_io_aware_38_gb300 import workloads  # noqa: E402

METRIC = "attention TFLOP/s fwd+bwd (bf16, causal N=8192 d=128) and % of BF16 tensor peak"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="fa", choices=["fa", "reference"])
    p.add_argument("--workload", default="c4", choices=sorted(workloads.WORKLOADS) + ["dec"],
                   help="dec: decode-shaped forward (informational; its own metric, HBM GB/s)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    p.add_argument("--no-secondary", action="store_true", help="skip the other workloads' figures (profiling runs)")
    p.add_argument("--heads", type=int, default=None, help="override H (smaller profiling cases only)")
    p.add_argument("--flush-l2", action="store_true",
                   help="write 256 MiB before each timed step (outside its events); step time from the events")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"bf16_tflops": d.get("bf16_tflops"), "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t_start", 0.0), getattr(self, "t_end", float("inf"))
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if not (t0 - 0.02 <= ts <= t1 + 0.02):
                    continue  # outside the timed region
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples_in_timed_region": len(sm),
                "reasons": sorted(reasons)}


def sources_sha256(paths):
    """sha256 prefix over the named source files (relative to the repo root), in order."""
    h = hashlib.sha256()
    for p in paths:
        h.update(p.encode())
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(name, workload_name, heads_override):
    """DRAM bytes per launch of `name` from the committed ncu record, or None when the record is
    for another workload or any source the kernel is built from has changed since the counters
    were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[name]
        digest = sources_sha256(rec["sources"])
    except (OSError, KeyError, ValueError, TypeError):
        return None
    if heads_override is not None or not rec["workload"].startswith(workload_name + ":"):
        return None
    if digest != rec["sources_sha256_prefix"]:
        return None
    return rec["dram_bytes_per_launch"]


def max_over_ranks(value, pg, device):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if pg is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_step(inp, head):
    """The fp64 oracle on one (b, h) head of the workload: forward and full backward."""
    import oracle

    b, h = head
    hk = h // (inp["q"].shape[1] // inp["k"].shape[1])  # K/V head read by query head h
    q, do = (inp[n][b, h].double().numpy() for n in ("q", "do"))
    k, v = (inp[n][b, hk].double().numpy() for n in ("k", "v"))
    bm = None if inp["block_mask"] is None else inp["block_mask"].numpy()
    L = None if inp["seqlens_k"] is None else int(inp["seqlens_k"][b])
    c, causal = inp["scale"], inp["causal"]
    oracle.head_forward(q, k, v, c, causal, bm, L)
    oracle.head_dq(q, k, v, do, c, causal, bm, L)
    N = q.shape[0]
    stats = oracle.head_row_stats(q, k, v, do, c, causal, bm, L)
    for a in range(0, N, 2048):
        oracle.head_dkdv(q, k, v, do, c, causal, bm, L, cols=np.arange(a, min(N, a + 2048)), stats=stats)


def percentiles(xs, qs=(10, 50, 90)):
    """Nearest-rank percentiles of the per-step times (ms)."""
    v = sorted(xs)
    return [v[min(len(v) - 1, max(0, -(-q * len(v) // 100) - 1))] for q in qs]


def useful_padding(w, seqlens, H, N, d, ms, world):
    """The secondary figure under key padding: 4 H d N sum_b L_b FLOPs per forward (x3.5 with the
    backward) over the same step time. None without key padding, and with the causal mask, where
    that count is not the work done."""
    if seqlens is None or w.causal:
        return None
    fl = 3.5 * rl.useful_padding_flops(H, N, d, np.asarray(seqlens))
    return {"value": fl * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "count": "4 H d N sum_b L_b per forward, x3.5 with the backward (key padding; secondary)"}


def sample_flops(w, inp):
    f = rl.attention_flops(1, 1, w.N, w.d, causal=w.causal,
                           block_mask=None if inp["block_mask"] is None else inp["block_mask"].numpy())
    return f["total"]


def workload_label(w, B, H, N, d):
    kv = "" if w.Hkv is None else f" Hkv{H // (w.H // w.kv_heads)}"
    return f"{w.name}: B{B} H{H}{kv} N{N} d{d}{' causal' if w.causal else ''}"


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    inp = workloads.make_inputs(w, H=w.H // w.kv_heads)  # one K/V head and its query heads
    fl = sample_flops(w, inp)
    for _ in range(args.warmup):
        cpu_oracle_step(inp, (0, 0))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_step(inp, (0, 0))
    dt = (time.perf_counter() - t0) / args.steps
    val = fl / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": {"workload": workload_label(w, w.B, w.H, w.N, w.d),
                   "sample": f"one head of {w.B * w.H} per step (forward + full backward)"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "one (b, h) head of the workload per step, fp64 numpy oracle"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# Decode shape: one new query row per sequence against an 8192-key cache, 8 K/V heads shared by 32
# query heads (the long-context shape of the benchmark, generating one token per sequence).
DEC = dict(B=8, H=32, Hkv=8, Nq=1, Nk=8192, d=128)


def run_decode(args):
    """Forward split over keys on the decode shape, timed with CUDA events on the launching
    stream; the metric is K/V bytes read per second (the path is HBM-bound: 256 MiB of cache per
    step, 4 KiB of queries). The unsplit forward is timed beside it."""
    import exact_io_aware_38_gb300 as fa
    from exact_io_aware_38_gb300 import build

    build.build()
    fa.lib()
    dev = torch.device("cuda", 0)
    c = DEC
    g = torch.Generator("cpu").manual_seed(2024)
    draw = lambda *shape: torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
    q = draw(c["B"], c["Nq"], c["H"], c["d"])
    k = draw(c["B"], c["Nk"], c["Hkv"], c["d"])
    v = draw(c["B"], c["Nk"], c["Hkv"], c["d"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((c["B"], c["H"], c["Nq"]), dtype=torch.float32, device=dev)
    p, _ = fa._problem(q, k, None, None, None, None, True, None)
    splits = fa.fa_fwd_splitkv_splits(p, torch.cuda.get_device_properties(dev).multi_processor_count)
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(p, splits), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    # the library's choice: a split count, or (count 1) the plain forward
    ms = timed(lambda: fa.fwd_splitkv(q, k, v, causal=True, out=o, lse=lse, workspace=ws, status=status))
    ms_unsplit = timed(lambda: fa.fwd_varlen(q, k, v, causal=True, out=o, lse=lse, status=status))
    sweep = {}
    for n in (1, 2, 4, 8, 16):
        wsn = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(p, n), dtype=torch.uint8, device=dev)
        sweep[n] = timed(lambda: fa.fwd_splitkv(q, k, v, num_splits=n, causal=True, out=o, lse=lse, workspace=wsn,
                                                status=status))
    # Batch 1 (32 CTAs without a split, fewer than the SMs): where splitting over keys pays.
    q1, k1, v1, o1 = q[:1].contiguous(), k[:1].contiguous(), v[:1].contiguous(), o[:1].contiguous()
    lse1 = lse[:1].contiguous()
    p1, _ = fa._problem(q1, k1, None, None, None, None, True, None)
    s1 = fa.fa_fwd_splitkv_splits(p1, torch.cuda.get_device_properties(dev).multi_processor_count)
    ws1 = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(p1, s1), dtype=torch.uint8, device=dev)
    ms_b1 = timed(lambda: fa.fwd_splitkv(q1, k1, v1, num_splits=s1, causal=True, out=o1, lse=lse1, workspace=ws1,
                                         status=status))
    ms_b1_unsplit = timed(lambda: fa.fwd_varlen(q1, k1, v1, causal=True, out=o1, lse=lse1, status=status))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    kv_bytes = 2 * c["B"] * c["Nk"] * c["Hkv"] * c["d"] * 2
    kv1 = kv_bytes // c["B"]
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    peaks = load_peaks()
    print(json.dumps({
        "metric": "decode attention forward, K/V bytes read per second (B8 H32 Hkv8 N_q1 N_k8192 d128)",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": "dec: " + " ".join(f"{k_}{v_}" for k_, v_ in c.items()), "num_splits": splits,
                   "l2": "K/V 256 MiB > 129 MB L2; no flush"},
        "unsplit": {"ms_per_step": ms_unsplit, "value": kv_bytes / (ms_unsplit * 1e-3) / 1e9},
        "splits_sweep_gbs": {str(n_): kv_bytes / (t * 1e-3) / 1e9 for n_, t in sweep.items()},
        "batch1": {"num_splits": s1, "split_gbs": kv1 / (ms_b1 * 1e-3) / 1e9,
                   "unsplit_gbs": kv1 / (ms_b1_unsplit * 1e-3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": f"{peaks['source']} HBM copy bandwidth"},
        "gpu_launches": 2 * args.steps,  # split pass + merge per step
    }), flush=True)


def make_device_buffers(w, H, seed, dev):
    """Seeded inputs of workload `w` on `dev` and the output / workspace buffers of one step."""
    import exact_io_aware_38_gb300 as fa

    inp = workloads.make_inputs(w, H=H, seed=seed)
    B, Hq, N, d = inp["q"].shape
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "do")}
    t["bm"] = None if inp["block_mask"] is None else inp["block_mask"].to(dev)
    t["sl"] = None if inp["seqlens_k"] is None else inp["seqlens_k"].to(dev)
    t["o"] = torch.empty_like(t["q"])
    t["lse"] = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    t["dq"], t["dk"], t["dv"] = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["k"])
    t["ws"] = torch.empty(fa.fa_bwd_workspace_bytes(B, Hq, N, d), dtype=torch.uint8, device=dev)
    t["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
    return inp, t


def time_device_steps(w, t, steps, warmup, flush_l2, stream, clocks=None, barrier=lambda: None, breakdown=True):
    """Per-step device times (ms) of fwd, the whole bwd call and its main pass, and the step, from
    CUDA events on the launching stream; the span over all steps. With flush_l2, 256 MiB are
    written before each step, outside its events. Without breakdown only the span is taken, with
    no event recorded between the launches it times."""
    import exact_io_aware_38_gb300 as fa

    kw = dict(causal=w.causal, block_mask=t["bm"], seqlens_k=t["sl"], scale=w.scale, status=t["status"])
    E = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(E(), E(), E(), E(), E()) for _ in range(steps)]
    warm_ev = (E(), E())

    def step(e):
        fa.fwd(t["q"], t["k"], t["v"], out=t["o"], lse=t["lse"], **kw)
        if e is not None:
            e[1].record(stream)
        fa.bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["do"], dq=t["dq"], dk=t["dk"], dv=t["dv"],
               workspace=t["ws"], main_events=(e[2], e[3]) if e is not None else warm_ev, **kw)

    for _ in range(max(3, warmup)):
        step(None)
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0, fa.fa_status_string(int(t["status"].item()))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=stream.device) if flush_l2 else None
    start, end = E(), E()
    barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
        clocks.mark("t_start")
    start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()  # evicts the previous step's data from the 129 MB L2
        if breakdown or flush is not None:
            ev[i][0].record(stream)
            step(ev[i])
            ev[i][4].record(stream)
        else:
            step(None)
    end.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark("t_end")
    barrier()
    assert int(t["status"].item()) == 0, fa.fa_status_string(int(t["status"].item()))
    if not (breakdown or flush is not None):
        return {"span_ms": start.elapsed_time(end) / steps}
    return {
        "span_ms": start.elapsed_time(end) / steps,
        "step": [e[0].elapsed_time(e[4]) for e in ev],
        "fwd": [e[0].elapsed_time(e[1]) for e in ev],
        "bwd": [e[1].elapsed_time(e[4]) for e in ev],
        "main": [e[2].elapsed_time(e[3]) for e in ev],
    }


def run_e2e(w, inp, t, steps, flops_total, dev, pg, world, barrier):
    """The same step end to end through the public API from pinned host buffers: every step copies
    its Q, K, V, dO in and its O, LSE, dQ, dK, dV out. Copies run on their own streams: dO's upload
    overlaps the forward, O/LSE's download the backward, and (two sets of device and host buffers)
    one step's downloads overlap the next step's uploads and forward."""
    import exact_io_aware_38_gb300 as fa

    B, H, N, d = inp["q"].shape
    host_in = {n: inp[n].pin_memory() for n in ("q", "k", "v", "do")}
    sets = []
    for _ in range(2):
        dv = {n: torch.empty_like(t[n]) for n in ("q", "k", "v", "do", "o", "lse", "dq", "dk", "dv", "ws")}
        hv = {n: torch.empty(t[n].shape, dtype=t[n].dtype).pin_memory() for n in ("o", "lse", "dq", "dk", "dv")}
        sets.append((dv, hv))
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in sets[0][1].values())
    s_c = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    E = lambda: torch.cuda.Event()
    ev = [{k: E() for k in ("qkv", "do", "fwd", "bwd", "out")} for _ in range(2)]
    kw = dict(causal=w.causal, block_mask=t["bm"], seqlens_k=t["sl"], scale=w.scale, status=t["status"])

    def e2e_step(i):
        D, Hh = sets[i % 2]
        e = ev[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(e["bwd"])  # step i - 2 has finished reading this set's inputs
            for n in ("q", "k", "v"):
                D[n].copy_(host_in[n], non_blocking=True)
            e["qkv"].record(s_in)
            D["do"].copy_(host_in["do"], non_blocking=True)
            e["do"].record(s_in)
        s_c.wait_event(e["qkv"])
        if i >= 2:
            s_c.wait_event(e["out"])  # step i - 2's results have left this set's output buffers
        fa.fwd(D["q"], D["k"], D["v"], out=D["o"], lse=D["lse"], stream=s_c, **kw)
        e["fwd"].record(s_c)
        s_c.wait_event(e["do"])
        fa.bwd(D["q"], D["k"], D["v"], D["o"], D["lse"], D["do"], dq=D["dq"], dk=D["dk"], dv=D["dv"],
               workspace=D["ws"], stream=s_c, **kw)
        e["bwd"].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e["fwd"])
            Hh["o"].copy_(D["o"], non_blocking=True)
            Hh["lse"].copy_(D["lse"], non_blocking=True)
            s_out.wait_event(e["bwd"])
            for n in ("dq", "dk", "dv"):
                Hh[n].copy_(D[n], non_blocking=True)
            e["out"].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        e2e_step(3 + i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_c)
    t1.record(s_out)
    torch.cuda.synchronize()
    assert int(t["status"].item()) == 0, fa.fa_status_string(int(t["status"].item()))
    ms = t0.elapsed_time(t1) / steps
    ms = max_over_ranks(ms, pg, dev)
    # the last step's results against the device-resident run (same inputs, same kernels)
    D, Hh = sets[(3 + steps - 1) % 2]
    assert torch.equal(Hh["o"], t["o"].cpu()) and torch.equal(Hh["dk"], t["dk"].cpu())
    return {"value": flops_total * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "copies": "pinned host <-> device on two copy streams, double-buffered, overlapping the kernels"}


def secondary_figures(names, steps, warmup, dev, peak):
    """Device step figures of the other workloads (each its own seeded inputs), with the fraction of
    the same peak; for the L2-resident ones also the figure with L2 flushed before each step."""
    out = {}
    stream = torch.cuda.current_stream(dev)
    for name in names:
        w = workloads.WORKLOADS[name]
        inp, t = make_device_buffers(w, None, w.seed, dev)
        B, H, N, d = inp["q"].shape
        fl = rl.attention_flops(B, H, N, d, causal=w.causal,
                                block_mask=None if inp["block_mask"] is None else inp["block_mask"].numpy())
        step_ms = time_device_steps(w, t, steps, warmup, False, stream, breakdown=False)["span_ms"]
        r = time_device_steps(w, t, steps, 0, False, stream)  # per-kernel figures (events between launches)
        rec = {"workload": workload_label(w, B, H, N, d) + " fwd+bwd", "ms_per_step": step_ms,
               "value": fl["total"] / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "fwd_ms": statistics.median(r["fwd"]), "bwd_ms": statistics.median(r["bwd"]),
               "bwd_main_ms": statistics.median(r["main"])}
        rec["frac"] = rec["value"] / peak
        in_bytes = sum(t[n].numel() * t[n].element_size() for n in ("q", "k", "v", "do"))
        if in_bytes <= 129e6:
            rf = time_device_steps(w, t, steps, warmup, True, stream)
            ms_f = statistics.median(rf["step"])
            rec["l2"] = f"inputs {in_bytes / 2**20:.0f} MiB fit in the 129 MB L2: value is L2-warm"
            rec["l2_flushed"] = {"ms_per_step": ms_f, "value": fl["total"] / (ms_f * 1e-3) / 1e12,
                                 "frac": fl["total"] / (ms_f * 1e-3) / 1e12 / peak}
        else:
            rec["l2"] = f"inputs {in_bytes / 2**20:.0f} MiB > 129 MB L2; no flush"
        up = useful_padding(w, None if inp["seqlens_k"] is None else inp["seqlens_k"].numpy(), H, N, d, step_ms, 1)
        if up is not None:
            rec["useful_padding"] = up
        out[name] = rec
        del t
        torch.cuda.empty_cache()
    return out


def fp8_forward_figure(steps, warmup, dev, peak_bf16):
    """The FP8 forward (e4m3 Q, K, V^T with per-head descales) on the long-context causal shape,
    CUDA events on the launching stream; FLOPs as the bf16 forward; the peak is the measured bf16
    burst figure times the nominal FP8 / BF16 ratio of 2."""
    import exact_io_aware_38_gb300 as fa

    w = workloads.WORKLOADS["c4"]
    inp = workloads.make_fp8_inputs(w)
    q8, k8, vt8 = (inp[n].to(dev) for n in ("q8", "k8", "vt8"))
    qs, ks, vs = (inp[n].to(dev) for n in ("q_descale", "k_descale", "v_descale"))
    B, H, N, d = q8.shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    run = lambda: fa.fwd_fp8(q8, k8, vt8, qs, ks, vs, causal=True, out=o, lse=lse, status=status)
    for _ in range(max(3, warmup)):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e in ev:
        e[0].record(stream)
        run()
        e[1].record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    fl = rl.attention_flops(B, H, N, d, causal=True)["fwd"]
    tf = fl / (ms * 1e-3) / 1e12
    peak = 2.0 * peak_bf16
    return {"workload": workload_label(w, B, H, N, d) + " forward, e4m3 inputs", "ms": ms, "value": tf,
            "unit": "TFLOP/s", "peak": peak, "frac": tf / peak,
            "peak_source": "measured bf16 burst x 2 (nominal FP8 / BF16 dense ratio)"}


def varlen_figure(steps, warmup, dev, peak):
    """The packed-sequence path on the key-padding workload's sequences: queries as in c2 (N rows
    per sequence), keys and values packed to each sequence's L_b rows (cu_seqlens, N_q != N_k),
    fwd_varlen + bwd_varlen per step. FLOPs are the useful count 4 H d N sum_b L_b per forward
    (x3.5 with the backward), the count of c2's useful_padding figure."""
    import exact_io_aware_38_gb300 as fa

    w = workloads.WORKLOADS["c2"]
    inp = workloads.make_inputs(w)
    B, H, N, d = inp["q"].shape
    lens = [int(x) for x in inp["seqlens_k"].tolist()]
    rows = lambda x: x.permute(0, 2, 1, 3).reshape(B * N, x.shape[1], d)  # [B*N, heads, d]
    q, do = (rows(inp[n]).contiguous().to(dev) for n in ("q", "do"))
    k, v = (torch.cat([inp[n][b, :, :lens[b]].permute(1, 0, 2) for b in range(B)]).contiguous().to(dev)
            for n in ("k", "v"))
    cu_q = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device=dev)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    kw = dict(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=N, max_seqlen_k=N, causal=False, scale=w.scale)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o, lse = fa.fwd_varlen(q, k, v, **kw, status=status)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p, _ = fa._problem(q, k, cu_q, cu_k, N, N, False, w.scale)
    ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(p), dtype=torch.uint8, device=dev)

    def run():
        fa.fwd_varlen(q, k, v, **kw, out=o, lse=lse, status=status)
        fa.bwd_varlen(q, k, v, o, lse, do, **kw, dq=dq, dk=dk, dv=dv, workspace=ws, status=status)

    for _ in range(max(3, warmup)):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    ms = a.elapsed_time(b) / steps
    tf = 3.5 * rl.useful_padding_flops(H, N, d, np.asarray(lens)) / (ms * 1e-3) / 1e12
    return {"workload": f"c2 sequences packed: B{B} H{H} N_q{N} per sequence, N_k = L_b (sum {sum(lens)}) d{d} "
            "fwd+bwd (fwd_varlen, bwd_varlen)", "ms_per_step": ms, "value": tf, "unit": "TFLOP/s",
            "frac": tf / peak, "count": "4 H d N sum_b L_b per forward, x3.5 with the backward",
            "l2": "inputs fit in the 129 MB L2: value is L2-warm"}


def ring_figure(steps, warmup, dev, peak, world=4):
    """Ring attention's per-rank schedule on the long-context causal shape, the W ranks run one
    after another on one GPU: the compute of a W-way sequence-sharded fwd + bwd step, without its
    K/V rotation. Per rank: the partial forwards of its query block over the key blocks it sees
    (the diagonal one causal), their log-sum-exp merges and the finalize; then the accumulating
    backward shares into fp32 dQ, dK, dV (zeroed each step). The FLOPs are the fused step's (the
    ring visits the same tiles), so the figure compares directly with it."""
    import exact_io_aware_38_gb300 as fa
    from exact_io_aware_38_gb300 import ring

    w = workloads.WORKLOADS["c4"]
    inp = workloads.make_inputs(w)
    t = {n: inp[n].permute(0, 2, 1, 3).contiguous() for n in ("q", "k", "v", "do")}  # [B, N, H, d]
    B, N, H, d = t["q"].shape
    Hkv = t["k"].shape[2]
    blk = N // world
    # each rank's own blocks (a rank holds its query, key, value and gradient blocks)
    blocks = {n: [t[n][:, r * blk:(r + 1) * blk].contiguous().to(dev) for r in range(world)] for n in t}
    dq = torch.zeros((B, N, H, d), dtype=torch.float32, device=dev)
    dk = torch.zeros((B, N, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.zeros_like(dk)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sched = [ring.ring_schedule(r, world, True) for r in range(world)]

    def run():
        dq.zero_()
        dk.zero_()
        dv.zero_()
        for r in range(world):
            qb, dob = blocks["q"][r], blocks["do"][r]
            acc = None
            for _, src, c in sched[r]:
                if c is None:
                    continue
                part = fa.fwd_partial(qb, blocks["k"][src], blocks["v"][src], causal=c, scale=w.scale, status=status)
                acc = part if acc is None else fa.merge_partials(qb, blocks["k"][src], acc, part)
            o, lse = fa.finalize_partials(qb, blocks["k"][r], acc)
            for _, src, c in sched[r]:
                if c is None:
                    continue
                fa.bwd_varlen_accumulate(qb, blocks["k"][src], blocks["v"][src], o, lse, dob,
                                         dq[:, r * blk:(r + 1) * blk], dk[:, src * blk:(src + 1) * blk],
                                         dv[:, src * blk:(src + 1) * blk], causal=c, scale=w.scale, status=status)

    for _ in range(max(3, warmup)):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        run()
    b.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
    ms = a.elapsed_time(b) / steps
    tf = rl.attention_flops(B, H, N, d, causal=True)["total"] / (ms * 1e-3) / 1e12
    return {"workload": workload_label(w, B, H, N, d) + f" fwd+bwd as a {world}-rank ring, ranks in sequence",
            "ms_per_step": ms, "value": tf, "unit": "TFLOP/s", "frac": tf / peak,
            "note": "compute only (no K/V rotation); same FLOPs as the fused step"}


def main():
    args = parse()
    if args.workload == "dec":
        return run_decode(args)
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import exact_io_aware_38_gb300 as fa
    from exact_io_aware_38_gb300 import build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    build.build()
    fa.lib()

    def barrier():
        if pg is not None:
            pg.barrier()

    inp, t = make_device_buffers(w, args.heads, w.seed + rank, dev)
    B, H, N, d = inp["q"].shape
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 4  # fwd kernel; bwd pre, main, post

    # ---- timed region (device-resident inputs; 4 x 64 MiB of inputs > L2, so no flush between steps)
    clocks = ClockSampler(local)
    r = time_device_steps(w, t, args.steps, args.warmup, args.flush_l2, stream, clocks, barrier, breakdown=False)
    clk = clocks.stop()
    ms = r["span_ms"] if not args.flush_l2 else statistics.mean(r["step"])  # flushes lie between steps
    ms = max_over_ranks(ms, pg, dev)
    # The per-kernel figures and the step percentiles come from a second pass of the same steps
    # with events around each launch.
    rb = time_device_steps(w, t, args.steps, 0, args.flush_l2, stream, None, barrier, breakdown=True)
    fwd_ms, bwd_ms, main_ms = (statistics.mean(rb[k]) for k in ("fwd", "bwd", "main"))
    step_pct = percentiles(rb["step"])  # this rank's steps (events between launches)

    flops = rl.attention_flops(B, H, N, d, causal=w.causal,
                               block_mask=None if inp["block_mask"] is None else inp["block_mask"].numpy())
    value = flops["total"] * world / (ms * 1e-3) / 1e12

    e2e = None if args.no_e2e else run_e2e(w, inp, t, args.steps, flops["total"], dev, pg, world, barrier)

    in_mib = sum(t[n].numel() * t[n].element_size() for n in ("q", "k", "v", "do")) / 2**20
    l2_note = (f"inputs {in_mib:.0f} MiB > 129 MB L2; no flush" if in_mib * 2**20 > 129e6 else
               f"inputs {in_mib:.0f} MiB fit in the 129 MB L2: L2-warm, not a contract number")
    if args.flush_l2:
        l2_note = f"inputs {in_mib:.0f} MiB; L2 flushed (256 MiB written) before each step, outside its events"
    peaks = load_peaks()
    # The timed region is short (tens of ms at full clock, no power cap), so the burst peak applies.
    peak = peaks["bf16_tflops"]
    # Dominant launch: the backward main kernel, timed alone by events around its launch.
    main_tflops = flops["bwd"] / (main_ms * 1e-3) / 1e12
    fwd_tflops = flops["fwd"] / (fwd_ms * 1e-3) / 1e12
    bwd_tflops = flops["bwd"] / (bwd_ms * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": {"workload": workload_label(w, B, H, N, d) + " fwd+bwd",
                   "parallelism": f"replicas x{world}", "l2": l2_note},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "peak_for_pct": f"{peak} TFLOP/s, {peaks['source']} bf16 burst (short timed region at full clock)",
        "kernels": {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "bwd_main_ms": main_ms, "fwd_tflops": fwd_tflops,
                    "bwd_tflops": bwd_tflops, "bwd_main_tflops": main_tflops,
                    "fwd_frac": fwd_tflops / peak, "bwd_frac": bwd_tflops / peak},
        "step_ms_p10_p50_p90": step_pct,
        "roofline": {"bound": "tensor", "kernel": f"bwd_tc_kernel<{d}> (events around its launch)",
                     "achieved": main_tflops, "peak": peak, "unit": "TFLOP/s", "frac": main_tflops / peak,
                     "traffic": kernel_traffic(f"bwd_tc_kernel<{d}>", w.name, args.heads),
                     "traffic_unit": "DRAM bytes per launch (ncu, profiles/traffic.json)",
                     "peak_source": f"{peaks['source']} bf16 burst (kernel timed in a short region at full clock)"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    up = useful_padding(w, None if inp["seqlens_k"] is None else inp["seqlens_k"].numpy(), H, N, d, ms, world)
    if up is not None:
        result["useful_padding"] = up
    if rank == 0 and not args.no_secondary and args.heads is None and args.workload == "c4":
        result["secondary"] = secondary_figures(["c5", "c3", "c2", "c4g"], min(args.steps, 20), args.warmup, dev, peak)
        result["secondary"]["fp8_fwd"] = fp8_forward_figure(min(args.steps, 20), args.warmup, dev, peak)
        result["secondary"]["ring"] = ring_figure(min(args.steps, 10), args.warmup, dev, peak)
        result["secondary"]["varlen_packed"] = varlen_figure(min(args.steps, 20), args.warmup, dev, peak)
    if rank == 0 and not args.no_cpu_baseline:
        heads = [(0, h) for h in range(min(3, H))]  # about 10 s of the oracle on the host cores
        t0 = time.perf_counter()
        for hd in heads:
            cpu_oracle_step(inp, hd)
        dt = time.perf_counter() - t0
        fl = sample_flops(w, inp) * len(heads)
        result["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                                  "kind": "oracle", "sample": f"{len(heads)} (b, h) heads of {B * H}, forward + full "
                                  f"backward each, fp64 numpy ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
