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
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="fa", choices=["fa", "reference"])
    p.add_argument("--workload", default="c4", choices=sorted(workloads.WORKLOADS) + ["dec"],
                   help="dec: decode-shaped forward (informational; its own metric, HBM GB/s)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
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

    inp = workloads.make_inputs(w, H=args.heads, seed=w.seed + rank)
    B, H, N, d = w.B, (w.H if args.heads is None else args.heads), w.N, w.d
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    bm = None if inp["block_mask"] is None else inp["block_mask"].to(dev)
    sl = None if inp["seqlens_k"] is None else inp["seqlens_k"].to(dev)
    kw = dict(causal=w.causal, block_mask=bm, seqlens_k=sl, scale=w.scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 4  # fwd kernel; bwd pre, main, post

    def step():
        fa.fwd(q, k, v, out=o, lse=lse, status=status, **kw)
        fa.bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, status=status, **kw)

    def barrier():
        if pg is not None:
            pg.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))

    # ---- timed region (device-resident inputs; inputs 4 x 64 MiB > L2, so no flush between steps)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if args.flush_l2 else None
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    clocks.mark("t_start")
    start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()  # evicts the previous step's data from the 129 MB L2
        ev[i][0].record(stream)
        fa.fwd(q, k, v, out=o, lse=lse, status=status, **kw)
        ev[i][1].record(stream)
        fa.bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, status=status, **kw)
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t_end")
    clk = clocks.stop()
    barrier()
    ms = start.elapsed_time(end) / args.steps
    if flush is not None:  # the flushes lie between the steps' events
        ms = statistics.mean(e[0].elapsed_time(e[2]) for e in ev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    step_pct = percentiles([e[0].elapsed_time(e[2]) for e in ev])  # this rank's steps
    ms = max_over_ranks(ms, pg, dev)
    assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))

    flops = rl.attention_flops(B, H, N, d, causal=w.causal,
                               block_mask=None if inp["block_mask"] is None else inp["block_mask"].numpy())
    value = flops["total"] * world / (ms * 1e-3) / 1e12

    # ---- end to end through the public API with pinned host buffers
    def run_e2e():
        hq, hk, hv, hdo = (inp[n].pin_memory() for n in ("q", "k", "v", "do"))
        ho, hdq = (torch.empty_like(hq).pin_memory() for _ in range(2))
        hdk, hdv = (torch.empty_like(hk).pin_memory() for _ in range(2))
        hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            do.copy_(hdo, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            hdq.copy_(dq, non_blocking=True)
            hdk.copy_(dk, non_blocking=True)
            hdv.copy_(dv, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = s2.elapsed_time(e2) / args.steps
        e2e_ms = max_over_ranks(e2e_ms, pg, dev)
        return {"value": flops["total"] * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    e2e = None if args.no_e2e else run_e2e()

    in_mib = sum(t.numel() * t.element_size() for t in (q, k, v, do)) / 2**20
    l2_note = (f"inputs {in_mib:.0f} MiB > 129 MB L2; no flush" if in_mib * 2**20 > 129e6 else
               f"inputs {in_mib:.0f} MiB fit in the 129 MB L2: L2-warm, not a contract number")
    if flush is not None:
        l2_note = f"inputs {in_mib:.0f} MiB; L2 flushed (256 MiB written) before each step, outside its events"
    peaks = load_peaks()
    # Dominant launch group: the backward call (pre + main + post in one event span).
    bwd_tflops = flops["bwd"] / (bwd_ms * 1e-3) / 1e12
    fwd_tflops = flops["fwd"] / (fwd_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"]
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": {"workload": workload_label(w, B, H, N, d) + " fwd+bwd",
                   "parallelism": f"replicas x{world}", "l2": l2_note},
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "kernels": {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops},
        "step_ms_p10_p50_p90": step_pct,
        "roofline": {"bound": "tensor", "kernel": "bwd_tc_kernel (timed as the fa_bwd span: pre + main + post)",
                     "achieved": bwd_tflops, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tflops / peak,
                     "traffic": kernel_traffic(f"bwd_tc_kernel<{d}>", w.name, args.heads),
                     "traffic_unit": "DRAM bytes per launch (ncu, profiles/traffic.json)",
                     "peak_source": f"{peaks['source']} bf16 sustained (kernel timed inside a long step)"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    up = useful_padding(w, None if inp["seqlens_k"] is None else inp["seqlens_k"].numpy(), H, N, d, ms, world)
    if up is not None:
        result["useful_padding"] = up
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
