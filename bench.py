"""Benchmark of the paged GQA attention hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--rows all|none]

Prints ONE JSON line (rank 0).  The headline workload is the batched decode
of the 0.6B Thinker shape: 32 requests, GQA 16/8, head_dim 128, contexts
~ U[200, 2000], 16-token pages scattered over a 4096-page pool.  One step is
one qa_decode_attn call over that batch (one split-K kernel launch that also
merges the splits).
The metric is the decode's algorithmic HBM bandwidth: K+V bytes of every
cached position read plus q and out, 4096 B per position + 8192 B per
request, divided by the device time of the call.

Timing: inputs resident in HBM; four rotating copies of the decode inputs
(about 4 x 144 MB, far above the 129 MB L2) so no step finds its K/V in L2;
steps run back to back inside CUDA graphs (launch overhead amortised) and are
timed with CUDA events on the launching stream; barrier + synchronize on both
sides, max over ranks.  nvidia-smi samples clocks during the timed region.

Other keys: `e2e` (the same metric through the C ABI with host buffers: q,
page table and lengths read from pinned host memory and the output written
there by the kernel, the host reading the result every step; the same step
with copy-engine copies under `e2e.copy_engine`),
`roofline` (the decode call against the measured HBM copy bandwidth),
`cpu_baseline` (the fp64 oracle on this host's cores, whole workload),
`rows` (the other hot-path operations measured the same way: ragged causal
prefill with page write, chunked prefill after cached positions, AuT windowed attention, long-context decode, the
decode step with the QK-norm + RoPE KV append, paged cross-attention decode,
a captured 28-layer decode step, the tiny case, the AuT encoder layer around
the window attention).  With --impl reference the oracle itself is timed as
the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm=float(pk["hbm_gbs"]), bf16=float(pk["bf16_tflops"]),
                    bf16_sustained=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), source="measured")
    except Exception:
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0, source="fallback")


def decode_bytes(lengths, hq=16, hkv=8, d=128):
    """Algorithmic bytes of one decode call: K and V rows of every cached
    position, plus q and out."""
    return int(np.sum(lengths)) * hkv * d * 2 * 2 + len(lengths) * hq * d * 2 * 2


def prefill_flops(lengths, hq=16, d=128):
    return int(sum(4 * hq * d * (int(L) * (int(L) + 1) // 2) for L in lengths))


def prefill_bytes(total, hq=16, hkv=8, d=128):
    # q + out (2 * hq rows), k + v read (2 * hkv rows), k + v page write (2 * hkv)
    return total * d * 2 * (2 * hq + 4 * hkv)


def window_flops(cu, h=14, d=64):
    n = np.diff(np.asarray(cu, np.int64))
    return int(4 * h * d * np.sum(n * n))


def window_bytes(total, h=14, d=64):
    return total * h * d * 2 * 4  # q, k, v, out


def source_digest(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_gqa_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name, digest):
    """DRAM bytes per launch from a committed ncu summary, when that summary
    was taken on the current kernel source (same digest); else None."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_digest") == digest:
            return int(float(kv["dram_bytes_per_launch_full_workload"]))
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, reasons, mx = [], set(), None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def nvtx_push(name):
    """Opens an NVTX range (a no-op without a profiler, or without NVTX)."""
    try:
        import torch

        torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


def nvtx_pop():
    try:
        import torch

        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


# ------------------------------------------------------------ device setup
def dev_tensor(a, device):
    import torch

    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def graph_time(fns, steps, warmup, stream, sampler=None, max_per_graph=64):
    """Runs `steps` calls (fns cycled) inside CUDA graphs; returns seconds of
    device time for exactly `steps` calls (events on the launching stream)."""
    import torch

    for i in range(warmup):
        fns[i % len(fns)]()
    torch.cuda.synchronize()
    per = min(max_per_graph, steps)
    if per >= len(fns):
        per -= per % len(fns)  # every graph starts on input copy 0
    graphs = []
    full, rem = divmod(steps, per)
    for n in ([per] if full else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fns[i % len(fns)]()
        graphs.append((g, n))
    torch.cuda.synchronize()
    for g, _ in graphs:  # warm the graphs
        g.replay()
    torch.cuda.synchronize()
    plan = [graphs[0][0]] * full + ([graphs[-1][0]] if rem else [])
    if sampler:
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for g in plan:
            g.replay()
        e1.record(stream)
    e1.synchronize()
    clocks = sampler.stop() if sampler else None
    return e0.elapsed_time(e1) / 1e3, clocks


def lone_call_time(call, copies, stream, device, n=50):
    """Median device time of one call with no neighbour to overlap: before
    each call the stream reads 512 MiB (evicting L2 with clean lines, so the
    call does not pay for write-backs, and giving the host time to queue the
    call), then CUDA events bracket the call alone."""
    import torch

    flush = torch.ones(128 << 20, dtype=torch.float32, device=device)
    acc = torch.zeros((), dtype=torch.float32, device=device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(3):  # warm-up
            call(copies[i % len(copies)])
        for i, (a, b) in enumerate(ev):
            torch.sum(flush, dim=0, out=acc)
            a.record(stream)
            call(copies[i % len(copies)])
            b.record(stream)
    torch.cuda.synchronize()
    del flush
    return statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3


# ------------------------------------------------------------------ arms
def cpu_oracle_decode(w, rank_threads=None, n_req=None):
    """The fp64 oracle over the decode workload (its first n_req requests,
    every query head, when n_req is given); returns (seconds, threads)."""
    import oracle

    n = rank_threads or (os.cpu_count() or 1)
    rows = None
    if n_req is not None and n_req < len(w["seq_lens"]):
        rows = np.arange(n_req * w["q"].shape[1], dtype=np.int32)
    t0 = time.perf_counter()
    oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"], rows=rows, n_threads=n)
    return time.perf_counter() - t0, n


REFERENCE_BUDGET_S = 120.0  # the timed steps of the reference arm, at most
CPU_LEG_BUDGET_S = 1.0  # one timed run of a cpu_baseline leg, about


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        return f"implementer {fields.get('cpu implementer', '?')} part {fields.get('cpu part', '?')}"
    except Exception:
        return "unknown"


def cpu_leg(run, work, n_units, unit_name, unit, scale, what):
    """The fp64 oracle on this host, once single-threaded and once on every
    core.  run(n, threads) runs it over the first n units of the workload;
    work(n) is their algorithmic bytes or flops.  For each thread count the
    sample grows from one unit until a run takes 0.1 s (or covers the whole
    workload), is then sized to about CPU_LEG_BUDGET_S, and the median of
    three runs of it is reported as work / time / scale."""
    legs = {}
    for threads in (1, os.cpu_count() or 1):
        def timed(n):
            t0 = time.perf_counter()
            run(n, threads)
            return time.perf_counter() - t0

        n = 1
        while True:
            t = timed(n)
            if t >= 0.1 or n >= n_units:
                break
            n = min(n_units, n * 4)
        n = int(min(n_units, max(n, n * CPU_LEG_BUDGET_S / max(t, 1e-6))))
        med = statistics.median(timed(n) for _ in range(3))
        legs[f"threads_{threads}"] = {
            "value": round(work(n) / med / scale, 4), "unit": unit, "threads": threads, "seconds": round(med, 4),
            "sample": f"first {n} of {n_units} {unit_name}" if n < n_units else f"all {n_units} {unit_name}"}
    return {"workload": what, **legs}


def cpu_leg_decode(w, what):
    import oracle

    hq = w["q"].shape[1]

    def run(n, threads):
        rows = None if n >= len(w["seq_lens"]) else np.arange(n * hq, dtype=np.int32)
        oracle.decode(w["q"], w["k_pages"], w["v_pages"], w["page_table"], w["seq_lens"], rows=rows,
                      n_threads=threads)

    return cpu_leg(run, lambda n: decode_bytes(w["seq_lens"][:n], hq=hq, hkv=w["k_pages"].shape[2]),
                   len(w["seq_lens"]), "requests (every query head)", "GB/s", 1e9, what)


def cpu_leg_prefill(w, what):
    import oracle

    cu, hq = w["cu_seqlens"], w["q"].shape[1]

    def run(n, threads):
        rows = None if n >= len(cu) - 1 else np.arange(int(cu[n]) * hq, dtype=np.int32)
        oracle.prefill(w["q"], w["k"], w["v"], cu, rows=rows, n_threads=threads)

    return cpu_leg(run, lambda n: prefill_flops(np.diff(cu)[:n], hq=hq), len(cu) - 1,
                   "requests (every token and query head)", "GFLOP/s", 1e9, what)


def cpu_leg_window(w, cu, what):
    import oracle

    h = w["q"].shape[1]

    def run(n, threads):
        rows = None if n >= len(cu) - 1 else np.arange(int(cu[n]) * h, dtype=np.int32)
        oracle.window(w["q"], w["k"], w["v"], cu, rows=rows, n_threads=threads)

    return cpu_leg(run, lambda n: window_flops(cu[:n + 1], h=h), len(cu) - 1, "windows (every token and head)",
                   "GFLOP/s", 1e9, what)


def cpu_leg_tiny(w, what):
    import oracle

    def run(n, threads):
        oracle.prefill(w["q"], w["k"], w["v"], w["cu_seqlens"], n_threads=threads)
        kp, vp = oracle.page_write(w["k"], w["v"], w["cu_seqlens"], w["page_table"], w["k_pages"], w["v_pages"])
        oracle.decode(w["decode_q"], kp, vp, w["page_table"], w["seq_lens"], n_threads=threads)

    # reported as steps per second: one step is the prefill of 64 tokens, its page write and one decode token
    return cpu_leg(run, lambda n: n, 1, "steps", "steps/s", 1.0, what)


def run_reference(args, world, rank):
    """The oracle as the reference arm, on this host's cores, rank 0 only.
    Each step is a bounded sample of the workload: all 32 requests when K
    steps of them fit in REFERENCE_BUDGET_S, else the first requests only
    (every query head of each), the bytes counted for that sample."""
    if rank != 0:
        return
    w = wl.decode_0p6b()
    B = len(w["seq_lens"])
    t_full, cores = cpu_oracle_decode(w)  # sizes the sample
    n_req = max(1, min(B, int(B * REFERENCE_BUDGET_S / (max(1, args.steps) * t_full))))
    nbytes = decode_bytes(w["seq_lens"][:n_req])
    for _ in range(args.warmup):
        cpu_oracle_decode(w, n_req=n_req)
    times = []
    for _ in range(args.steps):
        t, cores = cpu_oracle_decode(w, n_req=n_req)
        times.append(t)
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    sample = (f"first {n_req} of the {B} requests per step (every query head of each), fp64 oracle, "
              f"threads over rows")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": CONFIG_DECODE(w),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


METRIC = "paged GQA decode attn HBM GB/s (% of peak); prefill/window attn TFLOP/s"


def CONFIG_DECODE(w):
    return {"workload": "batched decode 0.6B Thinker shape: 32 requests, GQA 16/8, head_dim 128, "
                        "context ~U[200,2000], 16-token pages over a 4096-page pool (seeded shuffle)",
            "batch": int(len(w["seq_lens"])), "sum_seq_len": int(np.sum(w["seq_lens"])),
            "l2": "4 rotating layer copies of q and the KV pools (~576 MB > 129 MB L2); page table and "
                  "lengths shared by the layers of a step", "stable_metadata": 2, "parallelism": "replicas"}


def max_over_ranks(x, dist, device):
    """The largest x over all ranks (x itself when dist is None): the job's
    time is its slowest rank's."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, seconds, world):
    """Whole-job throughput: every rank processes units_per_rank (weak
    scaling, no data-path collective) in the slowest rank's time."""
    return units_per_rank * world / seconds


def run_ours(args, world, rank, local_rank):
    import torch

    import paged_kv_gqa_attention_gb300 as qa

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()
    dist = None
    if world > 1:
        import torch.distributed as dist  # timing barrier / max only; no data-path collective

    # ---------------- headline: batched decode 0.6B
    w = wl.decode_0p6b()
    nbytes = decode_bytes(w["seq_lens"])
    # Four rotating copies of the per-layer inputs (q and the KV pools: four
    # decoder layers' caches); the page table and lengths are shared, as they
    # are by every layer of one decode step.
    shared = {k: dev_tensor(w[k], device) for k in ("page_table", "seq_lens")}
    copies = []
    for _ in range(4):
        c = {k: dev_tensor(w[k], device) for k in ("q", "k_pages", "v_pages")}
        c.update(shared)
        copies.append(c)
    B = len(w["seq_lens"])
    ws_bytes = qa.qa_decode_workspace_size(B, int(w["seq_lens"].max()), num_pages=4096, max_pages_per_seq=125)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    out = torch.empty(B, 16, 128, dtype=torch.bfloat16, device=device)

    # The layers of a step share the page table and lengths and none of them
    # writes those or another layer's pools, so each call may read them, and
    # stream its first pages, before the previous layer's kernel ends
    # (stable_metadata = 2); the same calls at levels 0 and 1 are timed too.
    def mk(c, stable):
        return lambda: qa.qa_decode_attn(c["q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"], out,
                                         workspace=ws, stream=stream, stable_metadata=stable)

    fns = [mk(c, 2) for c in copies]
    nvtx_push("headline")
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    elapsed, clocks = graph_time(fns, args.steps, args.warmup, stream, sampler)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed = max_over_ranks(elapsed, dist, device)
    status = qa.qa_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed region")
    per_call = elapsed / args.steps
    gbs = nbytes / per_call / 1e9
    value = job_rate(nbytes, per_call, world) / 1e9
    by_level = {}
    for level in (0, 1):
        el, _ = graph_time([mk(c, level) for c in copies], args.steps, args.warmup, stream)
        el = max_over_ranks(el, dist, device)
        by_level[str(level)] = {"value": round(job_rate(nbytes, el / args.steps, world) / 1e9, 2), "unit": "GB/s",
                                "ms_per_step": round(el / args.steps * 1e3, 5)}
    by_level["note"] = ("the same calls at stable_metadata 0 (everything read after the wait) and 1 (lengths and "
                        "page table read before it); the headline uses 2 (first pool pages streamed before it too)")
    nvtx_pop()
    nvtx_push("lone_call")
    lone = lone_call_time(lambda c: mk(c, 0)(), copies, stream, device)
    nvtx_pop()
    lone_call = {"value": round(nbytes / lone / 1e9, 2), "unit": "GB/s", "us_per_call": round(lone * 1e6, 3),
                 "frac": round(nbytes / lone / 1e9 / peaks["hbm"], 4),
                 "mode": "one call at a time (stable_metadata 0): 512 MiB read before each call to evict L2, "
                         "then CUDA events around the call alone; median of 50 calls"}

    # ---------------- end to end: host buffers, copies inside the timed region
    # a step's inputs (q, page table, lengths) sit side by side in one pinned
    # staging buffer and go over in one copy, as a serving loop stages them
    q_np, pt_np, sl_np = w["q"].view(np.int16), w["page_table"], w["seq_lens"]
    sizes = [q_np.nbytes, pt_np.nbytes, sl_np.nbytes]
    offs = [0, sizes[0], sizes[0] + sizes[1]]
    assert all(o % 16 == 0 for o in offs)
    hin = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
    din = torch.empty(sum(sizes), dtype=torch.uint8, device=device)

    def views(buf):
        return (buf[offs[0]:offs[0] + sizes[0]].view(torch.bfloat16).view(q_np.shape),
                buf[offs[1]:offs[1] + sizes[1]].view(torch.int32).view(pt_np.shape),
                buf[offs[2]:offs[2] + sizes[2]].view(torch.int32).view(sl_np.shape))

    hq, hpt, hsl = views(hin)
    hq.view(torch.int16).copy_(torch.from_numpy(q_np))
    hpt.copy_(torch.from_numpy(pt_np))
    hsl.copy_(torch.from_numpy(sl_np))
    dq, dpt, dsl = views(din)
    hout = torch.empty(B, 16, 128, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 2000))
    checksum = 0.0

    def enqueue(c):  # one step's work on the stream: inputs in, the decode, the result out
        din.copy_(hin, non_blocking=True)
        qa.qa_decode_attn(dq, c["k_pages"], c["v_pages"], dpt, dsl, out, workspace=ws, stream=stream)
        hout.copy_(out, non_blocking=True)

    def e2e_eager(c):
        with torch.cuda.stream(stream):
            enqueue(c)
        stream.synchronize()
        return float(hout[0, 0, 0])  # the host reads the result

    # the same step captured once per layer copy as a CUDA graph (copies,
    # decode and read-back), replayed every step: how a serving loop issues it
    with torch.cuda.stream(stream):
        enqueue(copies[0])
    stream.synchronize()
    step_graphs = []
    for c in copies:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue(c)
        step_graphs.append(g)
    torch.cuda.synchronize()

    def e2e_graph(i):
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            step_graphs[i % 4].replay()
        stream.synchronize()
        return float(hout[0, 0, 0])  # the host reads the result

    def check_e2e(j):
        # the last step read back the right result: the same call on the
        # device-resident inputs of layer copy j gives the same output
        torch.cuda.synchronize()
        got = hout.float().clone()
        c = copies[j]
        qa.qa_decode_attn(c["q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"], out, workspace=ws,
                          stream=stream)
        stream.synchronize()
        diff = float((out.float().cpu() - got).abs().max())
        assert diff <= 1e-2, f"end-to-end step output differs from the device-resident call by {diff}"
        return True

    def e2e_time(step):
        nonlocal checksum
        for i in range(max(3, args.warmup)):
            step(i)
        torch.cuda.synchronize()
        hout.fill_(float("nan"))  # only the timed steps can leave a result there
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            checksum += step(i)
        return max_over_ranks(time.perf_counter() - t0, dist, device)

    e2e_elapsed = e2e_time(lambda i: e2e_graph(i))
    e2e_value = job_rate(nbytes, e2e_elapsed / e2e_steps, world) / 1e9
    check_e2e((e2e_steps - 1) % 4)
    e2e_eager_elapsed = e2e_time(lambda i: e2e_eager(copies[i % 4]))
    e2e_eager_value = job_rate(nbytes, e2e_eager_elapsed / e2e_steps, world) / 1e9
    check_e2e((e2e_steps - 1) % 4)
    del step_graphs

    # the same step with no copy engine: the kernel reads q, the page table
    # and the lengths straight out of the pinned staging buffer and writes its
    # output straight into pinned host memory (both reachable from the GPU
    # over NVLink-C2C with unified addressing), so a step is one launch and a
    # host read; captured once per layer copy with the library's own graph
    # API (qa_decode_graph_create) and launched every step (qa_graph_launch)
    hout_zc = torch.empty(B, 16, 128, dtype=torch.bfloat16).pin_memory()
    hout_zc_np = hout_zc.view(torch.int16).numpy()  # the host reads the result through this view
    zc_graphs = [qa.qa_decode_graph_create([hq], [c["k_pages"]], [c["v_pages"]], hpt, hsl, [hout_zc], workspace=ws)
                 for c in copies]
    torch.cuda.synchronize()

    def e2e_zc(i):
        zc_graphs[i % 4].launch(stream=stream)
        stream.synchronize()
        return float(hout_zc_np[0, 0, 0])  # the host reads the result

    def zc_time():
        nonlocal checksum
        for i in range(max(3, args.warmup)):
            e2e_zc(i)
        torch.cuda.synchronize()
        hout_zc.fill_(float("nan"))
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            checksum += e2e_zc(i)
        return max_over_ranks(time.perf_counter() - t0, dist, device)

    zc_elapsed = zc_time()
    zc_value = job_rate(nbytes, zc_elapsed / e2e_steps, world) / 1e9
    torch.cuda.synchronize()
    got_zc = hout_zc.float().clone()
    cj = copies[(e2e_steps - 1) % 4]
    qa.qa_decode_attn(cj["q"], cj["k_pages"], cj["v_pages"], cj["page_table"], cj["seq_lens"], out, workspace=ws,
                      stream=stream)
    stream.synchronize()
    diff = float((out.float().cpu() - got_zc).abs().max())
    assert diff <= 1e-2, f"zero-copy step output differs from the device-resident call by {diff}"
    for g in zc_graphs:
        g.close()
    h2d = hin.numel()  # q, page table and lengths
    d2h = hout.numel() * 2

    digest = source_digest("decode.cu", "common.cuh")
    roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm"], 4),
                "traffic": profiled_traffic("decode_splitk_decode0p6b.txt", digest),
                "kernel": "decode_splitk_kernel (one qa_decode_attn call = one launch)",
                "algorithmic_bytes_per_launch": nbytes, "peak_source": peaks["source"] + " (burst copy)",
                "source_digest": digest}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_call * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": CONFIG_DECODE(w),
        "clocks": clocks,
        "e2e": {"value": round(zc_value, 3), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": e2e_steps, "ms_per_step": round(zc_elapsed / e2e_steps * 1e3, 4),
                "mode": "each step through the C ABI with host buffers: the kernel reads q, the page table and the "
                        "lengths from one pinned host staging buffer and writes the output into pinned host memory "
                        "(those bytes cross the host link inside the timed region; the KV pools are the resident "
                        "cache), one launch per step (a one-kernel graph captured with qa_decode_graph_create, "
                        "launched with qa_graph_launch), then the host reads the result",
                "copy_engine": {"value": round(e2e_value, 3), "unit": "GB/s",
                                "ms_per_step": round(e2e_elapsed / e2e_steps * 1e3, 4),
                                "mode": "the same step with the inputs copied in (one copy from the pinned staging "
                                        "buffer) and the output copied back by the copy engine; copies and "
                                        "decode captured as one graph"},
                "eager_calls": {"value": round(e2e_eager_value, 3), "unit": "GB/s",
                                "ms_per_step": round(e2e_eager_elapsed / e2e_steps * 1e3, 4),
                                "mode": "the copy-engine step issued call by call from Python"}},
        "gpu_launches": args.steps, "roofline": roofline,
        "tokens_per_s": round(B / per_call * world, 1), "by_stable_metadata": by_level, "lone_call": lone_call,
    }
    del copies
    torch.cuda.empty_cache()

    rows = {"all": ROW_NAMES, "none": ()}.get(args.rows, tuple(r for r in args.rows.split(",") if r))
    unknown = set(rows) - set(ROW_NAMES)
    if unknown:
        raise SystemExit(f"unknown rows: {sorted(unknown)}")
    # the oracle on this host's cores (rank 0 of a single-GPU run only)
    cpu = {} if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rows:
        line["rows"] = measure_rows(qa, device, stream, peaks, args, rows, cpu)

    if cpu is not None:
        cpu["decode_0p6b"] = cpu_leg_decode(w, "batched decode 0.6B: 32 requests, L~U[200,2000]")
        head = cpu["decode_0p6b"][f"threads_{os.cpu_count() or 1}"]
        line["cpu_baseline"] = {"value": head["value"], "unit": "GB/s", "cores": head["threads"], "kind": "oracle",
                                "sample": f"batched decode 0.6B, {head['sample']}, fp64, median of 3 runs",
                                "cpu_model": cpu_model(), "cpu_count": os.cpu_count(),
                                "configs": cpu}
    if rank == 0:
        print(json.dumps(line))


ROW_NAMES = ("prefill", "chunk_prefill", "window", "decode_long", "decode_step", "cross_decode", "decode_graph",
             "tiny", "encoder_layer")


def measure_rows(qa, device, stream, peaks, args, which=ROW_NAMES, cpu=None):
    """The other hot-path operations, each timed the same way (graphs of
    back-to-back calls, inputs in HBM, above L2 or rotated).  With a `cpu`
    dict, the oracle's legs for the named workloads go there too."""
    import torch

    rows = {}
    steps = max(20, min(args.steps, 400))
    table = (("prefill", lambda: _row_prefill(qa, device, stream, peaks, steps, rows, cpu)),
             ("chunk_prefill", lambda: _row_chunk_prefill(qa, device, stream, peaks, steps, rows)),
             ("window", lambda: _row_window(qa, device, stream, peaks, steps, rows, cpu)),
             ("decode_long", lambda: _row_decode_long(qa, device, stream, peaks, steps, rows, cpu)),
             ("decode_step", lambda: _row_decode_step(qa, device, stream, peaks, steps, rows)),
             ("cross_decode", lambda: _row_cross_decode(qa, device, stream, peaks, steps, rows)),
             ("decode_graph", lambda: _row_decode_graph(qa, device, stream, peaks, steps, rows)),
             ("tiny", lambda: _row_tiny(qa, device, stream, steps, rows, cpu)),
             ("encoder_layer", lambda: _row_encoder_layer(qa, device, stream, peaks, steps, rows)))
    for name, run in table:
        if name in which:
            # an NVTX range per row, so a profiler can select one row's kernels
            # (e.g. ncu --nvtx --nvtx-include "row:window/")
            nvtx_push(f"row:{name}")
            run()
            nvtx_pop()
    status = qa.qa_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status:#x} after the row measurements")
    torch.cuda.empty_cache()
    return rows


def _row_prefill(qa, device, stream, peaks, steps, rows, cpu=None):
    """Ragged causal prefill with page write (16 requests, ~3.6K tokens)."""
    import torch

    w = wl.prefill_bucket()
    T = int(w["cu_seqlens"][-1])
    cps = []
    for _ in range(4):
        cps.append({k: dev_tensor(w[k], device) for k in ("q", "k", "v", "cu_seqlens", "page_table", "k_pages", "v_pages")})
    outp = torch.empty(T, 16, 128, dtype=torch.bfloat16, device=device)

    # no kernel of the sequence writes the segments or page tables: each call
    # may set its job up before the previous one ends (stable_metadata = 1)
    def mkp(c, level):
        return lambda: qa.qa_prefill_attn(c["q"], c["k"], c["v"], c["cu_seqlens"], c["page_table"], c["k_pages"],
                                          c["v_pages"], outp, stream=stream, stable_metadata=level)

    el, _ = graph_time([mkp(c, 1) for c in cps], steps, 5, stream)
    t = el / steps
    el0, _ = graph_time([mkp(c, 0) for c in cps], steps, 5, stream)
    fl, by = prefill_flops(w["lengths"]), prefill_bytes(T)
    rows["prefill"] = {"workload": "ragged causal prefill + KV page write: 16 requests, ceil(13 d)+40 tokens "
                                   "(d~U[1,30] s), GQA 16/8 x 128", "total_tokens": T, "us_per_call": round(t * 1e6, 2),
                       "tflops": round(fl / t / 1e12, 3), "gbs": round(by / t / 1e9, 1),
                       "frac_bf16_peak": round(fl / t / 1e12 / peaks["bf16"], 4),
                       "frac_hbm": round(by / t / 1e9 / peaks["hbm"], 4), "flops": fl, "bytes": by,
                       "gpu_launches_per_call": 1, "stable_metadata": 1,
                       "us_per_call_stable_metadata_0": round(el0 / steps * 1e6, 2)}
    if cpu is not None:
        cpu["prefill_bucket"] = cpu_leg_prefill(w, "ragged causal prefill: 16 requests, ceil(13 d)+40 tokens")


def _row_chunk_prefill(qa, device, stream, peaks, steps, rows):
    """Chunked prefill: 16 requests with their audio prompt cached, 16..128
    new tokens each."""
    import torch

    w = wl.chunk_reprefill()
    T = int(w["cu_seqlens"][-1])
    keys = ("q", "k", "v", "cu_seqlens", "n_past", "page_table", "k_pages", "v_pages")
    cps = [{k: dev_tensor(w[k], device) for k in keys} for _ in range(4)]
    outp = torch.empty(T, 16, 128, dtype=torch.bfloat16, device=device)

    def mk(c, level):
        return lambda: qa.qa_prefill_chunk_attn(c["q"], c["k"], c["v"], c["cu_seqlens"], c["n_past"],
                                                c["page_table"], c["k_pages"], c["v_pages"], outp, stream=stream,
                                                stable_metadata=level)

    el, _ = graph_time([mk(c, 1) for c in cps], steps, 5, stream)
    t = el / steps
    el0, _ = graph_time([mk(c, 0) for c in cps], steps, 5, stream)
    past, new = w["n_past"].astype(np.int64), w["lengths"].astype(np.int64)
    fl = int(np.sum(4 * 16 * 128 * (new * past + new * (new + 1) // 2)))
    by = int(prefill_bytes(T) + np.sum(past) * 8 * 128 * 2 * 2)  # + the cached K/V, once
    rows["chunk_prefill"] = {"workload": "chunked prefill: 16 requests, cached ceil(13 d)+40 tokens (d~U[1,30] s), "
                                         "16..128 new tokens, GQA 16/8 x 128, new K/V written at n_past",
                             "new_tokens": T, "cached_tokens": int(np.sum(past)), "us_per_call": round(t * 1e6, 2),
                             "tflops": round(fl / t / 1e12, 3), "gbs": round(by / t / 1e9, 1),
                             "frac_hbm": round(by / t / 1e9 / peaks["hbm"], 4), "flops": fl, "bytes": by,
                             "gpu_launches_per_call": 1, "stable_metadata": 1,
                             "us_per_call_stable_metadata_0": round(el0 / steps * 1e6, 2)}


def _row_window(qa, device, stream, peaks, steps, rows, cpu=None):
    """AuT windowed attention (8 requests, ~70K tokens, 14 x 64)."""
    import torch

    w = wl.window_aut()
    cu = qa.qa_window_plan(w["token_counts"])
    T = int(cu[-1])
    cps = []
    for _ in range(2):
        cps.append({k: dev_tensor(w[k], device) for k in ("q", "k", "v")})
    dcu = dev_tensor(cu, device)
    outw = torch.empty(T, 14, 64, dtype=torch.bfloat16, device=device)

    # jobs claimed from a counter in a workspace (the CTAs finish together);
    # the fixed job order (no workspace) is timed beside it
    ws = torch.zeros(qa.qa_window_workspace_size(), dtype=torch.uint8, device=device)

    def mkw(c, workspace):
        return lambda: qa.qa_window_attn(c["q"], c["k"], c["v"], dcu, outw, workspace=workspace, stream=stream)

    n = max(10, steps // 4)
    el, _ = graph_time([mkw(c, ws) for c in cps], n, 3, stream)
    t = el / n
    el_fixed, _ = graph_time([mkw(c, None) for c in cps], n, 3, stream)
    fl, by = window_flops(cu), window_bytes(T)
    rows["window"] = {"workload": "AuT windowed attention: 8 requests d~U[10,1200] s, 104-token windows, 14 x 64",
                      "total_tokens": T, "windows": int(len(cu) - 1), "us_per_call": round(t * 1e6, 2),
                      "us_per_call_fixed_job_order": round(el_fixed / n * 1e6, 2),
                      "tflops": round(fl / t / 1e12, 3), "gbs": round(by / t / 1e9, 1),
                      "frac_bf16_peak": round(fl / t / 1e12 / peaks["bf16"], 4),
                      "frac_hbm": round(by / t / 1e9 / peaks["hbm"], 4), "flops": fl, "bytes": by,
                      "gpu_launches_per_call": 1}
    if cpu is not None:
        cpu["window_aut"] = cpu_leg_window(w, cu, "AuT windowed attention: 8 requests, 104-token windows, 14 x 64")


def _row_decode_long(qa, device, stream, peaks, steps, rows, cpu=None):
    """Long-context decode 1.7B (64 requests, ~9K tokens each)."""
    import torch

    w = wl.decode_1p7b()
    c = {k: dev_tensor(w[k], device) for k in ("q", "k_pages", "v_pages", "page_table", "seq_lens")}
    B = len(w["seq_lens"])
    ws = torch.zeros(qa.qa_decode_workspace_size(B, int(w["seq_lens"].max()), num_pages=65536, max_pages_per_seq=1000),
                     dtype=torch.uint8, device=device)
    outd = torch.empty(B, 16, 128, dtype=torch.bfloat16, device=device)
    f = lambda: qa.qa_decode_attn(c["q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"], outd,  # noqa
                                  workspace=ws, stream=stream, stable_metadata=2)
    n = max(10, steps // 4)
    el, _ = graph_time([f], n, 3, stream)
    t = el / n
    by = decode_bytes(w["seq_lens"])
    rows["decode_long"] = {"workload": "long-context decode 1.7B Thinker shape: 64 requests, L~U[2000,16000], "
                                       "65536-page pool", "sum_seq_len": int(np.sum(w["seq_lens"])),
                           "us_per_call": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                           "frac_hbm": round(by / t / 1e9 / peaks["hbm"], 4), "bytes": by,
                           "tokens_per_s": round(B / t, 1), "gpu_launches_per_call": 1, "stable_metadata": 2}
    del c
    torch.cuda.empty_cache()
    if cpu is not None:
        cpu["decode_1p7b"] = cpu_leg_decode(w, "long-context decode 1.7B: 64 requests, L~U[2000,16000]")


def append_bytes(batch, hq=16, hkv=8, d=128):
    """Algorithmic bytes of one decode append: the new token's q, k, v read,
    the two gains, the rotated q written and the K/V slot rows written."""
    return batch * d * 2 * (hq + 2 * hkv) * 2 + 2 * d * 4


def _row_decode_step(qa, device, stream, peaks, steps, rows):
    """Decode step of the 0.6B workload: QK-norm + RoPE + KV append, then the
    paged decode (two launches, the second launched early)."""
    import torch

    w = wl.with_append(wl.decode_0p6b(), 2)
    B = len(w["seq_lens"])
    pt, sl = dev_tensor(w["page_table"], device), dev_tensor(w["seq_lens"], device)
    gq, gk = dev_tensor(w["q_gain"], device), dev_tensor(w["k_gain"], device)
    cps = []
    for _ in range(4):  # layer copies: new-token projections and the pools (> L2 in all)
        cps.append({k: dev_tensor(w[k], device) for k in ("q_new", "k_new", "v_new", "k_pages", "v_pages")})
    ws = torch.zeros(qa.qa_decode_workspace_size(B, int(w["seq_lens"].max()), num_pages=4096, max_pages_per_seq=125),
                     dtype=torch.uint8, device=device)
    q_rot = torch.empty(B, 16, 128, dtype=torch.bfloat16, device=device)
    outd = torch.empty(B, 16, 128, dtype=torch.bfloat16, device=device)

    def fused(c):
        return lambda: qa.qa_decode_step(c["q_new"], c["k_new"], c["v_new"], gq, gk, pt, sl, c["k_pages"],
                                         c["v_pages"], outd, workspace=ws, rms_eps=w["rms_eps"],
                                         rope_theta=w["rope_theta"], stream=stream, stable_metadata=2)

    def two_calls(c):
        def step():
            qa.qa_decode_append(c["q_new"], c["k_new"], c["v_new"], gq, gk, pt, sl, c["k_pages"], c["v_pages"],
                                q_out=q_rot, rms_eps=w["rms_eps"], rope_theta=w["rope_theta"], stream=stream)
            qa.qa_decode_attn(q_rot, c["k_pages"], c["v_pages"], pt, sl, outd, workspace=ws, stream=stream,
                              stable_metadata=True)
        return step

    n = max(20, steps // 2)
    el, _ = graph_time([fused(c) for c in cps], n, 5, stream)
    t = el / n
    el2, _ = graph_time([two_calls(c) for c in cps], n, 5, stream)
    t2 = el2 / n
    by = decode_bytes(w["seq_lens"]) + append_bytes(B)
    rows["decode_step"] = {"workload": "decode step 0.6B: per-head QK-norm + NEOX RoPE (theta 1e6) + KV append of "
                                       "the new token and paged GQA decode (qa_decode_step, one launch); "
                                       "32 requests, L~U[200,2000]",
                           "us_per_step": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                           "frac_hbm": round(by / t / 1e9 / peaks["hbm"], 4), "bytes": by,
                           "tokens_per_s": round(B / t, 1), "gpu_launches_per_step": 1,
                           "us_per_step_two_calls": round(t2 * 1e6, 2),
                           "two_calls": "qa_decode_append then qa_decode_attn (2 launches; the decode at "
                                        "stable_metadata 1: the append writes its pools)", "stable_metadata": 2}
    del cps
    torch.cuda.empty_cache()


def _row_cross_decode(qa, device, stream, peaks, steps, rows):
    """Paged cross-attention decode: 32 requests x 1500 encoder frames, 8 query
    heads over 8 KV heads (a cache written once, read every step)."""
    import torch

    B, L, H = 32, 1500, 8
    n_pages = B * -(-L // 16)
    w = wl.decode_workload(6, [L] * B, num_pages=n_pages, max_pages=-(-L // 16), hq=H, hkv=H)
    pt, sl = dev_tensor(w["page_table"], device), dev_tensor(w["seq_lens"], device)
    cps = [{k: dev_tensor(w[k], device) for k in ("q", "k_pages", "v_pages")} for _ in range(2)]  # 2 x 197 MB > L2
    ws = torch.zeros(qa.qa_decode_workspace_size(B, L, n_q_heads=H, n_kv_heads=H, num_pages=n_pages,
                                                 max_pages_per_seq=-(-L // 16)), dtype=torch.uint8, device=device)
    outd = torch.empty(B, H, 128, dtype=torch.bfloat16, device=device)

    def mk(c):
        return lambda: qa.qa_decode_attn(c["q"], c["k_pages"], c["v_pages"], pt, sl, outd, workspace=ws,
                                         stream=stream, stable_metadata=2)

    n = max(20, steps // 2)
    el, _ = graph_time([mk(c) for c in cps], n, 5, stream)
    t = el / n
    by = decode_bytes(w["seq_lens"], hq=H, hkv=H)
    rows["cross_decode"] = {"workload": "paged cross-attention decode: 32 requests x 1500 encoder frames, "
                                        "8 query heads over 8 KV heads x 128, 16-token pages",
                            "us_per_call": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                            "frac_hbm": round(by / t / 1e9 / peaks["hbm"], 4), "bytes": by,
                            "gpu_launches_per_call": 1, "stable_metadata": 2}
    del cps
    torch.cuda.empty_cache()


def _row_decode_graph(qa, device, stream, peaks, steps, rows):
    """A whole 28-layer decode step of the 0.6B workload captured once
    (qa_decode_graph_create) and replayed with one launch, against the same
    28 calls launched one by one from the host."""
    import torch

    n_layers = 28
    w = wl.decode_0p6b()
    B = len(w["seq_lens"])
    pt, sl = dev_tensor(w["page_table"], device), dev_tensor(w["seq_lens"], device)
    cps = [{k: dev_tensor(w[k], device) for k in ("q", "k_pages", "v_pages")} for _ in range(4)]  # > L2, cycled
    layers = [cps[i % 4] for i in range(n_layers)]
    outs = [torch.empty(B, 16, 128, dtype=torch.bfloat16, device=device) for _ in range(n_layers)]
    ws = torch.zeros(qa.qa_decode_workspace_size(B, int(w["seq_lens"].max()), num_pages=4096, max_pages_per_seq=125),
                     dtype=torch.uint8, device=device)
    g = qa.qa_decode_graph_create([c["q"] for c in layers], [c["k_pages"] for c in layers],
                                  [c["v_pages"] for c in layers], pt, sl, outs, workspace=ws, stable_metadata=2)
    n = max(5, min(50, steps // 40))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def run(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    def eager():
        for i, c in enumerate(layers):
            qa.qa_decode_attn(c["q"], c["k_pages"], c["v_pages"], pt, sl, outs[i], workspace=ws, stream=stream,
                              stable_metadata=2)

    t_graph = run(lambda: g.launch(stream=stream))
    t_eager = run(eager)
    g.close()
    by = decode_bytes(w["seq_lens"]) * n_layers
    rows["decode_graph"] = {"workload": "28-layer decode step of the 0.6B workload (32 requests, L~U[200,2000]) "
                                        "captured as one CUDA graph (qa_decode_graph_create)",
                            "us_per_step": round(t_graph * 1e6, 2), "us_per_layer": round(t_graph * 1e6 / n_layers, 2),
                            "gbs": round(by / t_graph / 1e9, 1), "frac_hbm": round(by / t_graph / 1e9 / peaks["hbm"], 4),
                            "us_per_step_eager_calls": round(t_eager * 1e6, 2), "gpu_launches_per_step": n_layers,
                            "stable_metadata": 2}
    del cps, layers
    torch.cuda.empty_cache()


def _row_tiny(qa, device, stream, steps, rows, cpu=None):
    """Tiny: prefill of 64 tokens then one decode token (latency)."""
    import torch

    w = wl.tiny()
    c = {k: dev_tensor(w[k], device) for k in ("q", "k", "v", "cu_seqlens", "page_table", "k_pages", "v_pages",
                                                "decode_q", "seq_lens")}
    outt = torch.empty(64, 16, 128, dtype=torch.bfloat16, device=device)
    outd = torch.empty(1, 16, 128, dtype=torch.bfloat16, device=device)
    ws = torch.zeros(qa.qa_decode_workspace_size(1, 64, num_pages=4, max_pages_per_seq=4), dtype=torch.uint8,
                     device=device)

    def tiny_step():
        qa.qa_prefill_attn(c["q"], c["k"], c["v"], c["cu_seqlens"], c["page_table"], c["k_pages"], c["v_pages"], outt,
                           stream=stream)
        qa.qa_decode_attn(c["decode_q"], c["k_pages"], c["v_pages"], c["page_table"], c["seq_lens"], outd,
                          workspace=ws, stream=stream)

    el, _ = graph_time([tiny_step], steps, 5, stream)
    rows["tiny"] = {"workload": "tiny: prefill of 64 tokens into 4 permuted pages, then 1 decode token",
                    "us_per_step": round(el / steps * 1e6, 2), "note": "latency-bound; no roofline fraction",
                    "gpu_launches_per_step": 2}
    if cpu is not None:
        cpu["tiny"] = cpu_leg_tiny(w, "tiny: prefill of 64 tokens, its page write, then 1 decode token")


def encoder_flops(T, cu, d=896, h=14, d_ffn=3584):
    """Algorithmic flops of one encoder layer: the four projections
    (2 T d (3 d + d + 2 d_ffn)) and the window attention."""
    return int(2 * T * d * (3 * d + d + 2 * d_ffn)) + window_flops(cu, h=h, d=d // h)


def _row_encoder_layer(qa, device, stream, peaks, steps, rows):
    """One AuT encoder layer (0.6B: d_model 896, 14 x 64 heads, FFN 3584)
    over the AuT window workload's 70 220 tokens: the whole layer (seven
    launches) and each projection alone, graphs of back-to-back calls."""
    import torch

    w = wl.encoder_layer_aut()
    cu = qa.qa_window_plan(w["token_counts"])
    T, d = w["x"].shape
    d_ffn = w["d_ffn"]
    x = dev_tensor(w["x"], device)
    dcu = dev_tensor(cu, device)
    W = {k: dev_tensor(v, device) for k, v in w["weights"].items()}
    ws = torch.empty(qa.qa_encoder_workspace_size(T, d, d_ffn), dtype=torch.uint8, device=device)
    out = torch.empty_like(x)

    def layer():
        qa.qa_encoder_layer(x, dcu, W, out, n_heads=w["n_heads"], ln_eps=w["eps"], workspace=ws, stream=stream)

    n = max(5, min(40, steps // 10))
    el, clocks = graph_time([layer], n, 3, stream, ClockSampler(0))
    t = el / n
    fl = encoder_flops(T, cu, d, w["n_heads"], d_ffn)
    # each projection alone (inputs and outputs > L2)
    a = torch.randn(T, d, device=device).to(torch.bfloat16)
    big = torch.randn(T, d_ffn, device=device).to(torch.bfloat16)
    qkv = torch.empty(T, 3 * d, dtype=torch.bfloat16, device=device)
    proj = {
        "qkv": (lambda: qa.qa_linear(a, W["w_qkv"], W["b_qkv"], qkv, stream=stream), 2 * T * d * 3 * d),
        "out_proj_residual": (lambda: qa.qa_linear(a, W["w_o"], W["b_o"], out, residual=x, stream=stream),
                              2 * T * d * d),
        "fc1_gelu": (lambda: qa.qa_linear(a, W["w_fc1"], W["b_fc1"], big, gelu=True, stream=stream),
                     2 * T * d * d_ffn),
        "fc2_residual": (lambda: qa.qa_linear(big, W["w_fc2"], W["b_fc2"], out, residual=x, stream=stream),
                         2 * T * d_ffn * d),
        "layer_norm": (lambda: qa.qa_layer_norm(x, W["ln1_g"], W["ln1_b"], a, eps=w["eps"], stream=stream), 0),
    }
    parts = {}
    m = max(5, min(40, steps // 10))
    for name, (fn, pfl) in proj.items():
        e, _ = graph_time([fn], m, 3, stream)
        tt = e / m
        parts[name] = {"us_per_call": round(tt * 1e6, 2)}
        if pfl:
            parts[name].update({"tflops": round(pfl / tt / 1e12, 1),
                                "frac_bf16_peak": round(pfl / tt / 1e12 / peaks["bf16"], 4),
                                "frac_bf16_sustained": round(pfl / tt / 1e12 / peaks["bf16_sustained"], 4)})
        else:
            by = 2 * T * d * 2
            parts[name].update({"gbs": round(by / tt / 1e9, 1), "frac_hbm": round(by / tt / 1e9 / peaks["hbm"], 4)})
    rows["encoder_layer"] = {
        "workload": "AuT encoder layer 0.6B (d_model 896, 14 x 64 heads, FFN 3584, LayerNorm eps 1e-5) over the "
                    "AuT window workload: 70 220 tokens, 680 windows of <= 104; synthetic weights",
        "total_tokens": T, "us_per_layer": round(t * 1e6, 2), "tflops": round(fl / t / 1e12, 1),
        "frac_bf16_peak": round(fl / t / 1e12 / peaks["bf16"], 4),
        "frac_bf16_sustained": round(fl / t / 1e12 / peaks["bf16_sustained"], 4), "flops": fl,
        "gpu_launches_per_layer": 7, "parts": parts, "clocks": clocks}
    del ws, big, qkv, a
    torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--rows", default="all",
                    help="other hot-path rows to measure: all, none, or a comma list of " + ",".join(ROW_NAMES))
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline leg")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local_rank)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
