"""Benchmark of the fused FP8 attention forward on one GB300 (or N replicas).

Headline: causal GQA prefill (B=2, Hq=32, Hkv=8, S=4096, d=dv=128, E4M3 in, bf16 out) in
TFLOP/s of algorithmic work (2*(d+dv) flops per unmasked (row, key) pair), against the
dense FP8 tensor peak.  The same line carries the paged decode workload (B=64, 1 token,
Hq=64, Hkv=8, d=dv=128, 16-token pages, keys ~U[1024,32768]) in GB/s against HBM, every
configured workload on its own roofline (`configs`), and the fp64 oracle's throughput on
each workload at one host thread and at all host threads (`cpu_baseline`).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Timing: W untimed steps, then K steps; before every step a 256 MB buffer is written to
flush L2 (129 MB); each step's forward call is bracketed by CUDA events on the launching
stream; ms_per_step is the mean over the K steps, max over ranks.  `e2e` repeats the
measurement through the public call with the inputs copied from pinned host memory and
the output copied back inside the timed region (pipelined over two buffer sets so that the
copies of neighbouring steps overlap the forward; the serial time is reported beside it).
`--impl reference` times the fp64 CPU oracle (the only reference this path has) on the same
workload: W warm-up and K timed steps, each a bounded sample of rows on all host cores.
Tensor-bound fractions also come as `frac_at_run_clock`: the measured peak was taken at a
lower SM clock (its median under load) than this run's, so the same work at this run's clock
is compared with the peak scaled to that clock.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_attention_forward_gb300 import inputs  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
METRIC = "FP8 attn fwd TFLOP/s (prefill) & decode HBM GB/s; % of GB300 roofline"

# DRAM bytes (read + write) per launch from one ncu capture of each timed kernel (summaries
# under profiles/), valid only while the kernel sources hash to the value recorded with it.
PROFILED_TRAFFIC = {
    "prefill": {"kernel": "prefill_kernel<128,128>", "bytes": 66.99e6,
                "sources": ["fa8_prefill.cuh", "fa8_kernel.cuh", "fa8_ptx.cuh"], "sha256_16": "72f1db867eccda7f"},
    "decode": {"kernel": "decode_kernel<128,128,8>", "bytes": 2073.87e6,
               "sources": ["fa8_decode.cuh", "fa8_kernel.cuh", "fa8_ptx.cuh"], "sha256_16": "a05c4dac8dc4257e"},
}


def _profiled_traffic(which):
    """The recorded per-launch DRAM traffic of a kernel, or None if its sources changed."""
    import hashlib

    rec = PROFILED_TRAFFIC[which]
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, "fp8_attention_forward_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["sha256_16"] else None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="fa8_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows)}


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The slowest rank's figure: replicas run independently and the job ends with the last."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def time_kernel(run, steps, warmup, flush):
    """Mean device time (ms) of `run()` over `steps` calls, L2 flushed before each."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.fill_(1)
        run()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush.fill_(1)
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def bench_case(case, steps, warmup, flush, fa8, num_splits=0, graph=False):
    """Kernel-only timings of one case (tensors on the GPU).  With ``graph`` the call is
    captured once in a CUDA graph and each timed step replays it, so the step's time holds
    no host-side argument marshalling (the form a serving loop runs a decode step in)."""
    splits, ws_bytes, _ = fa8.plan(case.q, case.k, case.v, cu_seqlens_q=case.cu_seqlens_q,
                                   cu_seqlens_k=case.cu_seqlens_k, block_table=case.block_table,
                                   page_size=case.page_size, num_splits=num_splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty(tuple(case.q.shape[:-1]) + (case.DV,), dtype=case.out_dtype, device="cuda")
    lse = (torch.empty((case.q.shape[0], case.Hq, case.q.shape[1]), dtype=torch.float32, device="cuda")
           if case.q.dim() == 4 else torch.empty((case.Hq, case.q.shape[0]), dtype=torch.float32, device="cuda"))

    def run():
        fa8.fwd_case(case, out=out, lse=lse, workspace=ws, num_splits=num_splits)

    step = run
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run()  # first call outside the capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        step = g.replay
    times = time_kernel(step, steps, warmup, flush)
    st = fa8.check()
    if st != fa8.FA8_SUCCESS:
        raise RuntimeError(f"device status {st}")
    # forward + combine in split mode, + the split plan kernel unless every launched split
    # fits in one wave of CTAs (then the host passes the cap and no plan kernel runs)
    launches = 1
    if splits > 1:
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        name = _decode_kernel_name(case)
        per_sm = 2 if name.startswith("decode_kernel<128,128,") else 1
        g = case.Hq // case.Hkv
        # positions per work unit: a 16-row decode tile or a 128-row tile
        pos = 16 // g if name.startswith("decode_kernel") else 128 // g
        mblocks = sum((lq + pos - 1) // pos for lq in case.seqlens_q)
        base = mblocks * case.Hkv
        launches = 2 + (1 if base * splits > per_sm * sms else 0)
    return {"ms": statistics.mean(times), "ms_min": min(times), "splits": splits,
            "launches_per_step": launches, "out": out, "lse": lse, "ws": ws}


E2E_SETS = 3  # buffer sets of the end-to-end pipeline


def bench_e2e(case, steps, warmup, flush, fa8, num_splits=0):
    """End-to-end through the public call: every step copies its inputs (Q/K/V and the small
    index tensors) from pinned host memory, runs the forward and copies O and LSE back to
    pinned host memory.  E2E_SETS buffer sets and three streams let the copies of
    neighbouring steps overlap the forward of the current one (H2D of the next steps and D2H
    of the previous ones run while step i computes), as a serving loop would; every step's copies are inside the
    timed region, which runs from the first H2D to the last D2H.  The L2 flush is issued on
    the compute stream before every forward.  Returns the pipelined and the serial time per
    step."""
    import dataclasses

    host = {}
    names = ["q", "k", "v", "descale_q", "descale_k", "descale_v", "cu_seqlens_q", "cu_seqlens_k",
             "block_table", "sink"]
    for n in names:
        t = getattr(case, n)
        if t is not None:
            host[n] = t.cpu().pin_memory()
    sets = []
    for _ in range(E2E_SETS):
        dst = {n: torch.empty_like(getattr(case, n)) for n in host}
        dcase = dataclasses.replace(case, **dst)
        out = torch.empty(tuple(dcase.q.shape[:-1]) + (dcase.DV,), dtype=dcase.out_dtype, device="cuda")
        lse = (torch.empty((dcase.q.shape[0], dcase.Hq, dcase.q.shape[1]), dtype=torch.float32, device="cuda")
               if dcase.q.dim() == 4 else torch.empty((dcase.Hq, dcase.q.shape[0]), dtype=torch.float32, device="cuda"))
        sets.append({"dst": dst, "case": dcase, "out": out, "lse": lse,
                     "out_h": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                     "lse_h": torch.empty(lse.shape, dtype=lse.dtype).pin_memory()})
    c0 = sets[0]["case"]
    splits, ws_bytes, _ = fa8.plan(c0.q, c0.k, c0.v, cu_seqlens_q=c0.cu_seqlens_q, cu_seqlens_k=c0.cu_seqlens_k,
                                   block_table=c0.block_table, page_size=c0.page_size, num_splits=num_splits)
    ws = [torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") for _ in range(E2E_SETS)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sets[0]["out"].numel() * sets[0]["out"].element_size() + sets[0]["lse"].numel() * sets[0]["lse"].element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_cmp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(n):
            S = sets[i % E2E_SETS]
            with torch.cuda.stream(s_in):
                if i >= E2E_SETS:
                    s_in.wait_event(ev_cmp[i - E2E_SETS])  # this set's inputs consumed by its last step
                for k_, t in host.items():
                    S["dst"][k_].copy_(t, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                if i >= E2E_SETS:
                    s_cmp.wait_event(ev_out[i - E2E_SETS])  # this set's outputs read back by its last step
                flush.fill_(1)
                fa8.fwd_case(S["case"], out=S["out"], lse=S["lse"], workspace=ws[i % E2E_SETS], num_splits=num_splits,
                             stream=s_cmp)
                ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                S["out_h"].copy_(S["out"], non_blocking=True)
                S["lse_h"].copy_(S["lse"], non_blocking=True)
                ev_out[i].record(s_out)
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    def serial():
        S = sets[0]
        for k_, t in host.items():
            S["dst"][k_].copy_(t, non_blocking=True)
        fa8.fwd_case(S["case"], out=S["out"], lse=S["lse"], workspace=ws[0], num_splits=num_splits)
        S["out_h"].copy_(S["out"], non_blocking=True)
        S["lse_h"].copy_(S["lse"], non_blocking=True)

    pipelined(max(warmup, 3))
    ms = pipelined(steps)
    ser = statistics.mean(time_kernel(serial, max(3, steps // 2), 3, flush))
    st = fa8.check()
    if st != fa8.FA8_SUCCESS:
        raise RuntimeError(f"device status {st}")
    return {"ms": ms, "ms_serial": ser, "h2d": h2d, "d2h": d2h}


def _row_pairs(case, rows):
    """Visible (row, key) pairs of the sampled (token, head) rows."""
    import numpy as np

    starts = np.concatenate([[0], np.cumsum(case.seqlens_q)])
    n = 0
    for tok, _ in rows:
        b = int(np.searchsorted(starts, tok, side="right") - 1)
        i = tok - starts[b]
        lq, lk = case.seqlens_q[b], case.seqlens_k[b]
        hi = lk - 1
        if case.causal:
            hi = min(hi, i + lk - lq)
        lo = 0 if case.window_left < 0 else max(0, i + lk - lq - case.window_left)
        n += max(0, hi - lo + 1)
    return n


def cpu_oracle_sample(case, budget_s=15.0, seed=0, threads=1, arrays=None):
    """Times the fp64 oracle on randomly sampled output rows of `case` until ~budget_s of
    wall time, with `threads` host threads working on independent rows (the C oracle runs
    without the interpreter lock); returns (pairs per second, rows, seconds).  The
    whole-workload time is the sampled time scaled by the workload's visible pairs."""
    import concurrent.futures as cf

    import numpy as np

    import oracle

    a = arrays if arrays is not None else oracle.problem_arrays(case)
    rng = np.random.default_rng(seed)
    per_call = 4
    pairs = 0
    rows_done = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        while time.perf_counter() - t0 < budget_s:
            batches = [[(int(rng.integers(0, case.total_q)), int(rng.integers(0, case.Hq))) for _ in range(per_call)]
                       for _ in range(threads)]
            list(ex.map(lambda r: oracle.attention_arrays(a, rows=r), batches))
            for r in batches:
                pairs += _row_pairs(case, r)
                rows_done += len(r)
    dt = time.perf_counter() - t0
    return pairs / dt, rows_done, dt


def cpu_baseline_for(case, bound, budget_s, threads):
    """The oracle's throughput on `case` in the workload's own unit (TFLOP/s or GB/s of the
    same algorithmic work the GPU figure counts), at one thread and at `threads` threads."""
    import oracle

    a = oracle.problem_arrays(case)
    out = {}
    for n in (1, threads):
        pps, rows, dt = cpu_oracle_sample(case, budget_s=budget_s, threads=n, arrays=a)
        t_full = case.pairs() / pps  # seconds for the whole workload at this rate
        if bound == "hbm":
            val, unit = inputs.algorithmic_bytes(case) / t_full / 1e9, "GB/s"
        else:
            val, unit = inputs.algorithmic_flops(case) / t_full / 1e12, "TFLOP/s"
        out["threads_1" if n == 1 else f"threads_{n}"] = {
            "value": val, "unit": unit, "cores": n, "rows": rows, "seconds": round(dt, 2),
            "whole_workload_s": t_full}
        if n == threads:
            break
    return out


def _decode_kernel_name(case):
    """The kernel include/fa8.h documents for this shape: the few-rows decode kernel when
    query positions x (Hq / Hkv) <= 16 with Hq / Hkv dividing 16 (batched q, dv % 128 = 0),
    carrying 4 or 8 rows when that product is at most 4 or 8, else 16; otherwise the persistent prefill kernel for dv <= 128 and the one-tile kernel above."""
    g = case.Hq // case.Hkv
    sq = case.seqlens_q[0]
    few = case.q_layout == "batched" and case.DV % 128 == 0 and 16 % g == 0 and sq * g <= 16
    if few:
        return f"decode_kernel<{case.D},{case.DV},{4 if sq * g <= 4 else (8 if sq * g <= 8 else 16)}>"
    return f"prefill_kernel<{case.D},{case.DV}>" if case.DV <= 128 else f"fwd_kernel<{case.D},{case.DV}>"


def decode_steps_suite(args):
    """Times every inputs.DECODE_STEP_SHAPES case (default split heuristic, L2 flushed before
    every step; the step replayed from a CUDA graph, and for comparison called directly) and
    prints one JSON line per shape."""
    import torch

    from fp8_attention_forward_gb300 import fa8

    peaks = _peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for shape in inputs.DECODE_STEP_SHAPES:
        case = inputs.decode_step(shape, device="cuda")
        r = bench_case(case, args.steps, args.warmup, flush, fa8, graph=True)
        eager = bench_case(case, args.steps, args.warmup, flush, fa8)
        nb = inputs.algorithmic_bytes(case)
        gbs = nb / (r["ms"] * 1e-3) / 1e9
        print(json.dumps({"suite": "decode-steps", "shape": shape[0], "us": r["ms"] * 1e3,
                          "us_min": r["ms_min"] * 1e3, "us_eager": eager["ms"] * 1e3,
                          "timing": "CUDA-graph replay of the step; us_eager: direct calls",
                          "splits": r["splits"],
                          "kernel": _decode_kernel_name(case),
                          "algorithmic_bytes": nb, "GB/s": gbs,
                          "frac_hbm": gbs / peaks["hbm_gbs"], "steps": args.steps,
                          "warmup": args.warmup, "l2": "256 MB buffer written before every step"}))
        del case, r, eager


WORKLOADS = [
    # (key, what, builder, bound): the five configured workloads; the tiny one is launch-bound
    # and reported for completeness only
    ("tiny_dense", "tiny dense (B=1, H=2, S=128, d=64)", lambda dev: inputs.tiny_dense().to(dev), "launch"),
    ("causal_gqa_prefill", "causal GQA prefill (B=2, Hq=32, Hkv=8, S=4096, d=dv=128)",
     lambda dev: inputs.causal_gqa_prefill("full", device=dev), "tensor"),
    ("paged_decode", "paged decode (B=64, 1 token, Hq=64, Hkv=8, keys U[1024,32768], 16-token pages)",
     lambda dev: inputs.paged_decode("full", device=dev), "hbm"),
    ("long_kv_sq1", "long-KV, 1 query row (Sk=131072, d=dv=256)", lambda dev: inputs.long_kv(1, "full", device=dev), "hbm"),
    ("long_kv_sq128", "long-KV, 128 query rows (Sk=131072, d=dv=256)",
     lambda dev: inputs.long_kv(128, "full", device=dev), "tensor"),
    ("varlen_swa_prefill", "varlen sliding-window prefill (16 seqs U[256,8192], d=192, dv=128, window 1024, sink)",
     lambda dev: inputs.varlen_swa_prefill("full", device=dev), "tensor"),
]


def _peak_clock_mhz():
    """The SM clock the measured peaks were taken at (their median under load), if recorded."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        c = d.get("clocks_under_load", {}).get("sm_mhz_median")
        return float(c) if c else None
    return None


def workload_line(key, what, case, bound, r, peaks, clk_mhz):
    """One workload's GPU figure against its roofline."""
    sec = r["ms"] * 1e-3
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    d = {"workload": key, "what": what, "kernel": _decode_kernel_name(case), "us": r["ms"] * 1e3,
         "us_min": r["ms_min"] * 1e3, "splits": r["splits"], "bound": bound}
    if bound == "hbm":
        val = inputs.algorithmic_bytes(case) / sec / 1e9
        d.update(value=val, unit="GB/s", peak=peaks["hbm_gbs"], frac=val / peaks["hbm_gbs"],
                 algorithmic_bytes=inputs.algorithmic_bytes(case))
    else:
        val = inputs.algorithmic_flops(case) / sec / 1e12
        d.update(value=val, unit="TFLOP/s", algorithmic_flops=inputs.algorithmic_flops(case))
        if bound == "tensor":
            d.update(peak=fp8_peak, frac=val / fp8_peak)
            pc = _peak_clock_mhz()
            if pc and clk_mhz:
                # the peak was measured at a lower clock under its own power draw: the same
                # fraction at this run's clock
                d["frac_at_run_clock"] = val / (fp8_peak * clk_mhz / pc)
    return d


def configs_suite(args):
    """Times the forward on every configured workload (L2 flushed before every step) and
    prints one JSON line each with its roofline fraction."""
    from fp8_attention_forward_gb300 import fa8

    peaks = _peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for key, what, make, bound in WORKLOADS:
        case = make("cuda")
        r = bench_case(case, args.steps, args.warmup, flush, fa8)
        line = workload_line(key, what, case, bound, r, peaks, None)
        line.update(suite="configs", steps=args.steps, warmup=args.warmup, l2="256 MB buffer written before every step")
        print(json.dumps(line))
        del case, r


def reference_arm(args, rank):
    """The fp64 CPU oracle (the only reference this path has) on the headline workload:
    W warm-up and K timed steps, each a bounded sample of output rows computed on all host
    cores; the value is the sample's throughput scaled to the workload's algorithmic flops."""
    if rank != 0:
        return
    import oracle

    case = inputs.causal_gqa_prefill("full", device="cpu")
    a = oracle.problem_arrays(case)
    threads = os.cpu_count() or 1
    step_s = min(5.0, max(0.5, args.cpu_budget / max(1, args.steps)))
    for _ in range(args.warmup):
        cpu_oracle_sample(case, budget_s=0.2, threads=threads, arrays=a)
    rates, rows = [], 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        pps, nr, _ = cpu_oracle_sample(case, budget_s=step_s, threads=threads, arrays=a, seed=100 + i)
        rates.append(pps)
        rows += nr
    wall = time.perf_counter() - t0
    pps = statistics.mean(rates)
    val = pps * 2.0 * (case.D + case.DV) / 1e12
    t_full = case.pairs() / pps
    sample = (f"{args.steps} steps of ~{step_s:.1f} s: {rows} random (token, head) rows of the workload on "
              f"{threads} host threads (fp64, independent rows per thread)")
    line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_full * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": HEADLINE, "impl": "fp64 CPU oracle (oracle/attn_ref.c)",
                       "ms_per_step": "the whole workload at the sampled rate"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line))


HEADLINE = "causal_gqa_prefill B=2 Hq=32 Hkv=8 Sq=Sk=4096 d=dv=128 e4m3->bf16"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fa8", choices=["fa8", "reference"])
    ap.add_argument("--no-decode", action="store_true", help="skip the paged-decode figure")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload section")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle time: the reference arm's total; per workload and thread count "
                         "in the default line, a tenth of it")
    ap.add_argument("--suite", default="", choices=["", "decode-steps", "configs"],
                    help="decode-steps: one JSON line per served-model decode step shape "
                         "(kernel time incl. the split combine); configs: one line per "
                         "configured workload with its roofline fraction; both instead of "
                         "the headline line")
    args = ap.parse_args()
    if args.suite == "decode-steps":
        return decode_steps_suite(args)
    if args.suite == "configs":
        return configs_suite(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank)
    peaks = _peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # dense FP8 = 2x dense bf16 (nominal 4.5 vs 2.25 PF)

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from fp8_attention_forward_gb300 import build as _build
    from fp8_attention_forward_gb300 import fa8

    if rank == 0:
        _build.build()
    _barrier(world)
    fa8.lib()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    prefill = inputs.causal_gqa_prefill("full", device="cuda")
    flops = inputs.algorithmic_flops(prefill)

    _barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with ClockSampler(local) as clocks:
        res = bench_case(prefill, args.steps, args.warmup, flush, fa8)
        torch.cuda.synchronize()
    _barrier(world)
    wall = time.perf_counter() - t_wall
    clk = clocks.summary()
    ms = _max_over_ranks(res["ms"], world)
    tflops_rank = flops / (ms * 1e-3) / 1e12
    value = tflops_rank * world

    e2e = bench_e2e(prefill, max(4, args.steps), max(3, args.warmup), flush, fa8)
    e2e_ms = _max_over_ranks(e2e["ms"], world)

    decode = None
    if not args.no_decode:
        dec = inputs.paged_decode("full", device="cuda")
        dbytes = inputs.algorithmic_bytes(dec)
        dres = bench_case(dec, args.steps, args.warmup, flush, fa8)
        dms = _max_over_ranks(dres["ms"], world)
        gbs = dbytes / (dms * 1e-3) / 1e9
        decode = {"workload": "paged_decode B=64 Sq=1 Hq=64 Hkv=8 d=dv=128 page=16 keys~U[1024,32768]",
                  "value": gbs * world, "unit": "GB/s", "ms_per_step": dms, "splits": dres["splits"],
                  "algorithmic_bytes": dbytes,
                  "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": gbs / peaks["hbm_gbs"], "traffic": _profiled_traffic("decode"),
                               "kernel": PROFILED_TRAFFIC["decode"]["kernel"] + " + combine_kernel",
                               "peak_source": peaks["source"] + " copy bandwidth"}}
        del dec, dres

    # every configured workload, each on its own roofline (fewer steps: a bounded section)
    configs = None
    if not args.no_configs:
        lines = []
        csteps, cwarm = max(3, min(args.steps, 10)), max(3, min(args.warmup, 3))
        with ClockSampler(local) as cclocks:
            for key, what, make, bound in WORKLOADS:
                case = make("cuda")
                r = bench_case(case, csteps, cwarm, flush, fa8)
                line = workload_line(key, what, case, bound, r, peaks, None)
                line.update(steps=csteps, warmup=cwarm)
                lines.append(line)
                del case, r
        cclk = cclocks.summary()
        pc = _peak_clock_mhz()
        for line in lines:
            if line["bound"] == "tensor" and pc and cclk.get("sm_mhz"):
                line["frac_at_run_clock"] = line["value"] / (line["peak"] * cclk["sm_mhz"] / pc)
        configs = {"steps": csteps, "warmup": cwarm, "clocks": cclk, "l2": "256 MB buffer written before every step",
                   "workloads": lines}

    cpu = None
    if rank == 0:
        threads = os.cpu_count() or 1
        budget = max(0.5, args.cpu_budget / 10.0)
        per_config = {}
        head = cpu_baseline_for(prefill.to("cpu"), "tensor", budget, threads)
        per_config["causal_gqa_prefill"] = head
        if configs is not None:
            for key, what, make, bound in WORKLOADS:
                if key in per_config:
                    continue
                ccase = make("cuda").to("cpu")  # drawn on the device (fast), read by the oracle on the host
                per_config[key] = cpu_baseline_for(ccase, "hbm" if bound == "hbm" else "tensor", budget, threads)
                del ccase
        st = head["threads_1"]
        cpu = {"value": st["value"], "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{st['rows']} random (token, head) rows of the prefill workload, {st['seconds']} s, "
                         f"single-thread fp64, scaled to the workload's algorithmic flops",
               "all_cores": head.get(f"threads_{threads}"), "host_threads": threads,
               "per_config": per_config}

    if rank == 0:
        pc = _peak_clock_mhz()
        roof = {"bound": "tensor", "achieved": tflops_rank, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": tflops_rank / fp8_peak, "traffic": _profiled_traffic("prefill"),
                "kernel": PROFILED_TRAFFIC["prefill"]["kernel"],
                "peak_source": f"{peaks['source']} bf16 burst x2 (dense FP8 = 2x bf16)"}
        if pc and clk.get("sm_mhz"):
            roof["frac_at_run_clock"] = tflops_rank / (fp8_peak * clk["sm_mhz"] / pc)
            roof["peak_clock_mhz"] = pc
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": {"workload": HEADLINE, "global_batch": 2 * world, "seq_len": 4096,
                       "parallelism": f"replicas x{world}", "l2": "256 MB buffer written before every step",
                       "flop_convention": "2*(d+dv) per unmasked (row,key) pair",
                       "algorithmic_flops": flops, "splits": res["splits"]},
            "roofline": roof,
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e_ms,
                    "mode": f"pipelined: {E2E_SETS} buffer sets, copy-in / compute / copy-out streams",
                    "ms_per_step_serial": e2e["ms_serial"]},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": clk, "decode": decode, "configs": configs, "cpu_baseline": cpu,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
