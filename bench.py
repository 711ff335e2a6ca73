"""Benchmark of the fused FP8 attention forward on one GB300 (or N replicas).

Headline: causal GQA prefill (B=2, Hq=32, Hkv=8, S=4096, d=dv=128, E4M3 in, bf16 out) in
TFLOP/s of algorithmic work (2*(d+dv) flops per unmasked (row, key) pair), against the
dense FP8 tensor peak.  The same line carries the paged decode workload (B=64, 1 token,
Hq=64, Hkv=8, d=dv=128, 16-token pages, keys ~U[1024,32768]) in GB/s against HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Timing: W untimed steps, then K steps; before every step a 256 MB buffer is written to
flush L2 (129 MB); each step's forward call is bracketed by CUDA events on the launching
stream; ms_per_step is the mean over the K steps, max over ranks.  `e2e` repeats the
measurement through the public call with the inputs copied from pinned host memory and
the output copied back inside the timed region (pipelined over two buffer sets so that the
copies of neighbouring steps overlap the forward; the serial time is reported beside it).
`--impl reference` times the fp64 CPU oracle (the only reference this path has) on a
bounded sample of the same workload.
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
    "prefill": {"kernel": "prefill_kernel<128,128>", "bytes": 68.41e6,
                "sources": ["fa8_prefill.cuh", "fa8_kernel.cuh", "fa8_ptx.cuh"], "sha256_16": "0000000000000000"},
    "decode": {"kernel": "decode_kernel<128,128>", "bytes": 2073.6e6,
               "sources": ["fa8_decode.cuh", "fa8_kernel.cuh", "fa8_ptx.cuh"], "sha256_16": "a855ada72c561ba6"},
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
        per_sm = 2 if name.startswith("decode_kernel<128,128>") else 1
        g = case.Hq // case.Hkv
        # positions per CTA: a 16-row decode tile, two 128-row tiles (prefill), or one
        pos = 16 // g if name.startswith("decode_kernel") else (2 if name.startswith("prefill") else 1) * (128 // g)
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


def cpu_oracle_sample(case, budget_s=15.0, seed=0):
    """Times the fp64 oracle (single thread) on randomly sampled output rows of `case`
    until ~budget_s of CPU work; returns (flop/s, rows, seconds)."""
    import numpy as np

    import oracle

    arrays = oracle.problem_arrays(case)
    rng = np.random.default_rng(seed)
    total_flops = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    lens_q = case.seqlens_q
    lens_k = case.seqlens_k
    starts = np.concatenate([[0], np.cumsum(lens_q)])
    while time.perf_counter() - t0 < budget_s:
        rows = []
        for _ in range(8):
            tok = int(rng.integers(0, case.total_q))
            rows.append((tok, int(rng.integers(0, case.Hq))))
        oracle.attention_arrays(arrays, rows=rows)
        for tok, _ in rows:
            b = int(np.searchsorted(starts, tok, side="right") - 1)
            i = tok - starts[b]
            lq, lk = lens_q[b], lens_k[b]
            hi = lk - 1
            if case.causal:
                hi = min(hi, i + lk - lq)
            lo = 0 if case.window_left < 0 else max(0, i + lk - lq - case.window_left)
            total_flops += 2.0 * (case.D + case.DV) * max(0, hi - lo + 1)
        rows_done += len(rows)
    dt = time.perf_counter() - t0
    return total_flops / dt, rows_done, dt


def _decode_kernel_name(case):
    """The kernel include/fa8.h documents for this shape: the few-rows decode kernel when
    query positions x (Hq / Hkv) <= 16 with Hq / Hkv dividing 16 (batched q, dv % 128 = 0);
    otherwise the two-tile prefill kernel for dv <= 128 and the one-tile kernel above."""
    g = case.Hq // case.Hkv
    sq = case.seqlens_q[0]
    few = case.q_layout == "batched" and case.DV % 128 == 0 and 16 % g == 0 and sq * g <= 16
    if few:
        return f"decode_kernel<{case.D},{case.DV}>"
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


def configs_suite(args):
    """Times the forward on every configured workload (L2 flushed before every step) and
    prints one JSON line each with its roofline fraction: tensor-bound workloads in TFLOP/s
    against the dense FP8 peak, HBM-bound ones in GB/s against the copy bandwidth."""
    import torch

    from fp8_attention_forward_gb300 import fa8

    peaks = _peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    work = [("causal GQA prefill", lambda: inputs.causal_gqa_prefill("full", device="cuda"), "tensor"),
            ("paged decode", lambda: inputs.paged_decode("full", device="cuda"), "hbm"),
            ("long-KV, 1 query row", lambda: inputs.long_kv(1, "full", device="cuda"), "hbm"),
            ("long-KV, 128 query rows", lambda: inputs.long_kv(128, "full", device="cuda"), "tensor"),
            ("varlen sliding-window prefill", lambda: inputs.varlen_swa_prefill("full", device="cuda"), "tensor")]
    for name, make, bound in work:
        case = make()
        r = bench_case(case, args.steps, args.warmup, flush, fa8)
        sec = r["ms"] * 1e-3
        if bound == "tensor":
            val, unit, peak = inputs.algorithmic_flops(case) / sec / 1e12, "TFLOP/s", fp8_peak
        else:
            val, unit, peak = inputs.algorithmic_bytes(case) / sec / 1e9, "GB/s", peaks["hbm_gbs"]
        print(json.dumps({"suite": "configs", "workload": case.name, "what": name, "us": r["ms"] * 1e3,
                          "value": val, "unit": unit, "bound": bound, "peak": peak, "frac": val / peak,
                          "splits": r["splits"], "steps": args.steps, "warmup": args.warmup,
                          "l2": "256 MB buffer written before every step"}))
        del case, r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fa8", choices=["fa8", "reference"])
    ap.add_argument("--no-decode", action="store_true", help="skip the paged-decode figure")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
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
    peaks = _peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # dense FP8 = 2x dense bf16 (nominal 4.5 vs 2.25 PF)
    workload = "causal_gqa_prefill B=2 Hq=32 Hkv=8 Sq=Sk=4096 d=dv=128 e4m3->bf16"

    if args.impl == "reference":
        if rank != 0:
            return
        case = inputs.causal_gqa_prefill("full", device="cpu")
        flops, rows, dt = cpu_oracle_sample(case, budget_s=args.cpu_budget)
        val = flops / 1e12
        sample = f"{rows} random (token, head) rows of the workload, {dt:.1f} s single-thread fp64"
        line = {"metric": METRIC, "value": val, "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": {"workload": workload, "impl": "fp64 CPU oracle (oracle/attn_ref.c)"},
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

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

    cpu = None
    if rank == 0:
        cpu_case = prefill.to("cpu")
        cflops, crows, cdt = cpu_oracle_sample(cpu_case, budget_s=args.cpu_budget)
        cpu = {"value": cflops / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{crows} random (token, head) rows of the prefill workload, {cdt:.1f} s, single-thread fp64"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": {"workload": workload, "global_batch": 2 * world, "seq_len": 4096,
                       "parallelism": f"replicas x{world}", "l2": "256 MB buffer written before every step",
                       "flop_convention": "2*(d+dv) per unmasked (row,key) pair",
                       "algorithmic_flops": flops, "splits": res["splits"]},
            "roofline": {"bound": "tensor", "achieved": tflops_rank, "peak": fp8_peak, "unit": "TFLOP/s",
                         "frac": tflops_rank / fp8_peak, "traffic": _profiled_traffic("prefill"),
                         "kernel": PROFILED_TRAFFIC["prefill"]["kernel"],
                         "peak_source": f"{peaks['source']} bf16 burst x2 (dense FP8 = 2x bf16)"},
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12 * world, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e_ms,
                    "mode": f"pipelined: {E2E_SETS} buffer sets, copy-in / compute / copy-out streams",
                    "ms_per_step_serial": e2e["ms_serial"]},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": clk, "decode": decode, "cpu_baseline": cpu, "wall_s_timed_region": wall,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
