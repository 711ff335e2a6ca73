"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

Small cases run every output row through the oracle; the full-size workloads are checked
on sampled rows, in the launch configuration the benchmark times.  Tolerances (unit-scale
V): max abs 3e-2, mean abs 4e-3, LSE abs 2e-3.  Bit-exactness is required where the
tiling is identical: paged vs contiguous K/V, and the split/combine path vs the direct
path when only the first split has keys.
"""
import dataclasses
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from fp8_attention_forward_gb300 import build, fa8, inputs
from parity_util import (LSE_ABS, MAX_ABS, MEAN_ABS, assert_parity, errors, gpu_outputs, record_margin,
                         run_gpu, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa8.lib()


# ------------------------------------------------------------------ the five workloads, small
def test_tiny_dense():
    assert_parity(inputs.tiny_dense())


def test_causal_gqa_prefill_small():
    assert_parity(inputs.causal_gqa_prefill("small"))


@pytest.mark.parametrize("splits", [2, 5])
def test_d96_split_combine(splits):
    """dv = 96: three output columns per lane in the combine kernel."""
    case = inputs.make_case(name="d96s", B=2, Hq=8, Hkv=2, D=96, DV=96, seqlens_q=[1] * 2,
                            seqlens_k=[1500, 700], kv_layout="paged", page_size=16, causal=True, seed=117)
    assert_parity(case, num_splits=splits)


@pytest.mark.parametrize("splits", [0, 1, 3, 7])
def test_paged_decode_small(splits):
    assert_parity(inputs.paged_decode("small"), num_splits=splits)


@pytest.mark.parametrize("sq", [1, 128])
@pytest.mark.parametrize("splits", [1, 0])
def test_long_kv_small(sq, splits):
    assert_parity(inputs.long_kv(sq, "small"), num_splits=splits)


def test_varlen_swa_prefill_small():
    assert_parity(inputs.varlen_swa_prefill("small"))


# ------------------------------------------------------------------ lazy rescale threshold
@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_lazy_rescale_staircase(kind):
    """Scores rising 0.5 q log2-units per 128 keys over 64 tiles, walked by one CTA (one
    split: the split heuristic would cut the staircase into short pieces): with the
    threshold 0.75 (below log2(448) - 8) no weight leaves the E4M3 range and the output
    meets the bar."""
    assert_parity(inputs.lazy_staircase(kind), num_splits=1)


def test_lazy_threshold_negative_control(tmp_path):
    """The same staircase through a build whose threshold is 4 (above log2(448) - 8): weights
    up to 2^12 saturate at 448 and the output misses the bar by a wide margin, so the
    staircase test does depend on the threshold."""
    lib = build.build(out_dir=str(tmp_path / "tau4"), defines=["FA8_TAU=4.0f"])
    out_file = tmp_path / "out.pt"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = (
        "import sys, torch\n"
        f"sys.path.insert(0, {root!r})\n"
        "from fp8_attention_forward_gb300 import fa8, inputs\n"
        "c = inputs.lazy_staircase('prefill', device='cuda')\n"
        "out, lse = fa8.fwd_case(c, num_splits=1)\n"
        "assert fa8.check() == fa8.FA8_SUCCESS\n"
        f"torch.save((out.cpu(), lse.cpu()), {str(out_file)!r})\n")
    subprocess.run([sys.executable, "-c", script], env=dict(os.environ, FA8_LIBRARY=lib),
                   check=True, timeout=600)
    out, lse = torch.load(out_file)
    case = inputs.lazy_staircase("prefill")
    o, l = gpu_outputs(case, out, lse)
    o_ref, l_ref = oracle.attention(case)
    mx, mean, le = errors(case, o, l, o_ref, l_ref)
    assert mx > 2 * MAX_ABS and mean > 2 * MEAN_ABS, (mx, mean, le)


# ------------------------------------------------------------------ feature matrix
VARIANTS = [
    dict(name="d64_causal_lq_lt_lk", B=2, Hq=4, Hkv=4, D=64, DV=64, seqlens_q=[70] * 2,
         seqlens_k=[300] * 2, causal=True, seed=101),
    dict(name="d64_causal_lq_gt_lk", B=1, Hq=2, Hkv=1, D=64, DV=64, seqlens_q=[300],
         seqlens_k=[200], causal=True, seed=102),
    dict(name="d128_noncausal_ragged", B=3, Hq=6, Hkv=2, D=128, DV=128, seqlens_q=[200] * 3,
         seqlens_k=[333] * 3, seed=103, v_dist=(0.5, 1.0)),
    dict(name="d128_gqa3_rows126", B=1, Hq=9, Hkv=3, D=128, DV=128, seqlens_q=[190],
         seqlens_k=[190], causal=True, seed=104),
    dict(name="d128_gqa16", B=2, Hq=32, Hkv=2, D=128, DV=128, seqlens_q=[20] * 2,
         seqlens_k=[500] * 2, causal=True, seed=105, descale_mode="per_bkv_uniform"),
    dict(name="d128_window_noncausal", B=1, Hq=2, Hkv=1, D=128, DV=128, seqlens_q=[260],
         seqlens_k=[400], window_left=100, seed=106),
    dict(name="d128_fp16_out", B=1, Hq=4, Hkv=2, D=128, DV=128, seqlens_q=[150],
         seqlens_k=[150], causal=True, out_dtype=torch.float16, seed=107),
    dict(name="d192_192_varlen_sink", B=3, Hq=4, Hkv=1, D=192, DV=192, seqlens_q=[90, 300, 10],
         seqlens_k=[90, 300, 10], q_layout="varlen", kv_layout="varlen", sink=True, seed=108),
    dict(name="d192_128_causal_window", B=2, Hq=4, Hkv=2, D=192, DV=128, seqlens_q=[400] * 2,
         seqlens_k=[400] * 2, causal=True, window_left=130, seed=109),
    dict(name="d256_causal", B=1, Hq=4, Hkv=2, D=256, DV=256, seqlens_q=[300], seqlens_k=[300],
         causal=True, seed=110, v_dist=(1.0, 0.1), descale_mode="tensor_amax"),
    dict(name="varlen_q_paged_kv", B=4, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[4, 1, 7, 2],
         seqlens_k=[37, 500, 129, 256], q_layout="varlen", kv_layout="paged", page_size=16,
         causal=True, seed=111, descale_mode="per_bkv_uniform"),
    dict(name="varlen_empty_seqs", B=4, Hq=4, Hkv=2, D=128, DV=128, seqlens_q=[0, 50, 0, 20],
         seqlens_k=[10, 0, 0, 200], q_layout="varlen", kv_layout="varlen", seed=112),
    dict(name="varlen_empty_seqs_sink", B=3, Hq=4, Hkv=2, D=64, DV=64, seqlens_q=[5, 30, 9],
         seqlens_k=[0, 40, 3], q_layout="varlen", kv_layout="varlen", causal=True, sink=True,
         seed=113),
]
VARIANTS += [
    dict(name="d96_causal_gqa", B=2, Hq=8, Hkv=2, D=96, DV=96, seqlens_q=[300] * 2, seqlens_k=[300] * 2,
         causal=True, descale_mode="tensor_amax", seed=114),
    dict(name="d96_decode_paged", B=3, Hq=8, Hkv=2, D=96, DV=96, seqlens_q=[1] * 3, seqlens_k=[900, 40, 2000],
         kv_layout="paged", page_size=16, causal=True, descale_mode="per_bkv_uniform", seed=115),
    dict(name="d96_varlen_window_sink_fp16", B=3, Hq=4, Hkv=4, D=96, DV=96, seqlens_q=[33, 200, 7],
         seqlens_k=[33, 200, 7], q_layout="varlen", kv_layout="varlen", causal=True, window_left=50,
         sink=True, out_dtype=torch.float16, seed=116),
]
for ps in (8, 64, 128, 256):
    VARIANTS.append(dict(name=f"paged_ps{ps}", B=3, Hq=8, Hkv=2, D=128, DV=128,
                         seqlens_q=[1] * 3, seqlens_k=[100, 700, 300], kv_layout="paged",
                         page_size=ps, causal=True, seed=120 + ps))


@pytest.mark.parametrize("spec", VARIANTS, ids=[v["name"] for v in VARIANTS])
def test_variant(spec):
    assert_parity(inputs.make_case(**spec))


def test_descale_broadcast_strides():
    """(B, Hkv) descales given as 0-stride expanded views are read in place."""
    case = inputs.make_case(name="bcast", B=2, Hq=4, Hkv=2, D=128, DV=128, seqlens_q=[64] * 2,
                            seqlens_k=[200] * 2, causal=True, seed=130)
    dq = torch.tensor(0.7).expand(2, 2)          # strides (0, 0)
    dk = torch.tensor([1.3, 0.6]).expand(2, 2)   # strides (0, 1)
    dv = torch.tensor([[1.5], [0.5]]).expand(2, 2)  # strides (1, 0)
    c = dataclasses.replace(case, descale_q=dq, descale_k=dk, descale_v=dv)
    assert dq.stride() == (0, 0) and dk.stride() == (0, 1) and dv.stride() == (1, 0)
    assert_parity(c)


# ------------------------------------------------------------------ bit-exactness
def _paged_to_contig(case):
    ks, vs = [], []
    for b, lk in enumerate(case.seqlens_k):
        pages = case.block_table[b, : (lk + case.page_size - 1) // case.page_size].long()
        ks.append(case.k.view(torch.uint8)[pages].reshape(-1, case.Hkv, case.D)[:lk])
        vs.append(case.v.view(torch.uint8)[pages].reshape(-1, case.Hkv, case.DV)[:lk])
    return dataclasses.replace(case, kv_layout="varlen", block_table=None, page_size=0,
                               k=torch.cat(ks).view(torch.float8_e4m3fn),
                               v=torch.cat(vs).view(torch.float8_e4m3fn))


@pytest.mark.parametrize("ps", [16, 64, 128])
def test_paged_bit_exact_vs_contiguous(ps):
    case = inputs.make_case(name="pg", B=3, Hq=16, Hkv=2, D=128, DV=128, seqlens_q=[1] * 3,
                            seqlens_k=[130, 1000, 555], kv_layout="paged", page_size=ps,
                            causal=True, descale_mode="per_bkv_uniform", seed=140)
    contig = _paged_to_contig(case)
    o1, l1 = run_gpu(case.to("cuda"), num_splits=1)
    o2, l2 = run_gpu(contig.to("cuda"), num_splits=1)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("splits", [1, 3], ids=["one_split", "three_splits"])
@pytest.mark.parametrize("ps", [16, 64, 128])
def test_rows128_paged_bit_exact_vs_contiguous(ps, splits):
    """The 128-row kernel (prefill, chunked prefill: more than 16 query rows per kv-head)
    reads paged K/V as page-aligned boxes and contiguous K/V as whole tiles; both land the
    same bytes in the same shared-memory tiles, so O and LSE must be bit-identical, with
    one split and with three."""
    case = inputs.make_case(name="pg128", B=2, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[200, 333],
                            seqlens_k=[600, 333], q_layout="varlen", kv_layout="paged", page_size=ps,
                            causal=True, sink=True, descale_mode="per_bkv_uniform", seed=143)
    assert max(case.seqlens_q) * case.Hq // case.Hkv > 16  # the 128-row kernel
    contig = _paged_to_contig(case)
    o1, l1 = run_gpu(case.to("cuda"), num_splits=splits)
    o2, l2 = run_gpu(contig.to("cuda"), num_splits=splits)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_split_path_bit_exact_when_one_split_has_keys():
    """Every request fits one 128-key tile: with 4 splits only split 0 has keys, and the
    combine must reproduce the direct path bit for bit (sink included)."""
    case = inputs.make_case(name="sp", B=5, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[1] * 5,
                            seqlens_k=[1, 17, 100, 128, 64], kv_layout="paged", page_size=16,
                            causal=True, sink=True, descale_mode="per_bkv_uniform", seed=141)
    c = case.to("cuda")
    o1, l1 = run_gpu(c, num_splits=1)
    o4, l4 = run_gpu(c, num_splits=4)
    assert torch.equal(o1.view(torch.int16), o4.view(torch.int16))
    assert torch.equal(l1, l4)


def test_repeat_runs_bit_identical():
    case = inputs.causal_gqa_prefill("small").to("cuda")
    o1, l1 = run_gpu(case)
    o2, l2 = run_gpu(case)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_causal_first_row_exact():
    """Lq == Lk causal: row 0 sees only key 0, P = 2^8 exactly, so O[0] = dv * V[0] rounded
    once to bf16 (the oracle's closed form, reached exactly on the GPU)."""
    case = inputs.make_case(name="row0", B=1, Hq=2, Hkv=2, D=128, DV=128, seqlens_q=[256],
                            seqlens_k=[256], causal=True, seed=142)
    out, _ = run_gpu(case.to("cuda"))
    want = case.v[0, 0].to(torch.float32).to(torch.bfloat16)
    # compared as values: a -0.0 in V may come out as +0.0 from the fp32 accumulator
    assert torch.equal(out[0, 0].cpu().float(), want.float())


# ------------------------------------------------------------------ full-size workloads (sampled)
def _full(case_fn, n_rows=48, **kw):
    case = case_fn()
    dev_case = case  # tensors already on the GPU
    out, lse = run_gpu(dev_case, **kw)
    cpu_case = case.to("cpu")
    rows = sample_rows(cpu_case, n_rows, seed=7)
    o, l = gpu_outputs(cpu_case, out, lse)
    o_ref, l_ref = oracle.attention(cpu_case, rows=rows)
    mx, mean, le = errors(cpu_case, o, l, o_ref, l_ref, rows=rows)
    record_margin(cpu_case, mx, mean, le, rows, extra="full size, sampled rows")
    assert mx <= MAX_ABS and mean <= MEAN_ABS and le <= LSE_ABS, (case.name, mx, mean, le)
    return out, lse


def test_full_causal_gqa_prefill():
    _full(lambda: inputs.causal_gqa_prefill("full", device="cuda"))


def test_full_paged_decode():
    _full(lambda: inputs.paged_decode("full", device="cuda"), n_rows=32)


@pytest.mark.parametrize("sq", [1, 128])
def test_full_long_kv_mean_preserved(sq):
    out, _ = _full(lambda: inputs.long_kv(sq, "full", device="cuda"), n_rows=8)
    # V ~ N(1, 0.1) at 131072 keys: the output mean must stay ~1 (no shrink)
    mean = float(out.float().mean())  # O carries the V descale already
    assert abs(mean - 1.0) < 0.02, mean


def test_full_long_kv_one_split_no_shrink():
    """One split over all 131072 keys (1024 tiles folded into the fp32 O)."""
    case = inputs.long_kv(1, "full", device="cuda")
    out, _ = run_gpu(case, num_splits=1)
    cpu_case = case.to("cpu")
    rows = [(0, h) for h in range(cpu_case.Hq)]
    o, l = gpu_outputs(cpu_case, out, None)
    o_ref, _ = oracle.attention(cpu_case, rows=rows)
    got = o[0]
    rel = np.sqrt(np.mean((got - o_ref) ** 2)) / np.sqrt(np.mean(o_ref ** 2))
    assert rel < 5e-3, rel  # pages report 0.12-0.17 % with two-level accumulation


def test_full_varlen_swa_prefill():
    _full(lambda: inputs.varlen_swa_prefill("full", device="cuda"))


# ------------------------------------------------------------------ device status
def test_bad_block_table_entry_reports_bounds():
    case = inputs.make_case(name="badbt", B=2, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[1] * 2,
                            seqlens_k=[300, 40], kv_layout="paged", page_size=16, causal=True,
                            seed=150)
    bt = case.block_table.clone()
    bt[0, 3] = 10 ** 6  # out of range: the kernel must read zeros and report it
    c = dataclasses.replace(case, block_table=bt).to("cuda")
    fa8.fwd_case(c)
    assert fa8.check() == fa8.FA8_ERR_DEVICE_BOUNDS
    assert fa8.check() == fa8.FA8_SUCCESS  # the status word was cleared


def test_wait_timeout_is_reported():
    fa8.set_wait_timeout_ns(200_000_000)
    try:
        assert fa8.debug_wait_probe() == fa8.FA8_ERR_DEVICE_TIMEOUT
    finally:
        fa8.set_wait_timeout_ns(2_000_000_000)
    # the context is still usable afterwards
    assert_parity(inputs.tiny_dense())


# ------------------------------------------------------------------ CUDA graph capture
def _step_128x1_1k():
    return inputs.decode_step(next(s for s in inputs.DECODE_STEP_SHAPES if s[1] == 128 and s[3] == 1024))


@pytest.mark.parametrize("make,splits", [(lambda: inputs.causal_gqa_prefill("small"), 0),
                                         (lambda: inputs.paged_decode("small"), 3),
                                         (_step_128x1_1k, 0)],
                         ids=["prefill", "decode_split3", "decode_step_plan_kernel"])
def test_graph_capture_replay_matches_direct(make, splits):
    """Launch choices depend only on shapes, so a call captured in a CUDA graph replays to
    the same bits as a direct call (workspace, outputs and inputs at fixed addresses)."""
    c = make().to("cuda")
    s, nbytes, _ = fa8.plan(c.q, c.k, c.v, cu_seqlens_q=c.cu_seqlens_q, cu_seqlens_k=c.cu_seqlens_k,
                            block_table=c.block_table, page_size=c.page_size, num_splits=splits)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    out_d, lse_d = run_gpu(c, num_splits=splits, workspace=ws)
    out = torch.empty_like(out_d)
    lse = torch.empty_like(lse_d)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fa8.fwd_case(c, out=out, lse=lse, workspace=ws, num_splits=splits)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    out.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa8.fwd_case(c, out=out, lse=lse, workspace=ws, num_splits=splits)
    g.replay()
    torch.cuda.synchronize()
    assert fa8.check() == fa8.FA8_SUCCESS
    assert torch.equal(out.view(torch.int16), out_d.view(torch.int16))
    assert torch.equal(lse, lse_d)


# ------------------------------------------------------------------ per-tile split counts
def test_split_counts_per_tile_varlen_window():
    """More launched splits than most tiles can use: every tile runs min(n, ceil(t/2))
    splits of its own key range, and the combine reads exactly those (varlen q: it finds
    each row's request by binary search)."""
    case = inputs.make_case(name="spv", B=4, Hq=8, Hkv=2, D=128, DV=128,
                            seqlens_q=[5, 300, 64, 1], seqlens_k=[900, 300, 2000, 40],
                            q_layout="varlen", kv_layout="varlen", causal=True, window_left=600,
                            sink=True, descale_mode="one", seed=151)
    assert_parity(case, num_splits=16)


@pytest.mark.parametrize("splits", [1, 3], ids=["one_split", "three_splits"])
def test_persistent_unit_stream(splits):
    """The prefill kernel is persistent: each CTA walks a list of work units and streams their
    KV tiles back to back, with a double-buffered Q, 4-deep hand-off rings and the next unit's
    QKs issued under the current unit's last tiles.  400 varlen sequences of 0-150 tokens
    (32 positions per unit, mostly one KV tile, some empty) under a causal 64-key window give
    thousands of short units per CTA, interleaved with units that have no keys in a split
    (written directly) and splits that do not run."""
    lens = inputs.uniform_lengths(400, 0, 150, seed=161)
    case = inputs.make_case(name="unit_stream", B=400, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=lens,
                            seqlens_k=lens, q_layout="varlen", kv_layout="varlen", causal=True,
                            window_left=64, sink=True, descale_mode="per_bkv_uniform", seed=161)
    from parity_util import sample_rows
    assert_parity(case, rows=sample_rows(case, 800, seed=161), num_splits=splits)


def test_split_counts_decode_wide_block_table():
    """Block tables sized for 32k keys, contexts of a few hundred to a few thousand keys: the
    default heuristic launches many splits, the short requests run few of them."""
    case = inputs.make_case(name="spw", B=3, Hq=32, Hkv=8, D=128, DV=128, seqlens_q=[1] * 3,
                            seqlens_k=[300, 4000, 17], kv_layout="paged", page_size=16,
                            table_width=2048, causal=True, descale_mode="per_bkv_uniform", seed=152)
    assert_parity(case, num_splits=0)


def test_split_path_bit_exact_when_tiles_use_one_split():
    """Key ranges of at most two 128-key tiles run one split whatever the launch: the 128-row
    kernel's split path then matches its direct path bit for bit."""
    case = inputs.make_case(name="sp1", B=2, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[200] * 2,
                            seqlens_k=[256] * 2, causal=True, sink=True, seed=153)
    c = case.to("cuda")
    o1, l1 = run_gpu(c, num_splits=1)
    o8, l8 = run_gpu(c, num_splits=8)
    assert torch.equal(o1.view(torch.int16), o8.view(torch.int16))
    assert torch.equal(l1, l8)
