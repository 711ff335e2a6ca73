"""The C ABI without a GPU: the library loads, exports every function include/fa8.h
declares, validates arguments on the host, and plans launches from shapes and the SM count
alone.  A call that would need the device fails loudly (FA8_ERR_CUDA), never silently."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from fp8_attention_forward_gb300 import build, fa8, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa8.h")
E4M3 = torch.float8_e4m3fn


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa8.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"FA8_API\s+[\w\s\*]*?\b(fa8_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa8_fwd", "fa8_fwd_workspace_size", "fa8_fwd_plan", "fa8_check", "fa8_last_error"):
        assert n in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(lib):
    exported = subprocess.run(["nm", "-D", "--defined-only", fa8.LIB_PATH], capture_output=True,
                              text=True, check=True).stdout
    dyn = {line.split()[-1] for line in exported.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in dyn]
    assert not missing, missing
    # nothing but the declared API is exported from the library's own code
    extra = sorted(n for n in dyn if n.startswith("fa8_") and n not in declared_functions())
    assert not extra, extra


def test_binding_covers_the_header(lib):
    assert set(declared_functions()) == set(fa8.SIGNATURES)
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_status_strings_and_version(lib):
    assert lib.fa8_version() == 100
    for st, word in [(0, b"success"), (1, b"invalid"), (2, b"unsupported"), (3, b"workspace"),
                     (4, b"CUDA"), (5, b"timed out"), (6, b"out of range"), (99, b"unknown")]:
        assert word in lib.fa8_status_string(st)


def test_wait_timeout_bounds(lib):
    assert lib.fa8_set_wait_timeout_ns(10) == fa8.FA8_ERR_INVALID_ARG
    assert b"timeout" in lib.fa8_last_error()
    assert lib.fa8_set_wait_timeout_ns(2_000_000_000) == fa8.FA8_SUCCESS


# ------------------------------------------------------------------ host-only planner
def qkv(B=2, Sq=333, Sk=333, Hq=32, Hkv=8, D=128, DV=128, dtype=E4M3):
    q = torch.zeros((B, Sq, Hq, D), dtype=torch.uint8).view(dtype)
    k = torch.zeros((B, Sk, Hkv, D), dtype=torch.uint8).view(dtype)
    v = torch.zeros((B, Sk, Hkv, DV), dtype=torch.uint8).view(dtype)
    return q, k, v


def plan(q, k, v, sm=152, **kw):
    return fa8.plan(q, k, v, sm_count=sm, **kw)


def test_plan_prefill_packs_gqa_rows(lib):
    # G = 4 q-heads per kv-head -> 32 positions x 4 heads per 128-row tile (one work unit of
    # the persistent prefill kernel); 2048 units > 8 per SM, so no split
    splits, ws, grid = plan(*qkv(B=2, Sq=4096, Sk=4096))
    assert splits == 1 and ws == 0
    assert grid == (2 * (4096 // 32), 8)
    # d = 256 (dv > 128) keeps the one-tile kernel: 32 positions per CTA
    assert plan(*qkv(B=2, Sq=4096, Sk=4096, D=256, DV=256))[2] == (2 * (4096 // 32), 8)


def test_plan_decode_splits_and_workspace(lib):
    B, Hq, Hkv, D = 64, 64, 8, 128
    q = torch.zeros((B, 1, Hq, D), dtype=torch.uint8).view(E4M3)
    kp = torch.zeros((4096, 16, Hkv, D), dtype=torch.uint8).view(E4M3)
    bt = torch.zeros((B, 2048), dtype=torch.int32)
    cu = torch.zeros((B + 1,), dtype=torch.int32)
    splits, ws, grid = plan(q, kp, kp, cu_seqlens_k=cu, block_table=bt, page_size=16)
    # decode kernel (8 rows per kv-head): 64 requests x 8 kv-heads = 512 CTAs < 8 x 152,
    # split 3 ways
    assert splits == 3
    rows = B * Hq * splits
    o_bytes = (rows * D * 4 + 255) // 256 * 256
    # partials, then 256 bytes where the forward kernel records its split cap
    assert ws == o_bytes + (rows * 4 + 255) // 256 * 256 + 256
    assert grid == (B, Hkv * splits)
    # an explicit split count is capped by the number of key tiles
    s2, _, _ = plan(q, kp, kp, cu_seqlens_k=cu, block_table=bt, page_size=16, num_splits=4096)
    assert s2 == 2048 * 16 // 128
    # and 1 disables splitting
    assert plan(q, kp, kp, cu_seqlens_k=cu, block_table=bt, page_size=16, num_splits=1)[0] == 1


def test_plan_depends_on_sm_count_only_through_the_split_heuristic(lib):
    q, k, v = qkv(B=1, Sq=1, Sk=65536, Hq=8, Hkv=1, D=256, DV=256)
    a = plan(q, k, v, sm=152)
    b = plan(q, k, v, sm=76)
    assert a[2][0] == b[2][0] == 1
    # decode kernel (one CTA per SM at d = 256), one (tile, kv-head) pair: as many splits as
    # fit one wave of CTAs, capped at 128 for the decode kernel (152 SMs) and 76 on 76 SMs
    assert a[0] == 128 and b[0] == 76
    c = plan(*qkv(B=1, Sq=1, Sk=1024, Hq=8, Hkv=1, D=256, DV=256), sm=152)
    assert c[0] == 4  # 8 key tiles -> at most half as many splits


def _dense_split_count(B, Sq, Sk, Hq, Hkv, D, DV, sm):
    """The planner's split count for dense K/V and batched q, restated: the heuristic (one
    wave of splits for few (tile, kv-head) pairs, else about eight waves), then, when the
    launch spans more than a wave, the host-chosen cap (the plan kernel's model with the
    one-wave candidate) and only the splits that run."""
    import math
    import numpy as np
    G = Hq // Hkv
    decode = DV % 128 == 0 and 16 % G == 0 and Sq * G <= 16
    P = 16 // G if decode else 128 // G
    per_sm = {(128, 128): 2}.get((D, DV), 1) if decode else 1
    slots = per_sm * sm
    mb = math.ceil(Sq / P)
    base = B * mb * Hkv
    t = math.ceil(Sk / 128)
    max_tiles = max(1, t)
    target = 8 * sm
    if base >= target or max_tiles < 4:
        return 1
    s = slots // base if 2 * base <= slots else math.ceil(target / base)
    s = max(1, min(s, max_tiles // 2, 128 if decode else 64))
    if s == 1 or base * s <= slots:
        return s
    f32 = np.float32
    F, BETA = f32(3.0), f32(0.4)
    t_fine = max(2, math.ceil(t / s))
    tiles = f32(B * t * mb)

    def cost(T):
        units = f32(B * mb * math.ceil(t / T)) * f32(Hkv)
        tail = F + f32(min(T, t))
        return tail if units <= f32(slots) else (F * units + tiles * f32(Hkv)) * (f32(1) / f32(slots)) + BETA * tail

    best, cap = f32(3.0e38), t_fine
    for T in [2 << c for c in range(9)] + [t_fine]:
        if T >= t_fine and cost(T) < best:
            best, cap = cost(T), T
    per_split = B * mb * Hkv
    if per_split <= slots:
        k = slots // per_split
        T = max(t_fine, math.ceil(t / k))
        if cost(T) < best:
            cap = T
    return max(1, min(s, math.ceil(t / cap)))


@pytest.mark.parametrize("shape", [
    (1, 64, 65536, 8, 1, 256, 256),     # four tile pairs: one wave of splits
    (1, 128, 131072, 8, 1, 256, 256),   # the long-KV 128-row workload: 19 splits
    (4, 512, 65536, 16, 2, 128, 128),   # 256 tile pairs: heuristic 5 splits, host cap
    (2, 1000, 40000, 32, 8, 192, 128),  # ragged last tile, d = 192
    (3, 2, 70000, 16, 2, 128, 128),     # decode kernel, two query tokens
    (8, 1, 300000, 64, 8, 128, 128),    # decode kernel, long keys, 64 tile pairs
    (30, 1, 9000, 32, 4, 256, 256),     # decode kernel at d = 256, 120 tile pairs
])
@pytest.mark.parametrize("sm", [152, 76, 148])
def test_plan_dense_split_count_follows_the_model(lib, shape, sm):
    B, Sq, Sk, Hq, Hkv, D, DV = shape
    s, _, _ = plan(*qkv(B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, D=D, DV=DV), sm=sm)
    assert s == _dense_split_count(B, Sq, Sk, Hq, Hkv, D, DV, sm)


def test_plan_128_row_kernel_split_cap(lib):
    # 128-row kernels (Sq x G > 16): at most 64 splits; both the prefill kernel (dv <= 128)
    # and the one-tile kernel (dv > 128) take 16 positions x 8 heads per tile.  Four (tile,
    # kv-head) pairs: as many splits as fit one wave of 152 CTAs, 38 (no plan kernel)
    q, k, v = qkv(B=1, Sq=64, Sk=65536, Hq=8, Hkv=1, D=128, DV=128)
    s, _, grid = plan(q, k, v, sm=152)
    assert grid[0] == 4 and s == 38
    q, k, v = qkv(B=1, Sq=64, Sk=65536, Hq=8, Hkv=1, D=256, DV=256)
    s, _, grid = plan(q, k, v, sm=152)
    assert grid[0] == 4 and s == 38
    # an explicit split count is kept (the host still picks the cap: no plan kernel)
    assert plan(q, k, v, sm=152, num_splits=64)[0] == 64


def test_plan_decode_rows_per_tile(lib):
    # Sq x G <= 16 with G dividing 16: one 16-row slot per request and kv-head
    q, k, v = qkv(B=3, Sq=2, Sk=4096, Hq=16, Hkv=2, D=128, DV=128)
    assert plan(q, k, v, num_splits=1)[2] == (3, 2)
    # G = 3 does not divide 16: the 128-row kernel (42 positions per tile)
    q, k, v = qkv(B=3, Sq=2, Sk=4096, Hq=6, Hkv=2, D=128, DV=128)
    assert plan(q, k, v, num_splits=1)[2] == (3, 2)
    # 4 tokens x G = 8 = 32 rows: the 128-row kernel (16 positions per tile, one tile)
    q, k, v = qkv(B=3, Sq=4, Sk=4096, Hq=16, Hkv=2, D=128, DV=128)
    assert plan(q, k, v, num_splits=1)[2] == (3, 2)


def test_plan_varlen_slots(lib):
    q = torch.zeros((1000, 16, 192), dtype=torch.uint8).view(E4M3)
    k = torch.zeros((3000, 4, 192), dtype=torch.uint8).view(E4M3)
    v = torch.zeros((3000, 4, 128), dtype=torch.uint8).view(E4M3)
    cu = torch.tensor([0, 100, 1000], dtype=torch.int32)
    cuk = torch.tensor([0, 1000, 3000], dtype=torch.int32)
    splits, ws, grid = plan(q, k, v, cu_seqlens_q=cu, cu_seqlens_k=cuk)
    # 32 positions (x 4 q-heads) per prefill work unit; one extra slot per request for slots
    # that straddle requests
    assert grid == ((1000 + 31) // 32 + 2, 4 * splits)


@pytest.mark.parametrize("mutate,status,needle", [
    (lambda q, k, v: (q.view(torch.uint8).view(torch.float8_e5m2), k.view(torch.uint8).view(torch.float8_e5m2),
                      v.view(torch.uint8).view(torch.float8_e5m2)), 2, "E5M2"),
    (lambda q, k, v: (q, k, v.view(torch.uint8).view(torch.float8_e5m2)), 2, "E5M2"),
    (lambda q, k, v: (q.view(torch.uint8).view(torch.bfloat16), k.view(torch.uint8).view(torch.bfloat16),
                      v.view(torch.uint8).view(torch.bfloat16)), 2, "E4M3"),
    (lambda q, k, v: (q[..., :80], k[..., :80], v[..., :80]), 2, "not supported"),
    (lambda q, k, v: (q[:, :, :30], k, v), 1, "multiple of kv heads"),
    (lambda q, k, v: (q, k[:1], v[:1]), 1, "batch"),
    (lambda q, k, v: (q, k, v[:, :5]), 1, "leading shapes"),
    (lambda q, k, v: (q[..., 8:], k[..., 8:], v[..., 8:]), 1, None),  # misaligned (and d=120)
])
def test_plan_rejects_bad_shapes(lib, mutate, status, needle):
    q, k, v = mutate(*qkv())
    with pytest.raises(fa8.Fa8Error) as ei:
        plan(q, k, v)
    assert ei.value.status in (status, 1, 2)
    assert ei.value.status == status or needle is None
    if needle:
        assert needle in str(ei.value)


def test_paged_plan_validation(lib):
    q = torch.zeros((2, 1, 8, 128), dtype=torch.uint8).view(E4M3)
    kp = torch.zeros((64, 16, 2, 128), dtype=torch.uint8).view(E4M3)
    cu = torch.zeros((3,), dtype=torch.int32)
    bt = torch.zeros((2, 8), dtype=torch.int32)
    with pytest.raises(fa8.Fa8Error, match="page_size"):
        plan(q, kp, kp, cu_seqlens_k=cu, block_table=bt, page_size=32)
    with pytest.raises(fa8.Fa8Error, match="cu_seqlens_k"):
        plan(q, kp, kp, block_table=bt, page_size=16)
    with pytest.raises(fa8.Fa8Error, match="block_table rows"):
        plan(q, kp, kp, cu_seqlens_k=cu, block_table=bt[:1], page_size=16)
    kp12 = torch.zeros((64, 12, 2, 128), dtype=torch.uint8).view(E4M3)
    with pytest.raises(fa8.Fa8Error, match="multiple of 8"):
        plan(q, kp12, kp12, cu_seqlens_k=cu, block_table=bt, page_size=12)


# ------------------------------------------------------------------ no silent CPU path
def test_forward_without_a_device_fails_loudly(lib):
    if torch.cuda.is_available():
        pytest.skip("checks the behaviour without a CUDA device")
    q, k, v = qkv(B=1, Sq=8, Sk=8, Hq=2, Hkv=2)
    out = torch.zeros((1, 8, 2, 128), dtype=torch.bfloat16)
    with pytest.raises(fa8.Fa8Error) as ei:
        fa8.fwd(q, k, v, out=out, workspace=torch.zeros(16, dtype=torch.uint8))
    assert ei.value.status == fa8.FA8_ERR_CUDA
    assert bool((out == 0).all())


def test_forward_validates_before_touching_the_device(lib):
    q, k, v = qkv(B=1, Sq=8, Sk=8, Hq=2, Hkv=2)
    out = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16)  # wrong dv
    with pytest.raises(fa8.Fa8Error) as ei:
        fa8.fwd(q, k, v, out=out, workspace=torch.zeros(16, dtype=torch.uint8))
    assert ei.value.status == fa8.FA8_ERR_INVALID_ARG and "dv" in str(ei.value)
    out = torch.zeros((1, 8, 2, 128), dtype=torch.float32)
    with pytest.raises(fa8.Fa8Error, match="bf16 or fp16"):
        fa8.fwd(q, k, v, out=out, workspace=torch.zeros(16, dtype=torch.uint8))


def test_decode_step_shapes_use_the_decode_kernel(lib):
    # every served-model decode step shape has <= 16 rows per kv-head: one decode-kernel slot
    # per request and kv-head, whatever the block table width (zero tensors of the shapes)
    for name, reqs, sq, ctx, hq, hkv, ps in inputs.DECODE_STEP_SHAPES:
        g = hq // hkv
        assert 16 % g == 0 and sq * g <= 16, name
        q = torch.zeros((reqs, sq, hq, 128), dtype=torch.uint8).view(E4M3)
        kp = torch.zeros((reqs * ctx // ps, ps, hkv, 128), dtype=torch.uint8).view(E4M3)
        bt = torch.zeros((reqs, 32768 // ps), dtype=torch.int32)
        cu = torch.zeros((reqs + 1,), dtype=torch.int32)
        s, _, grid = plan(q, kp, kp, cu_seqlens_k=cu, block_table=bt, page_size=ps, num_splits=1)
        assert s == 1 and grid == (reqs, hkv), name


def test_static_scratch_size_matches_the_header():
    """The binding's size limit for fa8_fwd_static_scratch is the header's."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+FA8_STATIC_SCRATCH_BYTES\s+\(\(size_t\)\s*(\d+)\s*\*\s*(\d+)\s*\*\s*(\d+)\)", text)
    assert m, "FA8_STATIC_SCRATCH_BYTES not found in include/fa8.h"
    a, b, c = (int(x) for x in m.groups())
    assert a * b * c == fa8.STATIC_SCRATCH_BYTES


def test_settings_from_many_threads_keep_plans_consistent(lib):
    """fa8_set_decode_kernel and fa8_set_wait_timeout_ns are process-wide and may be called
    from any host thread while others plan: every plan is one of the two valid ones (decode
    kernel on: up to 128 splits; off: the 128-row kernel's 64), never a mix."""
    import threading

    q, k, v = qkv(B=8, Sq=1, Sk=32768, Hq=16, Hkv=2)
    # the split heuristic caps the decode kernel at 128 splits, the 128-row kernel at 64
    on = fa8.plan(q, k, v, sm_count=152, num_splits=0)
    fa8.set_decode_kernel(False)
    off = fa8.plan(q, k, v, sm_count=152, num_splits=0)
    fa8.set_decode_kernel(True)
    assert on != off
    bad, stop = [], threading.Event()

    def toggler(i):
        n = 0
        while not stop.is_set():
            fa8.set_decode_kernel(n % 2 == 0)
            lib.fa8_set_wait_timeout_ns(1_000_000 + 1000 * i + n)
            n += 1

    def planner():
        for _ in range(300):
            got = fa8.plan(q, k, v, sm_count=152, num_splits=0)
            if got not in (on, off):
                bad.append(got)

    ts = [threading.Thread(target=toggler, args=(i,)) for i in range(2)]
    ps = [threading.Thread(target=planner) for _ in range(4)]
    for t in ts + ps:
        t.start()
    for t in ps:
        t.join()
    stop.set()
    for t in ts:
        t.join()
    fa8.set_decode_kernel(True)
    assert lib.fa8_set_wait_timeout_ns(2_000_000_000) == fa8.FA8_SUCCESS
    assert not bad, bad[:3]
