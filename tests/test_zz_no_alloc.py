"""fa8_fwd_static_scratch: the forward with its split-KV partials in the library's static
device scratch instead of a caller workspace.

Each call is compared with fa8_fwd (caller workspace) on the same inputs for two calls in a
row: both run the same plan and kernels, so the outputs must be bit-identical.  The file is
named so that it is collected last, and it also passes on its own in a fresh process.
"""
import pytest
import torch

from fp8_attention_forward_gb300 import build, fa8, inputs
from parity_util import LSE_ABS, MAX_ABS, MEAN_ABS, errors, gpu_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa8.lib()


def _case_args(c):
    return dict(descale_q=c.descale_q, descale_k=c.descale_k, descale_v=c.descale_v,
                cu_seqlens_q=c.cu_seqlens_q, cu_seqlens_k=c.cu_seqlens_k, block_table=c.block_table,
                page_size=c.page_size, causal=c.causal, window_left=c.window_left, sink=c.sink,
                softmax_scale=c.softmax_scale)


def _empty_outputs(c):
    out = torch.full(tuple(c.q.shape[:-1]) + (c.DV,), float("nan"), dtype=c.out_dtype, device=c.q.device)
    if c.q.dim() == 4:
        lse = torch.full((c.q.shape[0], c.Hq, c.q.shape[1]), float("nan"), device=c.q.device)
    else:
        lse = torch.full((c.Hq, c.total_q), float("nan"), device=c.q.device)
    return out, lse


def _static(c, num_splits):
    out, lse = _empty_outputs(c)
    fa8.fwd_static_scratch(c.q, c.k, c.v, out=out, lse=lse, num_splits=num_splits, **_case_args(c))
    return out, lse


def _reference(c, num_splits):
    out, lse = fa8.fwd(c.q, c.k, c.v, num_splits=num_splits, out_dtype=c.out_dtype, **_case_args(c))
    return out, lse


def _splits(c, num_splits):
    s, nbytes, _ = fa8.plan(c.q, c.k, c.v, cu_seqlens_q=c.cu_seqlens_q, cu_seqlens_k=c.cu_seqlens_k,
                            block_table=c.block_table, page_size=c.page_size, num_splits=num_splits)
    return s, nbytes


def _assert_identical(case_cpu, got, ref):
    """fa8_fwd_static_scratch runs fa8_fwd's plan and kernels; only the partials' address
    differs, so O and LSE must be bit-identical (the parity-tolerance errors are reported
    alongside, to tell a small difference from a large one)."""
    o, l = gpu_outputs(case_cpu, *got)
    o_ref, l_ref = gpu_outputs(case_cpu, *ref)
    mx, mean, le = errors(case_cpu, o, l, o_ref, l_ref)
    same_o = torch.equal(got[0].view(torch.int16), ref[0].view(torch.int16))
    same_l = torch.equal(got[1].view(torch.int32), ref[1].view(torch.int32))
    assert same_o and same_l, (
        f"{case_cpu.name}: not bit-identical to fa8_fwd (O {same_o}, LSE {same_l}); "
        f"max {mx:.3g} mean {mean:.3g} lse {le:.3g} (bars {MAX_ABS}, {MEAN_ABS}, {LSE_ABS})")


CASES = [
    ("paged_decode", lambda: inputs.paged_decode("small"), 4),
    ("long_kv_sq128_d256", lambda: inputs.long_kv(128, "small"), 0),
    ("varlen_swa_prefill", lambda: inputs.varlen_swa_prefill("small"), 2),
    ("causal_gqa_prefill_one_split", lambda: inputs.causal_gqa_prefill("small"), 1),
]


@pytest.mark.parametrize("name,make,num_splits", CASES, ids=[c[0] for c in CASES])
def test_two_calls_match_fwd(name, make, num_splits):
    case_cpu = make()
    c = case_cpu.to("cuda")
    splits, nbytes = _splits(c, num_splits)
    if num_splits != 1:
        assert splits > 1 and 0 < nbytes <= fa8.STATIC_SCRATCH_BYTES, (splits, nbytes)
    ref = _reference(c, num_splits)
    first = _static(c, num_splits)
    second = _static(c, num_splits)
    assert fa8.check() == fa8.FA8_SUCCESS
    _assert_identical(case_cpu, first, ref)
    _assert_identical(case_cpu, second, ref)


def test_back_to_back_problems_share_the_scratch():
    """Two different split problems on one stream, one after the other: the second call
    reuses the scratch only after the first call's merge has read it."""
    a_cpu, b_cpu = inputs.paged_decode("small"), inputs.long_kv(1, "small")
    a, b = a_cpu.to("cuda"), b_cpu.to("cuda")
    ref_a, ref_b = _reference(a, 3), _reference(b, 5)
    got_a = _static(a, 3)
    got_b = _static(b, 5)
    assert fa8.check() == fa8.FA8_SUCCESS
    _assert_identical(a_cpu, got_a, ref_a)
    _assert_identical(b_cpu, got_b, ref_b)


def test_oversized_plan_is_rejected_before_launch():
    """Partials larger than the static scratch: FA8_ERR_WORKSPACE, nothing enqueued."""
    B, S, Hq, Hkv, D = 1, 4096, 32, 8, 128
    q = torch.zeros((B, S, Hq, D), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    k = torch.zeros((B, S, Hkv, D), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    v = torch.zeros((B, S, Hkv, D), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    splits, nbytes, _ = fa8.plan(q, k, v, num_splits=2)
    assert splits == 2 and nbytes > fa8.STATIC_SCRATCH_BYTES
    out = torch.full((B, S, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa8.Fa8Error) as ei:
        fa8.fwd_static_scratch(q, k, v, out=out, num_splits=2)
    assert ei.value.status == fa8.FA8_ERR_WORKSPACE
    assert "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
