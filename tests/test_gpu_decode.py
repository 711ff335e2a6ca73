"""GPU parity of the decode kernel (batched q with at most 16 query rows per kv-head: keys on
the MMA's M dimension, query rows on N) against the fp64 oracle, and of the 128-row kernel on
the same shapes with the decode kernel switched off."""
import pytest
import torch

import oracle
from fp8_attention_forward_gb300 import build, fa8, inputs
from parity_util import assert_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa8.lib()
    yield
    fa8.set_decode_kernel(True)


DECODE = [
    # (name, kwargs): Hq / Hkv divides 16; shapes with Sq * (Hq / Hkv) <= 16 run the decode
    # kernel, the others (marked below) the 128-row kernel either way
    ("g8_paged16_causal", dict(B=4, Hq=16, Hkv=2, D=128, DV=128, seqlens_q=[1] * 4,
                               seqlens_k=[1, 129, 700, 2000], kv_layout="paged", page_size=16,
                               causal=True, descale_mode="per_bkv_uniform", seed=301)),
    ("g16_contig", dict(B=2, Hq=16, Hkv=1, D=128, DV=128, seqlens_q=[1] * 2, seqlens_k=[300] * 2,
                        causal=False, seed=302)),
    ("g1_mha_sq16_causal", dict(B=2, Hq=3, Hkv=3, D=128, DV=128, seqlens_q=[16] * 2,
                                seqlens_k=[500] * 2, causal=True, seed=303)),
    ("g4_sq4_causal_window", dict(B=3, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[4] * 3,
                                  seqlens_k=[1000] * 3, causal=True, window_left=200, seed=304)),
    ("g2_sq8_sink_fp16", dict(B=2, Hq=4, Hkv=2, D=128, DV=128, seqlens_q=[8] * 2,
                              seqlens_k=[257] * 2, causal=True, sink=True, out_dtype=torch.float16,
                              seed=305)),
    ("g8_d192_128_varlen_kv", dict(B=3, Hq=16, Hkv=2, D=192, DV=128, seqlens_q=[1] * 3,
                                   seqlens_k=[5, 400, 900], kv_layout="varlen", causal=True, seed=306)),
    ("g8_d256_paged64", dict(B=2, Hq=8, Hkv=1, D=256, DV=256, seqlens_q=[1] * 2,
                             seqlens_k=[1500, 64], kv_layout="paged", page_size=64, causal=True,
                             descale_mode="tensor_amax", seed=307)),
    ("g8_empty_kv", dict(B=3, Hq=8, Hkv=1, D=128, DV=128, seqlens_q=[1] * 3, seqlens_k=[0, 50, 0],
                         kv_layout="varlen", causal=True, sink=True, seed=308)),
    # tiles whose real rows (positions x q-heads per kv-head) fit in 4 or 8: the softmax and
    # fold carry 4 or 8 rows, with one or two query positions per tile
    ("g1_sq1_four_rows_carried", dict(B=3, Hq=2, Hkv=2, D=128, DV=128, seqlens_q=[1] * 3,
                                      seqlens_k=[90, 1, 1100], kv_layout="paged", page_size=16,
                                      causal=True, descale_mode="per_bkv_uniform", seed=318)),
    ("g2_sq2_four_rows_two_positions", dict(B=2, Hq=4, Hkv=2, D=128, DV=128, seqlens_q=[2] * 2,
                                            seqlens_k=[2, 777], kv_layout="varlen", causal=True,
                                            sink=True, seed=319)),
    ("g4_sq2_eight_rows_two_positions", dict(B=3, Hq=8, Hkv=2, D=128, DV=128, seqlens_q=[2] * 3,
                                             seqlens_k=[130, 640, 1], kv_layout="paged", page_size=16,
                                             causal=True, window_left=100, seed=320)),
    ("g2_sq1_d256_four_rows", dict(B=2, Hq=4, Hkv=2, D=256, DV=256, seqlens_q=[1] * 2,
                                   seqlens_k=[333, 1800], kv_layout="varlen", causal=False,
                                   descale_mode="tensor_amax", seed=321)),
    # more than 16 rows per kv-head (4 tokens x G 8, 8 x 8, 3 x 8): the 128-row kernel in
    # both runs, with causal masking across the tokens
    ("g8_sq4_two_slots", dict(B=3, Hq=16, Hkv=2, D=128, DV=128, seqlens_q=[4] * 3,
                              seqlens_k=[40, 700, 1300], kv_layout="paged", page_size=16,
                              causal=True, descale_mode="per_bkv_uniform", seed=315)),
    ("g8_sq8_four_slots_window_sink", dict(B=2, Hq=8, Hkv=1, D=128, DV=128, seqlens_q=[8] * 2,
                                           seqlens_k=[600, 2000], kv_layout="paged", page_size=16,
                                           causal=True, window_left=300, sink=True, seed=316)),
    ("g8_sq3_ragged_slot_d256", dict(B=2, Hq=8, Hkv=1, D=256, DV=256, seqlens_q=[3] * 2,
                                     seqlens_k=[3, 900], kv_layout="varlen", causal=True, seed=317)),
    # four query tokens per request, GQA 32/8, 64-token pages in a table as wide as 32k keys
    ("g4_sq4_paged64_wide_table", dict(B=3, Hq=32, Hkv=8, D=128, DV=128, seqlens_q=[4] * 3,
                                       seqlens_k=[700, 64, 1000], kv_layout="paged", page_size=64,
                                       table_width=512, causal=True, descale_mode="per_bkv_uniform",
                                       seed=309)),
]


def _case(kw, name):
    return inputs.make_case(name=name, **kw)


@pytest.mark.parametrize("name,kw", DECODE, ids=[d[0] for d in DECODE])
@pytest.mark.parametrize("decode_kernel", [True, False], ids=["decode", "rows128"])
def test_decode_shapes(name, kw, decode_kernel):
    case = _case(kw, name)
    fa8.set_decode_kernel(decode_kernel)
    try:
        assert_parity(case)
    finally:
        fa8.set_decode_kernel(True)


@pytest.mark.parametrize("splits", [1, 2, 5, 16])
def test_decode_splits(splits):
    case = _case(DECODE[0][1], "splits")
    assert_parity(case, num_splits=splits)


def test_decode_plan_uses_one_slot_per_request():
    case = _case(DECODE[0][1], "plan").to("cuda")
    s, _, grid = fa8.plan(case.q, case.k, case.v, cu_seqlens_k=case.cu_seqlens_k,
                          block_table=case.block_table, page_size=case.page_size, num_splits=1,
                          sm_count=152)
    assert grid == (case.B, case.Hkv)


@pytest.mark.parametrize("ps", [16, 128])
def test_decode_paged_bit_exact_vs_contiguous(ps):
    case = inputs.make_case(name="dpg", B=3, Hq=16, Hkv=2, D=128, DV=128, seqlens_q=[1] * 3,
                            seqlens_k=[130, 1000, 555], kv_layout="paged", page_size=ps,
                            causal=True, descale_mode="per_bkv_uniform", seed=310)
    from test_gpu_parity import _paged_to_contig
    contig = _paged_to_contig(case)
    o1, l1 = run_gpu(case.to("cuda"), num_splits=1)
    o2, l2 = run_gpu(contig.to("cuda"), num_splits=1)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_decode_split_bit_exact_when_one_split_has_keys():
    case = inputs.make_case(name="dsp", B=5, Hq=16, Hkv=2, D=128, DV=128, seqlens_q=[1] * 5,
                            seqlens_k=[1, 17, 100, 128, 64], kv_layout="paged", page_size=16,
                            causal=True, sink=True, descale_mode="per_bkv_uniform", seed=311)
    c = case.to("cuda")
    o1, l1 = run_gpu(c, num_splits=1)
    o4, l4 = run_gpu(c, num_splits=4)
    assert torch.equal(o1.view(torch.int16), o4.view(torch.int16))
    assert torch.equal(l1, l4)


def _model_cap(lens, Hkv, n, slots, lens_q=None, P=1):
    """The split cap the plan kernel should choose (the model restated on the host)."""
    import math
    F, BETA = 3.0, 0.4
    t = [math.ceil(x / 128) if x > 0 else 0 for x in lens]
    mb = [math.ceil(x / P) if x > 0 else 0 for x in (lens_q or [1] * len(lens))]
    t_max = max(t)
    fine = max(2, math.ceil(t_max / n))
    tiles = sum(a * b for a, b in zip(t, mb))
    best = None
    for T in [2 << c for c in range(9)] + [fine]:
        if T < fine:
            continue
        units = Hkv * sum(b * math.ceil(a / T) for a, b in zip(t, mb))
        tail = F + min(T, t_max)
        m = tail if units <= slots else (F * units + tiles * Hkv) / slots + BETA * tail
        if best is None or m < best[0]:
            best = (m, T)
    return best[1]


# (batches with more (request, kv-head) pairs than half a wave of decode CTAs: fewer launch
# as many splits as fit one wave, with the finest cap and no plan kernel)
@pytest.mark.parametrize("B,ctx,hq,hkv", [(32, 2048, 32, 8), (24, 16384, 32, 8), (96, 4096, 16, 2),
                                           (80, 32768, 16, 2), (40, None, 32, 8)])
def test_split_cap_follows_the_key_counts(B, ctx, hq, hkv):
    """The plan kernel's cap (left in the workspace) is the model's choice for these lengths,
    and the result still matches the oracle."""
    lens = [ctx] * B if ctx else inputs.uniform_lengths(B, 1024, 32768, seed=314)
    case = inputs.make_case(name="cap", B=B, Hq=hq, Hkv=hkv, D=128, DV=128, seqlens_q=[1] * B,
                            seqlens_k=lens, kv_layout="paged", page_size=16, table_width=2048,
                            causal=True, descale_mode="per_bkv_uniform", seed=314)
    c = case.to("cuda")
    splits, ws_bytes, _ = fa8.plan(c.q, c.k, c.v, cu_seqlens_k=c.cu_seqlens_k, block_table=c.block_table,
                                   page_size=c.page_size)
    slots = 2 * torch.cuda.get_device_properties(0).multi_processor_count  # two decode CTAs per SM
    if splits == 1 or B * hkv * splits <= slots:
        pytest.skip("this launch takes no plan kernel")
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    run_gpu(c, workspace=ws)
    cap = int(ws[ws_bytes - 256:ws_bytes - 252].view(torch.int32).item())
    assert cap == _model_cap(lens, hkv, splits, slots)
    rows = [(i, h) for i in range(B) for h in (0, hq - 1)]
    assert_parity(case, rows=rows)


@pytest.mark.parametrize("splits", [0, 1], ids=["heuristic_splits", "one_split"])
@pytest.mark.parametrize("decode_kernel", [True, False], ids=["decode", "rows128"])
def test_short_context_stress(decode_kernel, splits):
    """1024 one-token requests with 1-700 keys and per-(request, kv-head) descales ~U[0.5, 2]:
    short, peaked rows where a few keys carry most of the softmax mass, so one E4M3 term per
    weight (up to 2^-4 relative rounding) is not enough for the stated bar.  Both kernels must
    meet it on 600 sampled rows (the decode kernel with two P terms on every tile, the 128-row
    kernel with two terms wherever one key dominates its row's mass so far)."""
    lens = inputs.uniform_lengths(1024, 1, 700, seed=313)
    case = inputs.make_case(name="short_context_stress", B=1024, Hq=8, Hkv=2, D=128, DV=128,
                            seqlens_q=[1] * 1024, seqlens_k=lens, kv_layout="paged", page_size=16,
                            causal=True, descale_mode="per_bkv_uniform", seed=313)
    from parity_util import sample_rows
    rows = sample_rows(case, 600, seed=313)
    fa8.set_decode_kernel(decode_kernel)
    try:
        assert_parity(case, rows=rows, num_splits=splits)
    finally:
        fa8.set_decode_kernel(True)
