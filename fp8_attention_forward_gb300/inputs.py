"""Seeded synthetic workloads for the fused FP8 attention forward.

This module only *draws* inputs: Gaussian values, their E4M3 quantisation (the job of
whatever produces Q/K/V upstream of attention, not of attention itself), sequence
lengths, a shared page pool with its block table, descales and sink logits.  It holds
none of the attention arithmetic.  The CUDA path and the fp64 oracle both consume
exactly what it returns, so neither side ever sees inputs produced by the other.

Shapes, distributions and structure follow the five workloads the pages use for this
path (causal GQA prefill, paged decode with 16-token pages, long-KV with nonzero-mean
V, varlen sliding-window prefill with a learnable sink).  Quantisation with a
per-tensor descale of amax/448 follows the FP8 block-quantisation formula of the
FlashAttention-3 guide (section "Low-Precision FP8 Attention with Block Scaling"),
applied here with the whole tensor as one block.

Small tensors (lengths, page permutations, descales, sinks, and every tensor of a case
built on the CPU) are drawn from a CPU ``torch.Generator``; the large Q/K/V payloads of
a case built directly on a CUDA device are drawn from a CUDA generator seeded from the
same seed, so a case is reproducible on a given device type.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

E4M3_MAX = 448.0  # largest finite E4M3 magnitude (1.75 * 2**8)

LAYOUTS = ("batched", "varlen", "paged")


@dataclasses.dataclass
class Case:
    """One attention problem.

    Layouts (last dim contiguous everywhere):
      batched: q (B,Sq,Hq,D), k (B,Sk,Hkv,D), v (B,Sk,Hkv,DV)
      varlen : q (total_q,Hq,D), k (total_k,Hkv,D), v (total_k,Hkv,DV) + cu_seqlens_q/k
      paged  : q batched or varlen; k (num_pages,page_size,Hkv,D), v (...,DV),
               block_table (B,max_pages) int32, per-request key lengths in cu_seqlens_k
    """

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    DV: int
    seqlens_q: list
    seqlens_k: list
    q_layout: str  # "batched" | "varlen"
    kv_layout: str  # "batched" | "varlen" | "paged"
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    descale_q: Optional[torch.Tensor] = None
    descale_k: Optional[torch.Tensor] = None
    descale_v: Optional[torch.Tensor] = None
    cu_seqlens_q: Optional[torch.Tensor] = None
    cu_seqlens_k: Optional[torch.Tensor] = None
    block_table: Optional[torch.Tensor] = None
    page_size: int = 0
    causal: bool = False
    window_left: int = -1
    sink: Optional[torch.Tensor] = None
    softmax_scale: float = 0.0
    out_dtype: torch.dtype = torch.bfloat16

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.seqlens_k))

    def pairs(self) -> int:
        """Number of (query row, key) pairs that survive the mask, over all heads."""
        n = 0
        for lq, lk in zip(self.seqlens_q, self.seqlens_k):
            n += _visible_pairs(lq, lk, self.causal, self.window_left)
        return n * self.Hq

    def to(self, device) -> "Case":
        out = dataclasses.replace(self)
        for f in dataclasses.fields(self):
            val = getattr(self, f.name)
            if isinstance(val, torch.Tensor):
                setattr(out, f.name, val.to(device))
        return out


def _visible_pairs(lq: int, lk: int, causal: bool, window_left: int) -> int:
    """Counts pairs (i, j) with 0<=i<lq, 0<=j<lk, bottom-right causal / left window."""
    delta = lk - lq
    total = 0
    if not causal and window_left < 0:
        return lq * lk
    # closed-form sum over rows would be faster, but lengths here are <= a few 1e5
    import numpy as np

    i = np.arange(lq, dtype=np.int64)
    hi = np.full(lq, lk - 1, dtype=np.int64)
    if causal:
        hi = np.minimum(hi, i + delta)
    lo = np.zeros(lq, dtype=np.int64)
    if window_left >= 0:
        lo = np.maximum(lo, i + delta - window_left)
    cnt = np.clip(hi - lo + 1, 0, None)
    total = int(cnt.sum())
    return total


def quantise_e4m3(x: torch.Tensor, descale: Optional[torch.Tensor]) -> torch.Tensor:
    """x / descale, saturated to +-448, rounded to E4M3 by torch's cast (RNE).

    ``descale`` is a 0-d tensor or broadcastable to ``x``.
    """
    y = x if descale is None else x / descale
    return y.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)


def _randn(shape, gen_cpu: torch.Generator, device, seed: int, slot: int, mean=0.0, std=1.0,
           chunk_elems: int = 1 << 27) -> torch.Tensor:
    """Gaussian fp32 tensor; drawn on ``device`` with a generator seeded (seed, slot)."""
    device = torch.device(device)
    if device.type == "cpu":
        t = torch.randn(shape, generator=gen_cpu, dtype=torch.float32)
    else:
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + slot)
        t = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def _quantised_payload(shape, gen_cpu, device, seed, slot, mean, std, descale_mode):
    """Draws N(mean,std) and quantises to E4M3; returns (codes, per-tensor descale or None).

    Large payloads are drawn and cast in slices along dim 0 so fp32 temporaries stay small.
    """
    device = torch.device(device)
    n0 = shape[0]
    per = max(1, int((1 << 26) // max(1, math.prod(shape[1:]))))
    if descale_mode == "tensor_amax":
        # per-tensor descale needs the amax first: draw fully (only used at moderate sizes)
        x = _randn(shape, gen_cpu, device, seed, slot, mean, std)
        amax = x.abs().max().clamp_min(1e-12)
        ds = (amax / E4M3_MAX).to(torch.float32).reshape(())
        return quantise_e4m3(x, ds), ds
    out = torch.empty(shape, dtype=torch.float8_e4m3fn, device=device)
    if device.type == "cpu":
        for s in range(0, n0, per):
            e = min(n0, s + per)
            x = torch.randn((e - s,) + tuple(shape[1:]), generator=gen_cpu, dtype=torch.float32)
            if std != 1.0:
                x.mul_(std)
            if mean != 0.0:
                x.add_(mean)
            out[s:e] = quantise_e4m3(x, None)
    else:
        g = torch.Generator(device=device)
        g.manual_seed(seed * 1000 + slot)
        for s in range(0, n0, per):
            e = min(n0, s + per)
            x = torch.randn((e - s,) + tuple(shape[1:]), generator=g, dtype=torch.float32,
                            device=device)
            if std != 1.0:
                x.mul_(std)
            if mean != 0.0:
                x.add_(mean)
            out[s:e] = quantise_e4m3(x, None)
    return out, None


def make_case(*, name="case", B: int, Hq: int, Hkv: int, D: int, DV: int,
              seqlens_q: Sequence[int], seqlens_k: Sequence[int],
              q_layout="batched", kv_layout="batched", page_size=16, extra_pages=0,
              table_width: Optional[int] = None,
              causal=False, window_left=-1, sink=False, softmax_scale: Optional[float] = None,
              q_dist=(0.0, 1.0), k_dist=(0.0, 1.0), v_dist=(0.0, 1.0),
              descale_mode="none", out_dtype=torch.bfloat16, seed=0, device="cpu") -> Case:
    """Draws one case.

    descale_mode:
      "none"            no descale tensors (the op uses 1.0); payload = e4m3(N(mean,std))
      "one"             0-d descales equal to 1.0; payload = e4m3(N(mean,std))
      "tensor_amax"     per-tensor descale amax/448, payload = e4m3(x / descale)
      "per_bkv_uniform" (B,Hkv) descales ~ U[0.5,2] drawn independently for q, k, v;
                        payload = e4m3(N(mean,std))
    """
    assert q_layout in ("batched", "varlen")
    assert kv_layout in LAYOUTS
    assert Hq % Hkv == 0
    seqlens_q = [int(x) for x in seqlens_q]
    seqlens_k = [int(x) for x in seqlens_k]
    assert len(seqlens_q) == B and len(seqlens_k) == B
    if q_layout == "batched":
        assert len(set(seqlens_q)) == 1, "batched Q needs equal query lengths"
    if kv_layout == "batched":
        assert len(set(seqlens_k)) == 1, "batched K/V needs equal key lengths"

    gen = torch.Generator().manual_seed(seed)
    dev = torch.device(device)

    # ---- Q
    if q_layout == "batched":
        qshape = (B, seqlens_q[0], Hq, D)
    else:
        qshape = (sum(seqlens_q), Hq, D)
    # ---- K/V storage
    block_table = None
    if kv_layout == "batched":
        kshape = (B, seqlens_k[0], Hkv, D)
        vshape = (B, seqlens_k[0], Hkv, DV)
    elif kv_layout == "varlen":
        kshape = (sum(seqlens_k), Hkv, D)
        vshape = (sum(seqlens_k), Hkv, DV)
    else:
        assert page_size > 0
        npages = [(lk + page_size - 1) // page_size for lk in seqlens_k]
        pool = sum(npages) + extra_pages
        width = max(npages + [1]) if table_width is None else table_width
        assert width >= max(npages + [0])
        perm = torch.randperm(pool, generator=gen).to(torch.int32)
        block_table = torch.full((B, width), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(npages):
            block_table[b, :n] = perm[off:off + n]
            off += n
        kshape = (pool, page_size, Hkv, D)
        vshape = (pool, page_size, Hkv, DV)

    # ---- descales drawn before payloads so that they are identical across devices
    dq = dk = dvv = None
    if descale_mode == "one":
        dq = torch.ones((), dtype=torch.float32)
        dk = torch.ones((), dtype=torch.float32)
        dvv = torch.ones((), dtype=torch.float32)
    elif descale_mode == "per_bkv_uniform":
        dq = (torch.rand((B, Hkv), generator=gen) * 1.5 + 0.5).to(torch.float32)
        dk = (torch.rand((B, Hkv), generator=gen) * 1.5 + 0.5).to(torch.float32)
        dvv = (torch.rand((B, Hkv), generator=gen) * 1.5 + 0.5).to(torch.float32)
    elif descale_mode in ("none", "tensor_amax"):
        pass
    else:
        raise ValueError(descale_mode)

    sink_t = None
    if sink:
        sink_t = torch.randn((Hq,), generator=gen, dtype=torch.float32)

    q, q_ds = _quantised_payload(qshape, gen, dev, seed, 1, q_dist[0], q_dist[1], descale_mode)
    k, k_ds = _quantised_payload(kshape, gen, dev, seed, 2, k_dist[0], k_dist[1], descale_mode)
    v, v_ds = _quantised_payload(vshape, gen, dev, seed, 3, v_dist[0], v_dist[1], descale_mode)
    if descale_mode == "tensor_amax":
        dq, dk, dvv = q_ds.cpu(), k_ds.cpu(), v_ds.cpu()

    cu_q = cu_k = None
    if q_layout == "varlen":
        cu_q = torch.tensor([0] + list(_cumsum(seqlens_q)), dtype=torch.int32)
    if kv_layout in ("varlen", "paged"):
        cu_k = torch.tensor([0] + list(_cumsum(seqlens_k)), dtype=torch.int32)

    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)

    c = Case(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, DV=DV, seqlens_q=seqlens_q,
             seqlens_k=seqlens_k, q_layout=q_layout, kv_layout=kv_layout, q=q, k=k, v=v,
             descale_q=dq, descale_k=dk, descale_v=dvv, cu_seqlens_q=cu_q,
             cu_seqlens_k=cu_k, block_table=block_table,
             page_size=page_size if kv_layout == "paged" else 0, causal=bool(causal),
             window_left=int(window_left), sink=sink_t, softmax_scale=float(softmax_scale),
             out_dtype=out_dtype)
    return c.to(dev)


def _cumsum(xs):
    s = 0
    for x in xs:
        s += x
        yield s


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n integer lengths ~ U[lo, hi] (inclusive), from a CPU generator."""
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


# --------------------------------------------------------------------------------------
# The five workloads.  ``scale="full"`` gives the stated sizes; ``scale="small"`` keeps
# each workload's structure (masking, GQA ratio, paging, length mix, head dims) at a
# size the fp64 oracle finishes in seconds while still spanning several 128-key tiles
# and a ragged tail.
# --------------------------------------------------------------------------------------

def tiny_dense(device="cpu") -> Case:
    """B=1, Hq=Hkv=2, Sq=Sk=128, d=dv=64, non-causal, 0-d descales of 1.0, seed 0."""
    return make_case(name="tiny_dense", B=1, Hq=2, Hkv=2, D=64, DV=64, seqlens_q=[128],
                     seqlens_k=[128], descale_mode="one", softmax_scale=1.0 / 8.0,
                     out_dtype=torch.bfloat16, seed=0, device=device)


def causal_gqa_prefill(scale="full", device="cpu") -> Case:
    """Causal GQA prefill, d=dv=128, V ~ N(0.5,1), per-tensor amax/448 descales, seed 1."""
    if scale == "full":
        B, Hq, Hkv, S = 2, 32, 8, 4096
    else:
        B, Hq, Hkv, S = 2, 8, 2, 333
    return make_case(name=f"causal_gqa_prefill_{scale}", B=B, Hq=Hq, Hkv=Hkv, D=128, DV=128,
                     seqlens_q=[S] * B, seqlens_k=[S] * B, causal=True,
                     q_dist=(0.0, 1.0), k_dist=(0.0, 1.0), v_dist=(0.5, 1.0),
                     descale_mode="tensor_amax", out_dtype=torch.bfloat16, seed=1,
                     device=device)


def paged_decode(scale="full", device="cpu") -> Case:
    """One query token per request over a 16-token paged pool, d=dv=128, seed 2."""
    if scale == "full":
        B, Hq, Hkv, lo, hi = 64, 64, 8, 1024, 32768
    else:
        B, Hq, Hkv, lo, hi = 6, 16, 2, 100, 900
    lens = uniform_lengths(B, lo, hi, seed=2)
    return make_case(name=f"paged_decode_{scale}", B=B, Hq=Hq, Hkv=Hkv, D=128, DV=128,
                     seqlens_q=[1] * B, seqlens_k=lens, q_layout="batched",
                     kv_layout="paged", page_size=16, causal=True,
                     descale_mode="per_bkv_uniform", out_dtype=torch.bfloat16, seed=2,
                     device=device)


def long_kv(sq: int = 1, scale="full", device="cpu") -> Case:
    """B=1, Hq=8, Hkv=1, Sk=131072 keys, d=dv=256, V ~ N(1,0.1), per-tensor descales, seed 3."""
    sk = 131072 if scale == "full" else 2000
    return make_case(name=f"long_kv_sq{sq}_{scale}", B=1, Hq=8, Hkv=1, D=256, DV=256,
                     seqlens_q=[sq], seqlens_k=[sk], causal=False,
                     q_dist=(0.0, 1.0), k_dist=(0.0, 1.0), v_dist=(1.0, 0.1),
                     descale_mode="tensor_amax", out_dtype=torch.bfloat16, seed=3,
                     device=device)


def varlen_swa_prefill(scale="full", device="cpu") -> Case:
    """16 packed sequences ~U[256,8192], Hq=16/Hkv=4, d=192, dv=128, causal, window 1024,
    per-head sink ~ N(0,1), fp16 out, seed 4."""
    if scale == "full":
        n, lo, hi, Hq, Hkv, win = 16, 256, 8192, 16, 4, 1024
    else:
        n, lo, hi, Hq, Hkv, win = 4, 100, 700, 4, 2, 200
    lens = uniform_lengths(n, lo, hi, seed=4)
    return make_case(name=f"varlen_swa_prefill_{scale}", B=n, Hq=Hq, Hkv=Hkv, D=192, DV=128,
                     seqlens_q=lens, seqlens_k=lens, q_layout="varlen", kv_layout="varlen",
                     causal=True, window_left=win, sink=True, descale_mode="one",
                     out_dtype=torch.float16, seed=4, device=device)


# Per-layer decode steps of served models ("[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward
# for Hopper", Performance: requests x query tokens at a context length, 16-token pages,
# causal, with the split-KV combine).  The head counts per GPU are those of the public model
# configurations under the stated tensor parallelism; the d=256 windowed rows of that table
# are left out because the page does not give their head counts.  One more row runs the
# four-token shape with 64-token pages.
DECODE_STEP_SHAPES = [
    # (name, requests, query tokens, context, Hq, Hkv, page size)
    ("llama3.1-8b-tp1 1x1 4k", 1, 1, 4096, 32, 8, 16),
    ("llama3.1-8b-tp1 32x1 2k", 32, 1, 2048, 32, 8, 16),
    ("llama3.1-8b-tp1 128x1 1k", 128, 1, 1024, 32, 8, 16),
    ("llama3.1-8b-tp1 16x1 16k", 16, 1, 16384, 32, 8, 16),
    ("llama3.1-8b-tp1 32x4 4k", 32, 4, 4096, 32, 8, 16),
    ("llama3.1-70b-tp4 64x1 4k", 64, 1, 4096, 16, 2, 16),
    ("llama3.1-70b-tp4 8x1 32k", 8, 1, 32768, 16, 2, 16),
    ("qwen3-32b-tp2 32x1 8k", 32, 1, 8192, 32, 4, 16),
    ("llama3.1-8b-tp1 32x4 4k page64", 32, 4, 4096, 32, 8, 64),
]


def decode_step(shape, device="cpu", max_seqlen_k=32768) -> Case:
    """One of DECODE_STEP_SHAPES: e4m3(N(0,1)) Q/K/V, per-(batch, kv-head) descales, d=128,
    every request at the stated context, block tables as wide as max_seqlen_k."""
    name, reqs, sq, ctx, hq, hkv, ps = shape
    return make_case(name=name, B=reqs, Hq=hq, Hkv=hkv, D=128, DV=128, seqlens_q=[sq] * reqs,
                     seqlens_k=[ctx] * reqs, q_layout="batched", kv_layout="paged", page_size=ps,
                     table_width=max_seqlen_k // ps, causal=True, descale_mode="per_bkv_uniform",
                     out_dtype=torch.bfloat16, seed=5, device=device)


STAIRCASE_Q_LEVELS = (1.0, 1.25, 1.5, 1.75)  # exact E4M3 values


def lazy_staircase(kind="prefill", device="cpu", tiles=64) -> Case:
    """Scores that climb steadily along the keys, to exercise the lazy rescale threshold.

    Every row's largest score rises by 0.5 q log2-units per 128 keys for ``tiles`` blocks of
    128 keys, so an online softmax that moves its running max only after the block max has
    passed it by more than a threshold writes unnormalised weights up to 2^threshold: above
    the E4M3 range once the threshold exceeds log2(448) - 8.  Built from exact E4M3 values:
    Q rows are constant vectors of one of STAIRCASE_Q_LEVELS (cycling over rows and heads);
    key j of block t has n = max(0, 2 t - 3 (j mod 8)) leading components equal to 2 and
    the rest 0; with softmax_scale = ln 2 / 8 its log2-unit score is q n / 4.  V is
    e4m3(N(0,1)), seed 6.  ``kind`` "prefill": 64 query rows, 2 q-heads on one kv-head
    (the 128-row kernel); "decode": two one-token requests with 8 q-heads on one kv-head
    (the decode kernel).
    """
    if kind == "prefill":
        B, Sq, Hq = 1, 64, 2
    else:
        B, Sq, Hq = 2, 1, 8
    D = DV = 128
    sk = tiles * 128
    lev = torch.tensor(STAIRCASE_Q_LEVELS, dtype=torch.float32)
    idx = (torch.arange(Sq)[:, None] * Hq + torch.arange(Hq)[None, :]) % len(STAIRCASE_Q_LEVELS)
    q = lev[idx][None, :, :, None].expand(B, Sq, Hq, D).contiguous()
    j = torch.arange(sk)
    n = (2 * (j // 128) - 3 * (j % 8)).clamp_min(0)
    k = (torch.arange(D)[None, :] < n[:, None]).to(torch.float32) * 2.0
    k = k[None, :, None, :].expand(B, sk, 1, D).contiguous()
    gen = torch.Generator().manual_seed(6)
    v, _ = _quantised_payload((B, sk, 1, DV), gen, "cpu", 6, 3, 0.0, 1.0, "one")
    case = Case(name=f"lazy_staircase_{kind}", B=B, Hq=Hq, Hkv=1, D=D, DV=DV,
                seqlens_q=[Sq] * B, seqlens_k=[sk] * B, q_layout="batched", kv_layout="batched",
                q=quantise_e4m3(q, None), k=quantise_e4m3(k, None), v=v,
                softmax_scale=math.log(2.0) / 8.0, out_dtype=torch.bfloat16)
    return case.to(device)


def algorithmic_flops(case: Case) -> float:
    """2*(d+dv) flops per unmasked (row, key) pair, summed over heads."""
    return 2.0 * (case.D + case.DV) * case.pairs()


def algorithmic_bytes(case: Case) -> float:
    """Bytes the forward must move at least once: visible K/V rows per kv head (E4M3),
    Q (E4M3), O (2-byte) and LSE (fp32)."""
    kv = 0
    for lk in case.seqlens_k:
        kv += lk * case.Hkv * (case.D + case.DV)
    tq = case.total_q
    return float(kv + tq * case.Hq * case.D + tq * case.Hq * case.DV * 2 + tq * case.Hq * 4)
