"""Pins for the fp64 oracle (CPU only).

The oracle is only trusted after it agrees with things other than itself:
  * the E4M3 format definition and torch's independent float8_e4m3fn decoder;
  * a fully materialised brute-force softmax (matrix form, scipy logsumexp, torch's
    decoder) on tiny inputs;
  * closed forms: constant V, all-equal keys (with and without a sink), the causal
    first row, a zero-width window;
  * invariants: KV permutation, GQA == MHA with repeated heads, varlen == per-sequence,
    paged == gathered contiguous, linearity in the V descale, dq/dk symmetry;
  * the nonzero-mean V property at long key lengths.
``test_planted_mistakes_are_caught`` compiles the oracle with each planted mistake
(ORACLE_MUTANT=1..10) and checks that at least one of these pins fails for it.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from fp8_attention_forward_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------- helpers
def _dec(t):
    """torch's own E4M3 decoder -> float64 numpy (independent of the oracle's)."""
    return t.to(torch.float32).to(torch.float64).cpu().numpy()


def brute_force(case):
    """Materialised S -> masked softmax -> O, in fp64, one (request, head) at a time."""
    B, Hq, Hkv, D, DV = case.B, case.Hq, case.Hkv, case.D, case.DV
    G = Hq // Hkv
    q = _dec(case.q).reshape(-1, Hq, D)
    if case.kv_layout == "paged":
        kpool = _dec(case.k)
        vpool = _dec(case.v)
        bt = case.block_table.cpu().numpy()
    else:
        k_all = _dec(case.k).reshape(-1, Hkv, D)
        v_all = _dec(case.v).reshape(-1, Hkv, DV)
    dq = np.broadcast_to(_dscl(case.descale_q), (B, Hkv))
    dk = np.broadcast_to(_dscl(case.descale_k), (B, Hkv))
    dv = np.broadcast_to(_dscl(case.descale_v), (B, Hkv))
    sink = None if case.sink is None else case.sink.double().cpu().numpy()
    total_q = sum(case.seqlens_q)
    O = np.zeros((total_q, Hq, DV))
    L = np.zeros((total_q, Hq))
    q0 = k0 = 0
    for b in range(B):
        Lq, Lk = case.seqlens_q[b], case.seqlens_k[b]
        if case.kv_layout == "paged":
            pages = bt[b, : (Lk + case.page_size - 1) // case.page_size]
            Kb = kpool[pages].reshape(-1, Hkv, D)[:Lk]
            Vb = vpool[pages].reshape(-1, Hkv, DV)[:Lk]
        else:
            Kb = k_all[k0:k0 + Lk]
            Vb = v_all[k0:k0 + Lk]
        Qb = q[q0:q0 + Lq]
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        vis = np.ones((Lq, Lk), dtype=bool)
        if case.causal:
            vis &= j <= i + (Lk - Lq)
        if case.window_left >= 0:
            vis &= j >= i + (Lk - Lq) - case.window_left
        for h in range(Hq):
            g = h // G
            S = case.softmax_scale * dq[b, g] * dk[b, g] * (Qb[:, h, :] @ Kb[:, g, :].T)
            S = np.where(vis, S, -np.inf)
            if sink is not None:
                S = np.concatenate([S, np.full((Lq, 1), sink[h])], axis=1)
            lse = logsumexp(S, axis=1) if S.shape[1] else np.full(Lq, -np.inf)
            with np.errstate(invalid="ignore"):
                P = np.exp(S - lse[:, None])
            P = np.nan_to_num(P[:, :Lk], nan=0.0)
            O[q0:q0 + Lq, h] = dv[b, g] * (P @ Vb[:, g, :])
            L[q0:q0 + Lq, h] = lse
        q0 += Lq
        k0 += Lk
    return O, L


def _dscl(d):
    if d is None:
        return np.ones(())
    return d.double().cpu().numpy()


def _mk(**kw):
    base = dict(B=1, Hq=2, Hkv=1, D=32, DV=16, seqlens_q=[5], seqlens_k=[7])
    base.update(kw)
    return inputs.make_case(**base)


def _close(a, b, tol):
    a = np.asarray(a)
    b = np.asarray(b)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(np.nan_to_num(diff, nan=np.inf) <= tol))


def _with_bytes(case, field, new_codes):
    """Returns a copy of case with q/k/v replaced by the given uint8 codes."""
    import dataclasses

    c = dataclasses.replace(case)
    setattr(c, field, torch.as_tensor(new_codes, dtype=torch.uint8).view(torch.float8_e4m3fn))
    return c


# ------------------------------------------------------------------------- pins
# Each pin returns True when the oracle built with ``mutant`` passes it.

def pin_e4m3_torch(mutant):
    codes = np.arange(256, dtype=np.uint8)
    ref = _dec(torch.from_numpy(codes).view(torch.float8_e4m3fn))
    got = np.array([oracle.e4m3_decode(c, mutant) for c in codes])
    same_nan = np.isnan(ref) == np.isnan(got)
    return bool(np.all(same_nan) and np.all((ref == got) | np.isnan(ref)))


def pin_e4m3_golden(mutant):
    ok = True
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, val = line.split()
            got = oracle.e4m3_decode(int(code, 16), mutant)
            want = float(val)
            if math.isnan(want):
                ok &= math.isnan(got)
            else:
                ok &= (got == want) and (math.copysign(1, got) == math.copysign(1, want))
    return ok


BRUTE_CASES = [
    dict(name="dense", seed=11),
    dict(name="causal_gqa", Hq=4, Hkv=2, seqlens_q=[9], seqlens_k=[9], causal=True, seed=12,
         descale_mode="per_bkv_uniform"),
    dict(name="causal_lq_lt_lk", Hq=2, Hkv=1, seqlens_q=[4], seqlens_k=[11], causal=True,
         seed=13),
    dict(name="causal_lq_gt_lk", Hq=2, Hkv=1, seqlens_q=[9], seqlens_k=[4], causal=True,
         seed=14),
    dict(name="window_sink", B=2, Hq=4, Hkv=2, seqlens_q=[10, 6], seqlens_k=[10, 6],
         q_layout="varlen", kv_layout="varlen", causal=True, window_left=3, sink=True,
         seed=15),
    dict(name="window_noncausal", seqlens_q=[6], seqlens_k=[12], window_left=2, seed=16),
    dict(name="paged", B=3, Hq=4, Hkv=2, seqlens_q=[2, 2, 2], seqlens_k=[5, 17, 9],
         kv_layout="paged", page_size=4, extra_pages=3, causal=True,
         descale_mode="per_bkv_uniform", seed=17),
    dict(name="tensor_descales", seqlens_q=[6], seqlens_k=[6], v_dist=(0.5, 1.0),
         descale_mode="tensor_amax", seed=18, sink=True),
]


def pin_brute_force(mutant):
    ok = True
    for spec in BRUTE_CASES:
        spec = dict(spec)
        spec.pop("name")
        case = _mk(**spec)
        o, l = oracle.attention(case, mutant=mutant)
        ob, lb = brute_force(case)
        ok &= _close(o, ob, 1e-12) and _close(l, lb, 1e-12)
    return ok


def pin_constant_v(mutant):
    """V = c everywhere -> O = c * dv for every row with a visible key (no sink)."""
    case = _mk(B=2, Hq=4, Hkv=2, seqlens_q=[6, 6], seqlens_k=[9, 9], causal=True,
               descale_mode="per_bkv_uniform", seed=21)
    code = 0x3C  # 1.5
    vc = np.full(tuple(case.v.shape), code, dtype=np.uint8)
    case = _with_bytes(case, "v", vc)
    o, _ = oracle.attention(case, mutant=mutant)
    dv = case.descale_v.double().numpy()  # (B, Hkv)
    want = np.zeros_like(o)
    for b in range(2):
        for h in range(4):
            want[b * 6:(b + 1) * 6, h, :] = 1.5 * dv[b, h // 2]
    return _close(o, want, 1e-12)


def pin_rows_sum_to_one(mutant):
    """V = 1.0, dv = 1 -> O = sum_j P_ij = 1 on every row (window, GQA, varlen)."""
    case = _mk(B=2, Hq=4, Hkv=1, seqlens_q=[7, 3], seqlens_k=[7, 3], q_layout="varlen",
               kv_layout="varlen", causal=True, window_left=2, seed=22)
    case = _with_bytes(case, "v", np.full(tuple(case.v.shape), 0x38, dtype=np.uint8))
    o, _ = oracle.attention(case, mutant=mutant)
    return _close(o, np.ones_like(o), 1e-12)


def _equal_keys_case(sink, seed):
    case = _mk(B=1, Hq=2, Hkv=1, D=32, DV=16, seqlens_q=[3], seqlens_k=[10], seed=seed,
               sink=sink, descale_mode="per_bkv_uniform")
    k = case.k.view(torch.uint8).numpy().copy()  # (1, Lk, Hkv, D)
    k[:, :] = k[:, 0:1]  # every key row equal to row 0
    return _with_bytes(case, "k", k)


def pin_equal_keys(mutant):
    """All keys equal -> s_j = s; O = dv*mean(V); LSE = s + ln n (closed form)."""
    ok = True
    for sink in (False, True):
        case = _equal_keys_case(sink, 23 + sink)
        o, lse = oracle.attention(case, mutant=mutant)
        q = _dec(case.q).reshape(-1, 2, 32)
        k = _dec(case.k).reshape(-1, 1, 32)
        v = _dec(case.v).reshape(-1, 1, 16)
        dq = float(case.descale_q[0, 0]); dk = float(case.descale_k[0, 0])
        dv = float(case.descale_v[0, 0])
        n = 10
        for i in range(3):
            for h in range(2):
                s = case.softmax_scale * dq * dk * float(q[i, h] @ k[0, 0])
                if sink:
                    sg = float(case.sink[h])
                    lse_w = math.log(n * math.exp(s) + math.exp(sg))
                    frac = n * math.exp(s) / (n * math.exp(s) + math.exp(sg))
                else:
                    lse_w = s + math.log(n)
                    frac = 1.0
                o_w = dv * frac * v[:, 0, :].mean(axis=0)
                ok &= abs(lse[i, h] - lse_w) < 1e-12 and _close(o[i, h], o_w, 1e-12)
    return ok


def pin_causal_first_row(mutant):
    """Lq == Lk, causal: row 0 sees key 0 only -> O = dv * V_0, LSE = s_00."""
    case = _mk(B=1, Hq=2, Hkv=2, seqlens_q=[8], seqlens_k=[8], causal=True, seed=25,
               descale_mode="per_bkv_uniform")
    o, lse = oracle.attention(case, mutant=mutant)
    v = _dec(case.v).reshape(-1, 2, 16)
    q = _dec(case.q).reshape(-1, 2, 32)
    k = _dec(case.k).reshape(-1, 2, 32)
    ok = True
    for h in range(2):
        dv = float(case.descale_v[0, h])
        s = case.softmax_scale * float(case.descale_q[0, h]) * float(case.descale_k[0, h]) \
            * float(q[0, h] @ k[0, h])
        ok &= _close(o[0, h], dv * v[0, h], 1e-12) and abs(lse[0, h] - s) < 1e-12
    return ok


def pin_zero_window(mutant):
    """window_left = 0 (causal) keeps only key i + (Lk - Lq): O = dv * V_{i+Lk-Lq}."""
    case = _mk(B=1, Hq=1, Hkv=1, seqlens_q=[4], seqlens_k=[9], causal=True, window_left=0,
               seed=26)
    o, _ = oracle.attention(case, mutant=mutant)
    v = _dec(case.v).reshape(-1, 1, 16)
    return all(_close(o[i, 0], v[i + 5, 0], 1e-12) for i in range(4))


def pin_permutation(mutant):
    """Non-causal, no window: permuting K/V rows jointly leaves O and LSE unchanged."""
    case = _mk(B=1, Hq=2, Hkv=1, seqlens_q=[5], seqlens_k=[13], seed=27, sink=True)
    o1, l1 = oracle.attention(case, mutant=mutant)
    perm = torch.randperm(13, generator=torch.Generator().manual_seed(0))
    k = case.k.view(torch.uint8)[:, perm].numpy().copy()
    v = case.v.view(torch.uint8)[:, perm].numpy().copy()
    c2 = _with_bytes(_with_bytes(case, "k", k), "v", v)
    o2, l2 = oracle.attention(c2, mutant=mutant)
    return _close(o1, o2, 1e-12) and _close(l1, l2, 1e-12)


def pin_gqa_equals_mha(mutant):
    """GQA (Hkv=2, G=3) == MHA with each kv head repeated for its q-head group."""
    import dataclasses

    case = _mk(B=1, Hq=6, Hkv=2, seqlens_q=[4], seqlens_k=[8], causal=True, seed=28,
               descale_mode="per_bkv_uniform")
    o1, l1 = oracle.attention(case, mutant=mutant)
    rep = lambda t: t.view(torch.uint8).repeat_interleave(3, dim=2).view(torch.float8_e4m3fn)
    c2 = dataclasses.replace(case, Hkv=6, k=rep(case.k), v=rep(case.v),
                             descale_q=case.descale_q.repeat_interleave(3, dim=1),
                             descale_k=case.descale_k.repeat_interleave(3, dim=1),
                             descale_v=case.descale_v.repeat_interleave(3, dim=1))
    o2, l2 = oracle.attention(c2, mutant=mutant)
    return _close(o1, o2, 1e-12) and _close(l1, l2, 1e-12)


def pin_varlen_equals_dense(mutant):
    """A varlen batch equals one dense call per sequence."""
    import dataclasses

    lens = [5, 9, 3]
    case = _mk(B=3, Hq=2, Hkv=1, seqlens_q=lens, seqlens_k=lens, q_layout="varlen",
               kv_layout="varlen", causal=True, seed=29, sink=True)
    o, l = oracle.attention(case, mutant=mutant)
    ok = True
    off = 0
    for b, n in enumerate(lens):
        sub = dataclasses.replace(case, B=1, seqlens_q=[n], seqlens_k=[n], q_layout="batched",
                                  kv_layout="batched", q=case.q[off:off + n][None],
                                  k=case.k[off:off + n][None], v=case.v[off:off + n][None],
                                  cu_seqlens_q=None, cu_seqlens_k=None)
        ob, lb = oracle.attention(sub, mutant=mutant)
        ok &= _close(o[off:off + n], ob, 1e-15) and _close(l[off:off + n], lb, 1e-15)
        off += n
    return ok


def pin_paged_equals_contiguous(mutant):
    """Paged K/V equals the same keys gathered into a contiguous varlen layout."""
    import dataclasses

    case = _mk(B=2, Hq=4, Hkv=2, seqlens_q=[3, 3], seqlens_k=[11, 6], kv_layout="paged",
               page_size=4, extra_pages=2, causal=True, seed=30,
               descale_mode="per_bkv_uniform")
    o1, l1 = oracle.attention(case, mutant=mutant)
    ks, vs = [], []
    for b, lk in enumerate(case.seqlens_k):
        pages = case.block_table[b, : (lk + 3) // 4].long()
        ks.append(case.k.view(torch.uint8)[pages].reshape(-1, 2, 32)[:lk])
        vs.append(case.v.view(torch.uint8)[pages].reshape(-1, 2, 16)[:lk])
    c2 = dataclasses.replace(case, kv_layout="varlen", block_table=None, page_size=0,
                             k=torch.cat(ks).view(torch.float8_e4m3fn),
                             v=torch.cat(vs).view(torch.float8_e4m3fn))
    o2, l2 = oracle.attention(c2, mutant=mutant)
    return _close(o1, o2, 0.0) and _close(l1, l2, 0.0)


def pin_descale_structure(mutant):
    """O is linear in the V descale; dq and dk enter only through their product."""
    import dataclasses

    case = _mk(B=1, Hq=2, Hkv=1, seqlens_q=[4], seqlens_k=[6], seed=31,
               descale_mode="per_bkv_uniform")
    o1, l1 = oracle.attention(case, mutant=mutant)
    c2 = dataclasses.replace(case, descale_v=case.descale_v * 3.0)
    o2, l2 = oracle.attention(c2, mutant=mutant)
    c3 = dataclasses.replace(case, descale_q=case.descale_k, descale_k=case.descale_q)
    o3, l3 = oracle.attention(c3, mutant=mutant)
    return (_close(o2, 3.0 * o1, 1e-12) and _close(l2, l1, 0.0) and _close(o3, o1, 1e-12)
            and _close(l3, l1, 1e-12))


def pin_nonzero_mean_v(mutant):
    """V ~ N(1, 0.1) independent of the scores, 131072 keys (the long-KV length): the
    softmax-weighted mean of V equals the plain mean of the dequantised V up to sampling
    noise (std ~1e-4 here: 0.1 / sqrt(effective key count ~5e4), averaged over 64 columns).
    A reduced-precision O accumulator that loses a little of every add shrinks it by far more
    ("[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward for Hopper", Design, "Two-level PV
    accumulation": the output shrinks with the key count when the accumulator truncates)."""
    case = inputs.make_case(B=1, Hq=2, Hkv=1, D=64, DV=32, seqlens_q=[1], seqlens_k=[131072],
                            v_dist=(1.0, 0.1), descale_mode="tensor_amax", seed=32)
    o, _ = oracle.attention(case, mutant=mutant)
    dv = float(case.descale_v)
    v_mean = float(case.v.float().double().mean()) * dv
    return abs(float(o.mean()) - v_mean) < 1e-3 and abs(v_mean - 1.0) < 0.02


def pin_split_merge(mutant):
    """Keys split into a prefix and the rest: merging the two partial results by their LSEs
    (LSE = log(e^LSE_1 + e^LSE_2), O = sum_s e^(LSE_s - LSE) O_s, in fp64) gives the single
    pass.  The sink goes with one part only."""
    import dataclasses

    case = _mk(B=1, Hq=2, Hkv=1, seqlens_q=[4], seqlens_k=[11], seed=30, sink=True,
               descale_mode="per_bkv_uniform")
    o, l = oracle.attention(case, mutant=mutant)
    a = 4
    k8, v8 = case.k.view(torch.uint8), case.v.view(torch.uint8)
    part = lambda t: t.contiguous().view(torch.float8_e4m3fn)
    c1 = dataclasses.replace(case, seqlens_k=[a], k=part(k8[:, :a]), v=part(v8[:, :a]))
    c2 = dataclasses.replace(case, seqlens_k=[11 - a], k=part(k8[:, a:]), v=part(v8[:, a:]),
                             sink=None)
    o1, l1 = oracle.attention(c1, mutant=mutant)
    o2, l2 = oracle.attention(c2, mutant=mutant)
    lm = np.logaddexp(l1, l2)
    om = np.exp(l1 - lm)[..., None] * o1 + np.exp(l2 - lm)[..., None] * o2
    return _close(om, o, 1e-12) and _close(lm, l, 1e-12)


PINS = [pin_e4m3_torch, pin_e4m3_golden, pin_brute_force, pin_constant_v,
        pin_rows_sum_to_one, pin_equal_keys, pin_causal_first_row, pin_zero_window,
        pin_permutation, pin_gqa_equals_mha, pin_varlen_equals_dense,
        pin_paged_equals_contiguous, pin_descale_structure, pin_nonzero_mean_v,
        pin_split_merge]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle_lib, pin):
    assert pin(0)


def test_sampled_rows_match_full(oracle_lib):
    case = _mk(B=2, Hq=4, Hkv=2, seqlens_q=[6, 4], seqlens_k=[6, 4], q_layout="varlen",
               kv_layout="varlen", causal=True, sink=True, seed=40)
    o, l = oracle.attention(case)
    rows = [(0, 0), (5, 3), (7, 1), (9, 2)]
    os_, ls_ = oracle.attention(case, rows=rows)
    for r, (t, h) in enumerate(rows):
        assert np.array_equal(os_[r], o[t, h]) and ls_[r] == l[t, h]


def test_empty_rows(oracle_lib):
    """Lq > Lk causal: early rows see no key -> O = 0, LSE = -inf (sink: LSE = sink)."""
    case = _mk(B=1, Hq=2, Hkv=1, seqlens_q=[6], seqlens_k=[2], causal=True, seed=41)
    o, l = oracle.attention(case)
    assert np.all(o[:4] == 0) and np.all(np.isneginf(l[:4]))
    import dataclasses

    c2 = dataclasses.replace(case, sink=torch.tensor([0.25, -1.0]))
    o2, l2 = oracle.attention(c2)
    assert np.all(o2[:4] == 0) and np.allclose(l2[:4], [[0.25, -1.0]] * 4, atol=0, rtol=0)


N_MUTANTS = 10


@pytest.mark.parametrize("mutant", range(1, N_MUTANTS + 1))
def test_planted_mistakes_are_caught(oracle_lib, mutant):
    oracle.build(mutant)
    failed = [p.__name__ for p in PINS if not p(mutant)]
    assert failed, f"mutant {mutant} passes every pin"
