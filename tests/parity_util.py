"""Shared helpers for the GPU parity tests: run the CUDA path and the fp64 oracle on the same
seeded case and measure the error the way the tolerances are stated (unit-scale V: the
error on O is divided by the RMS of the dequantised V of the row's request and kv-head)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fp8_attention_forward_gb300 import fa8

# Tolerances for the E4M3 path against the fp64 oracle over the dequantised inputs.
MAX_ABS = 3e-2   # max |O - O_ref| / scale(V)
MEAN_ABS = 4e-3  # mean |O - O_ref| / scale(V)
LSE_ABS = 2e-3   # max |LSE - LSE_ref| (natural log)


def row_meta(case):
    """For every packed (token, q-head): batch index and kv-head index."""
    b_of_tok = np.repeat(np.arange(case.B), case.seqlens_q)
    g_of_head = np.arange(case.Hq) // (case.Hq // case.Hkv)
    return b_of_tok, g_of_head


def v_scale(case):
    """(B, Hkv) RMS of the dequantised V (descale * E4M3 value) over each request's keys.

    The tolerances are stated for unit-scale V, so errors on O are divided by this scale:
    it is the V descale when the payload is unit-normal, and ~1 when V itself is unit-scale
    and only the payload carries an amax/448 descale."""
    dv = np.ones((case.B, case.Hkv))
    if case.descale_v is not None:
        dv = np.broadcast_to(case.descale_v.double().cpu().numpy(), (case.B, case.Hkv))
    out = np.ones((case.B, case.Hkv))
    off = 0
    for b, lk in enumerate(case.seqlens_k):
        if lk == 0:
            continue
        v8 = case.v.view(torch.uint8)  # byte view: float8 tensors cannot be indexed everywhere
        if case.kv_layout == "batched":
            rows = v8[b]
        elif case.kv_layout == "varlen":
            rows = v8[off:off + lk]
        else:
            pages = case.block_table[b, : (lk + case.page_size - 1) // case.page_size].long()
            rows = v8[pages.to(case.v.device)].reshape(-1, case.Hkv, case.DV)[:lk]
        off += lk
        rows = rows.view(torch.float8_e4m3fn)
        ms = rows.float().pow(2).mean(dim=(0, 2)).double().cpu().numpy()
        out[b] = np.sqrt(ms) * dv[b]
    return out


def scale_of_rows(case):
    """(total_q, Hq) error scale for every output row (see ``v_scale``)."""
    b_of_tok, g_of_head = row_meta(case)
    return v_scale(case)[b_of_tok][:, g_of_head]


def gpu_outputs(case, out, lse):
    """Packed (total_q, Hq, DV) fp64 O and (total_q, Hq) LSE from the library's layouts."""
    o = out.double().cpu().numpy().reshape(case.total_q, case.Hq, case.DV)
    if lse is None:
        return o, None
    l = lse.double().cpu().numpy()
    if case.q_layout == "batched":  # (B, Hq, Sq) -> (B*Sq, Hq)
        l = l.transpose(0, 2, 1).reshape(case.total_q, case.Hq)
    else:  # (Hq, total_q)
        l = l.T
    return o, l


def errors(case, o, l, o_ref, l_ref, rows=None):
    """(max_abs, mean_abs, lse_max_abs) in unit-V units over all rows or the sampled rows."""
    dv = scale_of_rows(case)
    if rows is not None:
        toks = np.array([r[0] for r in rows])
        heads = np.array([r[1] for r in rows])
        o = o[toks, heads]
        l = l[toks, heads]
        dv = dv[toks, heads]
    e = np.abs(o - o_ref) / dv[..., None]
    both_inf = np.isinf(l) & np.isinf(l_ref) & (np.sign(l) == np.sign(l_ref))
    le = np.where(both_inf, 0.0, np.abs(l - l_ref))
    le = np.nan_to_num(le, nan=np.inf)
    return float(np.nan_to_num(e, nan=np.inf).max()), float(np.nan_to_num(e, nan=np.inf).mean()), float(le.max())


def run_gpu(case, **kw):
    out, lse = fa8.fwd_case(case, **kw)
    st = fa8.check()
    assert st == fa8.FA8_SUCCESS, f"device status {st}"
    return out, lse


# Every parity check made in this process: (test, case, rows checked, max, mean, LSE error,
# and the bars), printed by the test session's summary and written to FA8_PARITY_LOG when set.
MARGINS = []


def record_margin(case_cpu, mx, mean, le, rows=None, extra=""):
    import os

    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    MARGINS.append({"test": test, "case": case_cpu.name + (f" {extra}" if extra else ""),
                    "rows": "all" if rows is None else len(rows), "max_abs": mx, "mean_abs": mean,
                    "lse_abs": le, "bars": [MAX_ABS, MEAN_ABS, LSE_ABS],
                    "ok": bool(mx <= MAX_ABS and mean <= MEAN_ABS and le <= LSE_ABS)})


def assert_parity(case_cpu, rows=None, device="cuda", **kw):
    """Runs the case on the GPU and the oracle (all rows or `rows`) and checks tolerances."""
    c = case_cpu.to(device)
    out, lse = run_gpu(c, **kw)
    o, l = gpu_outputs(case_cpu, out, lse)
    o_ref, l_ref = oracle.attention(case_cpu, rows=rows)
    mx, mean, le = errors(case_cpu, o, l, o_ref, l_ref, rows=rows)
    record_margin(case_cpu, mx, mean, le, rows)
    assert mx <= MAX_ABS and mean <= MEAN_ABS and le <= LSE_ABS, (
        f"{case_cpu.name}: max {mx:.3g} mean {mean:.3g} lse {le:.3g}")
    return mx, mean, le, out, lse


def sample_rows(case, n, seed=0):
    """n distinct (token, head) rows, always including the first and last token."""
    g = np.random.default_rng(seed)
    toks = g.integers(0, case.total_q, size=n)
    toks[0] = 0
    toks[-1] = case.total_q - 1
    heads = g.integers(0, case.Hq, size=n)
    return sorted(set(zip(toks.tolist(), heads.tolist())))
