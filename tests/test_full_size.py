"""Parity at the full workload sizes, in the launch configuration bench.py times.

The whole tensors are computed on the GPU; the fp64 oracle recomputes sampled
(batch, head) slices — exactly, for every element of the slice — or, where a
slice is too long for the CPU, sampled query rows (forward) and sampled query
and key rows (backward).  Every sample includes the first and last rows and
the first and last heads.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs
from helpers import check_grad, check_lse, check_o

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def gpu_fwd_bwd(x, w, fused=False):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.attention_fwd(q, k, v, scale=w.sm_scale, causal=w.causal)
    grads = None
    if w.backward:
        bwd = fa.attention_bwd_fused if fused else fa.attention_bwd
        grads = bwd(q, k, v, o, lse, x["dO"].cuda(), scale=w.sm_scale, causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    out = {"o": o.cpu(), "lse": lse.cpu()}
    if grads is not None:
        out.update(dq=grads[0].cpu(), dk=grads[1].cpu(), dv=grads[2].cpu())
    return out


def head_slices(x, b, kh, g):
    """The query heads of kv head kh (g of them) of batch b, as a B=1 problem."""
    hs = slice(kh * g, (kh + 1) * g)
    return {"q": x["q"][b:b + 1, :, hs], "k": x["k"][b:b + 1, :, kh:kh + 1], "v": x["v"][b:b + 1, :, kh:kh + 1],
            "dO": x["dO"][b:b + 1, :, hs] if x["dO"] is not None else None}


def sample_rows(N, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(n, N), replace=False).tolist()) | {0, 1, N - 2, N - 1}
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int32)


def check_sampled(oracle_mod, w, x, got, groups, rows=None, grad_rows=None):
    g = w.H // w.Hkv
    for (b, kh) in groups:
        xs = head_slices(x, b, kh, g)
        hs = slice(kh * g, (kh + 1) * g)
        what = f"{w.name} b{b} kv-head {kh}"
        o_ref, lse_ref = oracle_mod.attention_fwd(xs["q"], xs["k"], xs["v"], w.sm_scale, w.causal, rows=rows)
        sel = slice(None) if rows is None else rows
        check_o(got["o"][b:b + 1, sel, hs].float().numpy().astype(np.float64), o_ref, what)
        check_lse(got["lse"][b:b + 1, hs][:, :, sel].numpy().astype(np.float64), lse_ref, what)
        if not w.backward:
            continue
        qr = kr = None if grad_rows is None else grad_rows
        dq, dk, dv = oracle_mod.attention_bwd(xs["q"], xs["k"], xs["v"], xs["dO"], w.sm_scale, w.causal,
                                              qrows=qr, kvrows=kr)
        gsel = slice(None) if grad_rows is None else grad_rows
        check_grad(got["dq"][b:b + 1, gsel, hs], dq, what + " dQ")
        check_grad(got["dk"][b:b + 1, gsel, kh:kh + 1], dk, what + " dK")
        check_grad(got["dv"][b:b + 1, gsel, kh:kh + 1], dv, what + " dV")


def test_headline_b4_h16_n8192_d128(oracle_mod):
    w = inputs.headline()
    x = inputs.make_inputs(w)
    got = gpu_fwd_bwd(x, w)
    check_sampled(oracle_mod, w, x, got, groups=[(0, 0), (w.B - 1, w.H - 1)])


def test_fused_backward_headline_b4_h16_n8192_d128(oracle_mod):
    # the CTA-pair fused backward (fa_bwd_fused) on the headline workload
    w = inputs.headline()
    x = inputs.make_inputs(w)
    got = gpu_fwd_bwd(x, w, fused=True)
    check_sampled(oracle_mod, w, x, got, groups=[(0, 0), (w.B - 1, w.H - 1)])


def test_causal_outliers_b8_h16_n4096_d128(oracle_mod):
    w = inputs.causal_outliers()
    x = inputs.make_inputs(w)
    got = gpu_fwd_bwd(x, w)
    check_sampled(oracle_mod, w, x, got, groups=[(0, 0), (3, 8), (w.B - 1, w.H - 1)])


def test_long_gqa_b1_h32_hkv8_n32768_d128_fwd(oracle_mod):
    w = inputs.long_gqa()
    x = inputs.make_inputs(w, with_dO=False)
    got = gpu_fwd_bwd(x, w)
    rows = sample_rows(w.N, 256, 33)
    check_sampled(oracle_mod, w, x, got, groups=[(0, 0), (0, w.Hkv - 1)], rows=rows)


@pytest.mark.parametrize("w", inputs.sweep(), ids=lambda w: w.name.replace(" ", "_"))
def test_head_dim_sweep(oracle_mod, w):
    x = inputs.make_inputs(w, with_dO=w.backward)
    got = gpu_fwd_bwd(x, w)
    rows = sample_rows(w.N, 192, w.seed)
    check_sampled(oracle_mod, w, x, got, groups=[(0, 0), (w.B - 1, w.H - 1)], rows=rows,
                  grad_rows=rows if w.N > 4096 else None)


def test_packed_workload_full_size(oracle_mod):
    """The packed batch bench.py --workload varlen times (65536 tokens, 128..16384-row
    sequences, H16 d128 causal), computed whole; the oracle recomputes sampled rows of
    the shortest, a middle and the longest sequence for the first and last heads."""
    w = inputs.packed_causal()
    x = inputs.make_packed_inputs(w)
    q, k, v, dO = (x[n].cuda() for n in ("q", "k", "v", "dO"))
    cu = x["cu_seqlens"].cuda()
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, w.max_seqlen, scale=w.sm_scale, causal=w.causal)
    dq, dk, dv = fa.attention_bwd_varlen(q, k, v, o, lse, dO, cu, w.max_seqlen, scale=w.sm_scale, causal=w.causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse, dq, dk, dv = (t.cpu() for t in (o, lse, dq, dk, dv))
    bounds = w.cu_seqlens()
    lens = list(w.lens)
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    for b in (order[0], order[len(order) // 2], order[-1]):
        a, e = bounds[b], bounds[b + 1]
        L = e - a
        rows = sample_rows(L, 96, w.seed + b)
        for h in (0, w.H - 1):
            kh = h // (w.H // w.Hkv)
            sl = lambda t, hh: t[a:e, hh:hh + 1][None]  # one sequence, one head: [1, L, 1, d]
            what = f"packed seq {b} ({L} rows) head {h}"
            o_ref, lse_ref = oracle_mod.attention_fwd(sl(x["q"], h), sl(x["k"], kh), sl(x["v"], kh), w.sm_scale,
                                                      w.causal, rows=rows)
            check_o(o[a:e][rows, h:h + 1][None].float().numpy().astype(np.float64), o_ref, what)
            check_lse(lse[h, a:e][rows][None, None].numpy().astype(np.float64), lse_ref, what)
            rq, rk, rv = oracle_mod.attention_bwd(sl(x["q"], h), sl(x["k"], kh), sl(x["v"], kh), sl(x["dO"], h),
                                                  w.sm_scale, w.causal, qrows=rows, kvrows=rows)
            check_grad(dq[a:e][rows, h:h + 1][None], rq, what + " dQ")
            if w.H == w.Hkv:  # dK, dV of a kv head sum over its query heads: compare only 1:1 heads
                check_grad(dk[a:e][rows, kh:kh + 1][None], rk, what + " dK")
                check_grad(dv[a:e][rows, kh:kh + 1][None], rv, what + " dV")
