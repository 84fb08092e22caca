"""Backward parity: dQ, dK, dV from the CUDA library (through its C ABI)
against the fp64 oracle on the same seeded bf16 inputs (relative L2 per tensor,
plus an element-wise bound scaled to the tensor's magnitude)."""
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs
from helpers import check_grad

pytestmark = pytest.mark.gpu


def run(q, k, v, dO, scale, causal):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.attention_fwd(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = fa.attention_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    return dq.cpu(), dk.cpu(), dv.cpu()


def check_all(got, ref, what):
    """Relative L2 per tensor (the target, 1e-2), plus the same measure per
    128-row tile of each (batch, head) so that one wrong tile cannot hide in a
    whole-tensor norm.  The tile bound is 3e-2, its denominator floored at a
    tenth of the typical tile norm (a tile whose exact gradient nearly cancels,
    e.g. one-hot softmax rows where dP_ij ~ D_i, carries the bf16 rounding of
    O in D = rowsum(dO * O) without a matching signal)."""
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        check_grad(g, r, f"{what} {name}")
        if np.linalg.norm(r) == 0.0:
            continue
        gg = g.float().numpy().astype(np.float64)
        B, N, Hx, d = r.shape
        pad = (-N) % 128
        e = np.pad(gg - r, ((0, 0), (0, pad), (0, 0), (0, 0))).reshape(B, -1, 128, Hx, d)
        rr = np.pad(r, ((0, 0), (0, pad), (0, 0), (0, 0))).reshape(B, -1, 128, Hx, d)
        err_t = np.sqrt((e ** 2).sum(axis=(2, 4)))
        ref_t = np.sqrt((rr ** 2).sum(axis=(2, 4)))
        floor = 0.1 * np.sqrt((ref_t ** 2).mean())
        rel = err_t / np.maximum(ref_t, floor)
        assert (rel <= 3e-2).all(), f"{what} {name}: tile (b, tile, head) {np.unravel_index(rel.argmax(), rel.shape)} rel {rel.max():.3e}"


def test_tiny_workload_full(oracle_mod):
    w = inputs.tiny()
    x = inputs.make_inputs(w)
    got = run(x["q"], x["k"], x["v"], x["dO"], w.sm_scale, w.causal)
    ref = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dO"], w.sm_scale, w.causal)
    check_all(got, ref, w.name)


CASES = [
    # B, N, H, Hkv, d, causal
    (1, 128, 1, 1, 128, False),
    (1, 256, 2, 2, 128, False),
    (2, 384, 2, 2, 128, True),
    (1, 1, 1, 1, 128, False),
    (1, 77, 2, 2, 128, True),
    (1, 300, 2, 2, 128, False),
    (1, 513, 1, 1, 128, True),
    (1, 256, 4, 2, 128, False),
    (1, 384, 4, 1, 128, True),
    (1, 256, 2, 2, 64, False),
    (1, 395, 2, 2, 64, True),
    (2, 200, 4, 2, 64, True),
    # more head-dim-64 key tiles than SMs: persistent dK/dV CTAs run several units
    (8, 333, 16, 8, 64, True),
    (4, 640, 8, 8, 64, False),
    (1, 256, 2, 2, 256, False),
    (1, 333, 2, 1, 256, True),
    (2, 128, 2, 2, 256, True),
    # either side of the lengths where head-dim-128 dK/dV moves from one CTA per
    # key tile to CTA pairs (2048 rows, 4096 causal); the longer ones are ragged
    (1, 2048, 2, 2, 128, False),
    (1, 2049, 2, 1, 128, False),
    (1, 4096, 1, 1, 128, True),
    (1, 4097, 1, 1, 128, True),
]


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", CASES)
def test_small_shapes_full(oracle_mod, B, N, H, Hkv, d, causal):
    seed = 2000 + N + 7 * d + H + causal
    q = inputs.random_bf16((B, N, H, d), seed)
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1)
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2)
    dO = inputs.random_bf16((B, N, H, d), seed + 3)
    scale = 1.0 / math.sqrt(d)
    got = run(q, k, v, dO, scale, causal)
    ref = oracle_mod.attention_bwd(q, k, v, dO, scale, causal)
    check_all(got, ref, f"B{B} N{N} H{H}/{Hkv} d{d} causal={causal}")


def test_outliers(oracle_mod):
    w = inputs.Workload("outliers", 1, 2, 2, 640, 128, True, 9, outliers=True)
    x = inputs.make_inputs(w)
    got = run(x["q"], x["k"], x["v"], x["dO"], w.sm_scale, w.causal)
    ref = oracle_mod.attention_bwd(x["q"], x["k"], x["v"], x["dO"], w.sm_scale, w.causal)
    check_all(got, ref, w.name)
