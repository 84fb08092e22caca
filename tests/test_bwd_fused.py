"""The fused CTA-pair backward (fa_bwd_fused, head dim 128) against the oracle.

One KV-stationary kernel on cluster pairs computes dK, dV and dQ partials; the
pair exchanges dS halves through distributed shared memory and adds dQ with
fp32 reductions (FlashAttention-4 paper summary, section 2.C).  dK and dV come
from the same MMAs on the same bf16 operands as fa_bwd's pair kernel, so they
must be bitwise equal to fa_bwd's; dQ is summed in a run-dependent order and
must match the oracle within the backward tolerance (relative L2 1e-2 per
tensor and 3e-2 per 128-row tile).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs
from helpers import check_grad

pytestmark = pytest.mark.gpu

CASES = [
    # B, N, H, Hkv, causal
    (1, 128, 1, 1, False),   # one key tile: its partner holds no rows
    (1, 256, 2, 2, False),
    (2, 384, 2, 2, True),    # the last pair is half empty; the pair's second tile masks a query tile whole
    (1, 77, 2, 2, True),     # ragged single tile
    (1, 1, 1, 1, False),     # a single row
    (1, 1000, 2, 1, False),  # GQA, ragged tail inside the second tile of a pair
    (2, 640, 4, 2, True),    # GQA, causal, odd tile count
]


def tile_rel_l2(g, r, what):
    # per (batch, head) and 128-row tile, so a wrong tile cannot hide in the tensor norm
    B, N, Hx, _ = r.shape
    for b in range(B):
        for h in range(Hx):
            for t0 in range(0, N, 128):
                rr = r[b, t0:t0 + 128, h]
                nr = np.linalg.norm(rr)
                if nr > 0:
                    e = np.linalg.norm(g[b, t0:t0 + 128, h] - rr) / nr
                    assert e <= 3e-2, f"{what}: tile (b{b} h{h} rows {t0}) relative L2 {e:.3e}"


@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES)
def test_fused_backward_matches_oracle(oracle_mod, B, N, H, Hkv, causal):
    d = 128
    seed = 8100 + N + H + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    split = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    fused = fa.attention_bwd_fused(q, k, v, o, lse, dO, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), scale, causal)
    what = f"fused B{B} N{N} H{H}/{Hkv} causal={causal}"
    for name, g, r in zip(("dQ", "dK", "dV"), fused, ref):
        check_grad(g.cpu(), r, f"{what} {name}")
        if np.linalg.norm(r) > 0:
            tile_rel_l2(g.float().cpu().numpy(), r, f"{what} {name}")
    for name, a, b in zip(("dK", "dV"), fused[1:], split[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what}: {name} differs from fa_bwd"


def test_fused_backward_outliers(oracle_mod):
    w = inputs.Workload("outliers", 1, 2, 2, 640, 128, True, 9, outliers=True)
    x = inputs.make_inputs(w, device="cuda")
    o, lse = fa.attention_fwd(x["q"], x["k"], x["v"], scale=w.sm_scale, causal=True)
    got = fa.attention_bwd_fused(x["q"], x["k"], x["v"], o, lse, x["dO"], scale=w.sm_scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(*(x[n].cpu() for n in ("q", "k", "v", "dO")), w.sm_scale, True)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        check_grad(g.cpu(), r, f"fused outliers {name}")


def test_fused_rejects_other_head_dims_and_small_workspaces():
    A = 0x10000
    assert fa.fa_bwd_fused_workspace_bytes(1, 2, 2, 256, 64) == 0
    assert fa.fa_bwd_fused(A, A, A, A, A, A, A, A, A, 1, 2, 2, 256, 64, 0.1, 0, A, 1 << 20, 0) == fa.FA_ERR_UNSUPPORTED
    nb = fa.fa_bwd_fused_workspace_bytes(1, 2, 2, 256, 128)
    assert nb == fa.fa_bwd_workspace_bytes(1, 2, 2, 256, 128) + 256 * 2 * 128 * 4
    assert fa.fa_bwd_fused(A, A, A, A, A, A, A, A, A, 1, 2, 2, 256, 128, 0.1, 0, A, nb - 1, 0) == fa.FA_ERR_WORKSPACE
