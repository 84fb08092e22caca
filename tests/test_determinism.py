"""Run-to-run reproducibility.

The backward has no atomics: dK/dV come from a key/value-stationary kernel and
dQ from a query-stationary one, each summing in a fixed order (the pages'
deterministic backward mode, FA4 paper summary, section 3).  So repeated calls
on the same inputs must give the same bits, and the staged entry points
(fa_bwd_prepare, fa_bwd_dkdv, fa_bwd_dq) must give exactly what fa_bwd gives.
The forward is checked the same way.
"""
import math

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [
    # B, N, H, Hkv, d, causal
    (2, 1000, 4, 2, 128, True),
    (1, 2048, 2, 2, 128, False),
    (2, 700, 4, 4, 64, False),
    (1, 600, 2, 1, 256, True),
]


def same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", CASES)
def test_repeat_calls_are_bitwise_equal(B, N, H, Hkv, d, causal):
    seed = 7000 + N + d
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    runs = []
    for _ in range(3):
        o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
        runs.append((o, lse) + fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    names = ("O", "LSE", "dQ", "dK", "dV")
    for r in runs[1:]:
        for name, a, b in zip(names, runs[0], r):
            assert same_bits(a, b), f"{name} differs between calls"


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", CASES)
def test_staged_entry_points_match_fa_bwd(B, N, H, Hkv, d, causal):
    seed = 7100 + N + d
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    ref = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    nb = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert fa.fa_bwd_prepare(o, lse, dO, B, H, Hkv, N, d, ws, nb) == fa.FA_OK
    assert fa.fa_bwd_dkdv(q, k, v, dO, dk, dv, B, H, Hkv, N, d, scale, causal, ws, nb) == fa.FA_OK
    assert fa.fa_bwd_dq(q, k, v, dO, dq, B, H, Hkv, N, d, scale, causal, ws, nb) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert same_bits(a, b), f"{name}: staged entry points differ from fa_bwd"
