"""The allocation-free backward entry point, fa_bwd_noalloc.

It exists for callers that cannot allocate device memory when they run the
backward pass (a plug-in inside a host framework that owns every device
allocation through its own pool, or a loop that forbids cudaMalloc after
start-up).  It must give what fa_bwd gives with a caller-provided workspace.
This file is collected last on purpose, and it also passes alone in a fresh
process.
"""
import math

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs
from helpers import rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-2  # the backward tolerance of the parity tests (relative L2)


def make(B, N, H, Hkv, d, seed):
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    return q, k, v, dO


def compare_once(B, N, H, Hkv, d, causal, seed):
    q, k, v, dO = make(B, N, H, Hkv, d, seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    ref = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    got = [torch.full_like(t, float("nan")) for t in ref]  # every element must be written
    st = fa.fa_bwd_noalloc(q, k, v, o, lse, dO, got[0], got[1], got[2], B, H, Hkv, N, d, scale, causal)
    assert st == fa.FA_OK, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.isfinite(g.float()).all(), name
        rn = r.float().cpu().numpy()
        assert rel_l2(g, rn) <= TOL, (name, rel_l2(g, rn))


def test_matches_workspace_backward_on_two_calls_in_a_row():
    # the second call reuses the scratch the first one left behind, with a
    # different shape (more rows, GQA, non-causal)
    compare_once(1, 700, 4, 2, 128, True, 5100)
    compare_once(2, 1024, 4, 4, 64, False, 5200)


def test_rejects_sizes_beyond_the_builtin_scratch():
    B, H, Hkv, N, d = 64, 64, 64, 8192, 128
    assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d) > fa.FA_BWD_NOALLOC_SCRATCH_BYTES
    a = 0x10000  # never dereferenced: the size check comes before any launch
    st = fa.fa_bwd_noalloc(a, a, a, a, a, a, a, a, a, B, H, Hkv, N, d, 0.088, 0)
    assert st == fa.FA_ERR_WORKSPACE
