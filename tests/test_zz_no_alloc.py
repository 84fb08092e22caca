"""The allocation-free backward entry point, fa_bwd_noalloc.

Some callers cannot allocate device memory when they run the backward pass: a
plug-in inside a host framework that owns every device allocation through its
own pool, or a training or serving loop that forbids cudaMalloc after start-up
(it synchronises the device and fragments memory).  fa_bwd_noalloc serves them
with a scratch array built into the library; it runs the same kernels as
fa_bwd, so its results must be bitwise those of fa_bwd with a workspace.

The file name makes pytest collect it last, so that a run which stops at the
first failure has already run every other test.  It depends on no other test
and also passes alone in a fresh process.
"""
import math

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs

pytestmark = pytest.mark.gpu


def make(B, N, H, Hkv, d, causal, seed):
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    o, lse = fa.attention_fwd(q, k, v, scale=1.0 / math.sqrt(d), causal=causal)
    return q, k, v, o, lse, dO


def noalloc(x, out, B, N, H, Hkv, d, causal):
    q, k, v, o, lse, dO = x
    st = fa.fa_bwd_noalloc(q, k, v, o, lse, dO, out[0], out[1], out[2], B, H, Hkv, N, d, 1.0 / math.sqrt(d), causal)
    assert st == fa.FA_OK, fa.status_string(st)


def compare_once(B, N, H, Hkv, d, causal, seed):
    x = make(B, N, H, Hkv, d, causal, seed)
    q, k, v, o, lse, dO = x
    ref = fa.attention_bwd(q, k, v, o, lse, dO, scale=1.0 / math.sqrt(d), causal=causal)
    got = [torch.full_like(t, float("nan")) for t in ref]  # every element must be written
    noalloc(x, got, B, N, H, Hkv, d, causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(g.view(torch.int16), r.view(torch.int16)), f"{name} differs from fa_bwd"


def test_matches_workspace_backward_bitwise_on_two_calls_in_a_row():
    # the second call reuses the scratch the first one left behind, with a
    # different shape (more rows, GQA, non-causal, another head dim)
    compare_once(1, 700, 4, 2, 128, True, 5100)
    compare_once(2, 1024, 4, 4, 64, False, 5200)


def test_allocates_no_device_memory():
    B, N, H, Hkv, d = 1, 512, 2, 2, 128
    x = make(B, N, H, Hkv, d, True, 5300)
    out = [torch.empty_like(x[0]), torch.empty_like(x[1]), torch.empty_like(x[2])]
    noalloc(x, out, B, N, H, Hkv, d, True)  # first call on the device: address look-up, kernel loading
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    noalloc(x, out, B, N, H, Hkv, d, True)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert fa.fa_last_device_status() == fa.FA_OK


def test_rejects_sizes_beyond_the_builtin_scratch():
    B, H, Hkv, N, d = 64, 64, 64, 8192, 128
    assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d) > fa.fa_bwd_noalloc_scratch_bytes()
    a = 0x10000  # never dereferenced: the size check comes before any launch
    st = fa.fa_bwd_noalloc(a, a, a, a, a, a, a, a, a, B, H, Hkv, N, d, 0.088, 0)
    assert st == fa.FA_ERR_WORKSPACE
