"""Packed variable-length batches (cu_seqlens) against the fp64 oracle, which
solves each sequence as its own single-sequence problem.

The length mixes cover empty sequences, one-row sequences, exact multiples of
the 128-row tile, one row past a tile, and sequences that end mid-tile next to
a following sequence.  The output tensor has sentinel rows after `total`: the
kernels must write nothing past the packed rows.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs
from helpers import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu

SENTINEL_ROWS = 131

FWD_CASES = [
    # lengths, H, Hkv, d, causal
    ([1, 127, 128, 129, 300, 0, 513], 4, 2, 128, False),
    ([1, 127, 128, 129, 300, 0, 513], 4, 2, 128, True),
    ([700, 3, 256], 2, 2, 128, True),
    ([5, 200, 64, 385], 2, 2, 64, False),
    ([5, 200, 64, 385], 4, 1, 64, True),
    ([333, 17, 256], 2, 1, 256, False),
    ([333, 17, 256], 2, 2, 256, True),
]


def pack(lens, H, Hkv, d, seed, with_dO=False):
    total = sum(lens)
    q = inputs.random_bf16((total, H, d), seed, "cuda")
    k = inputs.random_bf16((total, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((total, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((total, H, d), seed + 3, "cuda") if with_dO else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    return q, k, v, dO, cu, total


def with_sentinel(shape_rows, H, d):
    buf = torch.full((shape_rows + SENTINEL_ROWS, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    return buf, buf[:shape_rows]


@pytest.mark.parametrize("lens,H,Hkv,d,causal", FWD_CASES)
def test_fwd_matches_oracle(oracle_mod, lens, H, Hkv, d, causal):
    q, k, v, _, cu, total = pack(lens, H, Hkv, d, 9000 + sum(lens) + d + causal)
    scale = 1.0 / math.sqrt(d)
    buf, o = with_sentinel(total, H, d)
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal, out=o)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert (buf[total:] == 7.0).all(), "rows past the packed batch were written"
    o_ref, lse_ref = oracle_mod.attention_fwd_varlen(q, k, v, cu, scale, causal)
    what = f"lens {lens} H{H}/{Hkv} d{d} causal={causal}"
    check_o(o, o_ref, what)
    check_lse(lse, lse_ref, what)


@pytest.mark.parametrize("d,causal", [(128, False), (128, True), (64, True), (256, False)])
def test_equal_lengths_match_the_fixed_length_path_bitwise(d, causal):
    B, N, H, Hkv = 3, 300, 4, 2
    q = inputs.random_bf16((B, N, H, d), 9100 + d, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), 9101 + d, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), 9102 + d, "cuda")
    o, lse = fa.attention_fwd(q, k, v, causal=causal)
    cu = torch.arange(B + 1, dtype=torch.int32, device="cuda") * N
    ov, lv = fa.attention_fwd_varlen(q.reshape(B * N, H, d), k.reshape(B * N, Hkv, d), v.reshape(B * N, Hkv, d), cu,
                                     N, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(ov.view(torch.int16), o.reshape(B * N, H, d).view(torch.int16))
    assert torch.equal(lv.view(torch.int32), lse.permute(1, 0, 2).reshape(H, B * N).view(torch.int32))


def test_empty_batch_launches_nothing():
    A = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(3, dtype=torch.int32, device="cuda")
    assert fa.fa_fwd_varlen(A, A, A, A, None, cu, 2, 128, 0, 2, 2, 128, 0.1, 0) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK


BWD_CASES = [
    # lengths, H, Hkv, d, causal
    ([1, 127, 128, 129, 300, 0, 513], 4, 2, 128, False),
    ([1, 127, 128, 129, 300, 0, 513], 4, 2, 128, True),
    ([5, 200, 64, 385], 2, 2, 64, True),
    ([333, 17, 256], 2, 1, 256, True),
    ([333, 17, 256], 2, 2, 256, False),
    # 40 sequences of 0-299 rows at head dim 64: 240 key-tile units, many past
    # their sequence, on persistent dK/dV CTAs that each run several
    ([(37 * i * i + 11 * i) % 300 for i in range(40)], 4, 2, 64, True),
]


@pytest.mark.parametrize("lens,H,Hkv,d,causal", BWD_CASES)
def test_bwd_matches_oracle(oracle_mod, lens, H, Hkv, d, causal):
    q, k, v, dO, cu, total = pack(lens, H, Hkv, d, 9500 + sum(lens) + d + causal, with_dO=True)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal)
    # sentinel rows after `total` in every gradient: nothing may be written there
    bufs = [with_sentinel(total, q.shape[1], d), with_sentinel(total, k.shape[1], d), with_sentinel(total, k.shape[1], d)]
    nbytes = fa.fa_bwd_workspace_bytes(len(lens), H, Hkv, max(lens), d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dq, dk, dv = (b[1] for b in bufs)
    st = fa.fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu, len(lens), max(lens), total, H, Hkv, d, scale, causal,
                          ws, nbytes)
    assert st == fa.FA_OK, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for name, (buf, _) in zip(("dQ", "dK", "dV"), bufs):
        assert (buf[total:] == 7.0).all(), f"{name}: rows past the packed batch were written"
    ref = oracle_mod.attention_bwd_varlen(q, k, v, dO, cu, scale, causal)
    bounds = np.concatenate([[0], np.cumsum(lens)])
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        for s_, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
            if b > a:  # per sequence, so one sequence cannot hide in the others' norm
                check_grad(g[a:b], r[a:b], f"lens {lens} d{d} causal={causal} seq {s_} ({b - a} rows) {name}")


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (256, True)])
def test_bwd_equal_lengths_match_the_fixed_length_path_bitwise(d, causal):
    B, N, H, Hkv = 2, 300, 4, 2
    q = inputs.random_bf16((B, N, H, d), 9600 + d, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), 9601 + d, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), 9602 + d, "cuda")
    dO = inputs.random_bf16((B, N, H, d), 9603 + d, "cuda")
    o, lse = fa.attention_fwd(q, k, v, causal=causal)
    ref = fa.attention_bwd(q, k, v, o, lse, dO, causal=causal)
    cu = torch.arange(B + 1, dtype=torch.int32, device="cuda") * N
    flat = lambda x: x.reshape(B * N, x.shape[2], d)
    lse_v = lse.permute(1, 0, 2).reshape(H, B * N).contiguous()
    got = fa.attention_bwd_varlen(flat(q), flat(k), flat(v), flat(o), lse_v, flat(dO), cu, N, causal=causal)
    torch.cuda.synchronize()
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(a.view(torch.int16), flat(b).view(torch.int16)), name
