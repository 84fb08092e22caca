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
