"""dQ on CTA pairs (tcgen05 cta_group::2), the build option FA_DQ_PAIR=1.

The default library computes dQ at head dim 128 with one CTA per 128-row query
tile.  The pair form lets two CTAs of a cluster share one 256-row query tile:
each M = 256 MMA reads half of every K and V tile from each CTA (FlashAttention-4
paper summary, section 2.C).  It measured slower than the one-CTA kernel on
GB300 except at the longest causal sequences, so it is not the default, but it
stays built and tested: it must match the oracle and give the same bits as the
default library on shapes whose last query tile has no partner, whose partner
lies wholly past the end, under the causal mask, with GQA and in packed batches.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_grad

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def pair_dq_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("dqpair") / "libfa_dqpair.so")
    build.build(force=True, extra_flags=["-DFA_DQ_PAIR=1"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_varlen", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


CASES = [
    # B, N, H, Hkv, causal
    (1, 128, 2, 2, False),   # one query tile: its partner holds no rows
    (1, 384, 2, 2, True),    # three tiles: the last pair is half empty
    (2, 640, 4, 2, True),    # GQA, causal, odd tile count
    (1, 1000, 2, 1, False),  # ragged tail inside the second tile of a pair
    (2, 1024, 2, 2, True),   # whole pairs under the causal mask
    (1, 1, 1, 1, True),      # a single row
]


@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES)
def test_pair_dq_matches_oracle_and_default_bits(oracle_mod, pair_dq_lib, B, N, H, Hkv, causal):
    d = 128
    seed = 7500 + N + H + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    default = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    nb = pair_dq_lib.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = pair_dq_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                            got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), B, H, Hkv, N, d, scale,
                            int(causal), ws.data_ptr(), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert pair_dq_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), scale, causal)
    what = f"B{B} N{N} H{H}/{Hkv} causal={causal}"
    check_grad(got[0].cpu(), ref[0], f"pair dQ {what}")
    # the same MMAs on the same bf16 operands in the same key order, whichever
    # SM holds which query rows; dK and dV come from the same kernel in both builds
    for name, a, b in zip(("dQ", "dK", "dV"), got, default):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what} {name}: pair and default differ"


@pytest.mark.parametrize("causal", [False, True])
def test_pair_dq_packed_batch(oracle_mod, pair_dq_lib, causal):
    # empty, one-row and tile-edge sequences; each sequence's query tiles pair up on their own
    lens, H, Hkv, d = [1, 127, 128, 129, 300, 0, 513], 4, 2, 128
    total = sum(lens)
    seed = 7700 + causal
    q = inputs.random_bf16((total, H, d), seed, "cuda")
    k = inputs.random_bf16((total, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((total, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((total, H, d), seed + 3, "cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal)
    default = fa.attention_bwd_varlen(q, k, v, o, lse, dO, cu, max(lens), scale=scale, causal=causal)
    nb = pair_dq_lib.fa_bwd_workspace_bytes(len(lens), H, Hkv, max(lens), d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    # seven sentinel rows after the packed batch: nothing may be written there
    buf = torch.full((total + 7, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = buf[:total], torch.empty_like(k), torch.empty_like(v)
    P = lambda t: t.data_ptr()
    st = pair_dq_lib.fa_bwd_varlen(P(q), P(k), P(v), P(o), P(lse), P(dO), P(dq), P(dk), P(dv), P(cu), len(lens),
                                   max(lens), total, H, Hkv, d, scale, int(causal), P(ws), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert pair_dq_lib.fa_last_device_status(None) == fa.FA_OK
    assert (buf[total:] == 7.0).all(), "rows past the packed batch were written"
    ref = oracle_mod.attention_bwd_varlen(q, k, v, dO, cu, scale, causal)
    bounds = np.concatenate([[0], np.cumsum(lens)])
    for s_, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        if b > a:
            check_grad(dq[a:b], ref[0][a:b], f"pair dQ causal={causal} seq {s_} ({b - a} rows)")
    assert torch.equal(dq.view(torch.int16), default[0].view(torch.int16)), "packed dQ: pair and default differ"
