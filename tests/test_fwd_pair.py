"""The CTA-pair forward against the one-CTA forward, at head dims 256 and 128.

At head dim 256 the default library runs the forward on clusters of two CTAs
that share 256 query rows (128 each): M = 256 `cta_group::2` MMAs, each CTA
loading half of K_j (64 key rows) and half of V_j (half the head dim), S
double-buffered in TMEM (FA4 paper summary, section 2.C).  At head dim 128 the
default keeps two query tiles per CTA (the pair form measured slower there).
One variant build swaps both (FA_FWD256_PAIR=0, FA_FWD128_PAIR=1).  Every form
must match the oracle on shapes whose pair's second tile is empty or ragged,
under the causal mask (the pair's first tile masks the last key block whole),
with GQA, for a single row and on packed batches.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_lse, check_o

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def variant_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("fwdv") / "libfa_fwdv.so")
    build.build(force=True, extra_flags=["-DFA_FWD256_PAIR=0", "-DFA_FWD128_PAIR=1"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_fwd_varlen", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


CASES = [
    # B, N, H, Hkv, causal
    (1, 128, 2, 2, False),   # one query tile: the pair's second is empty
    (1, 384, 2, 1, True),    # three tiles: the last pair is half empty; GQA
    (2, 300, 4, 2, True),    # ragged tail in the pair's second tile
    (1, 1000, 2, 2, False),  # ragged, several pairs
    (1, 1, 1, 1, True),      # a single row
]


@pytest.mark.parametrize("d", [256, 128])
@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES)
def test_default_and_variant_forward_match_oracle(oracle_mod, variant_lib, d, B, N, H, Hkv, causal):
    seed = 8100 + N + H + causal + d
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    o1, lse1 = torch.empty_like(q), torch.empty_like(lse)
    assert variant_lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), lse1.data_ptr(), B, H, Hkv,
                               N, d, scale, int(causal), None) == fa.FA_OK
    torch.cuda.synchronize()
    assert variant_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle_mod.attention_fwd(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    what = f"d{d} B{B} N{N} H{H}/{Hkv} causal={causal}"
    for name, oo, ll in (("default", o, lse), ("variant", o1, lse1)):
        check_o(oo.float().cpu().numpy().astype(np.float64), o_ref, f"{name} {what}")
        check_lse(ll.cpu().numpy().astype(np.float64), lse_ref, f"{name} {what}")


@pytest.mark.parametrize("causal", [False, True])
def test_pair_forward_packed_batch(oracle_mod, causal):
    # empty, one-row and tile-edge sequences; rows after the batch must stay untouched
    lens, H, Hkv, d = [1, 127, 128, 129, 300, 0, 513], 4, 2, 256
    total = sum(lens)
    seed = 8300 + causal
    q = inputs.random_bf16((total, H, d), seed, "cuda")
    k = inputs.random_bf16((total, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((total, Hkv, d), seed + 2, "cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    buf = torch.full((total + 5, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal, out=buf[:total])
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert (buf[total:] == 7.0).all(), "rows past the packed batch were written"
    o_ref, lse_ref = oracle_mod.attention_fwd_varlen(q, k, v, cu, scale, causal)
    check_o(o, o_ref, f"packed d256 causal={causal}")
    check_lse(lse, lse_ref, f"packed d256 causal={causal}")
