"""Head-dim-64 forward: the two-tile form against the short form and the oracle.

At head dim 64 the library runs the forward in one of two forms: two query
tiles per CTA (each with its own S buffer in TMEM, the tiles' softmax and MMAs
interleaved), or, for sequences of at most 4096 rows, the short form of one
tile per CTA with two CTAs per SM.  The default library reaches the two-tile
form only above 4096 rows; a build with that limit at 0 takes it at every
length.  It must match the oracle and give bitwise the same O and LSE as the
default library: every row sees the same bf16 operands, the same MMAs and the
same exponent and rescale arithmetic whichever form runs it.  The shapes cover
ragged tails, the causal mask's extra key block on the second tile, a second
tile past the sequence, GQA, N = 1, packed batches and inputs whose outliers
force rescales of O.
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

D = 64


@pytest.fixture(scope="module")
def two_tile_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("twotile") / "libfa_twotile.so")
    build.build(force=True, extra_flags=["-DFA_FWD_SHORT_MAX_N_D64=0"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_fwd_varlen", "fa_last_device_status", "fa_rescale_count"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


def rescale_count(lib) -> int:
    c = ctypes.c_uint(0)
    assert lib.fa_rescale_count(None, ctypes.addressof(c)) == fa.FA_OK
    return int(c.value)


def fwd_two_tile(lib, q, k, v, scale, causal):
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, N, d, scale,
                      int(causal), None) == fa.FA_OK
    torch.cuda.synchronize()
    assert lib.fa_last_device_status(None) == fa.FA_OK
    return o, lse


CASES = [
    # B, N, H, Hkv, causal
    (2, 1000, 4, 2, False),  # 8 key blocks, ragged last one
    (2, 1000, 4, 2, True),   # tile 1 of each pair has one block more
    (1, 129, 2, 1, True),    # one row past the first tile
    (3, 200, 2, 2, False),
    (1, 100, 2, 2, False),   # the second tile lies past the sequence
    (1, 1, 1, 1, True),
    (1, 2048, 2, 2, True),   # 16 key blocks
]


@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES)
def test_two_tile_form_matches_oracle_and_short_form(oracle_mod, two_tile_lib, B, N, H, Hkv, causal):
    seed = 7900 + N + H + causal
    q = inputs.random_bf16((B, N, H, D), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, D), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, D), seed + 2, "cuda")
    scale = 1.0 / math.sqrt(D)
    o, lse = fwd_two_tile(two_tile_lib, q, k, v, scale, causal)
    o_ref, lse_ref = oracle_mod.attention_fwd(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    what = f"B{B} N{N} H{H}/{Hkv} causal={causal}"
    check_o(o.cpu(), o_ref, what)
    check_lse(lse.cpu(), lse_ref, what)
    o1, lse1 = fa.attention_fwd(q, k, v, scale=scale, causal=causal)  # the default library's form
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(o.view(torch.int16), o1.view(torch.int16)), f"{what}: O differs between the forms"
    assert torch.equal(lse, lse1), f"{what}: LSE differs between the forms"


@pytest.mark.parametrize("causal", [False, True])
def test_two_tile_form_rescales_with_outliers(oracle_mod, two_tile_lib, causal):
    """x20 outliers in Q and K move row maxima past the rescale threshold on later key blocks:
    the two-tile form rescales O and stays exact."""
    w = inputs.Workload("outliers d64", 1, 2, 2, 1536, D, causal, 11, outliers=True)
    x = inputs.make_inputs(w, device="cuda", with_dO=False)
    rescale_count(two_tile_lib)  # reset
    o, lse = fwd_two_tile(two_tile_lib, x["q"], x["k"], x["v"], w.sm_scale, causal)
    assert rescale_count(two_tile_lib) > 0
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), w.sm_scale, causal)
    check_o(o.cpu(), o_ref, w.name)
    check_lse(lse.cpu(), lse_ref, w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_two_tile_form_packed_batch(oracle_mod, two_tile_lib, causal):
    lens = [1, 127, 128, 129, 300, 0, 513, 1000, 64]
    H, Hkv = 4, 2
    total = sum(lens)
    q = inputs.random_bf16((total, H, D), 7950 + causal, "cuda")
    k = inputs.random_bf16((total, Hkv, D), 7951 + causal, "cuda")
    v = inputs.random_bf16((total, Hkv, D), 7952 + causal, "cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device="cuda")
    assert two_tile_lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      cu.data_ptr(), len(lens), max(lens), total, H, Hkv, D, scale, int(causal),
                                      None) == fa.FA_OK
    torch.cuda.synchronize()
    assert two_tile_lib.fa_last_device_status(None) == fa.FA_OK
    o_ref, lse_ref = oracle_mod.attention_fwd_varlen(q, k, v, cu, scale, causal)
    what = f"packed d64 causal={causal}"
    check_o(o, o_ref, what)
    check_lse(lse, lse_ref, what)
    o1, lse1 = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o1.view(torch.int16)), f"{what}: O differs between the forms"
    assert torch.equal(lse, lse1), f"{what}: LSE differs between the forms"
