"""Persistent CTAs against one CTA (or CTA pair) per tile.

The default library runs the one-CTA dK/dV kernel (head dim 64, and 128 up to
the lengths where the CTA pairs take over), the dQ kernel (head dims 64 and
128) and the head-dim-256 CTA-pair forward on at most one CTA (pair) per SM
(pair), each taking tile units blockIdx.x, blockIdx.x + gridDim.x, ... and
carrying its rings, TMEM buffers and barrier phases from one unit into the
next (dK/dV: the next unit's K and V load as soon as the last MMA that read
the previous ones completes; dQ: the next unit's Q and dO follow this unit's
last K and V in the ring; pair forward: each CTA loads its next Q tile once the
unit's last S has read the previous one).  Epilogues without a stage of their own write each
row straight to global memory.  Some long causal shapes run one CTA per unit
instead.  A build with every threshold at 0 runs every shape one CTA per
unit.  Both must match the oracle, and they must give bitwise equal
gradients: each unit's MMAs see the same bf16 operands in the same order
whichever CTA runs it.  The shapes give block 0 several units (more units than
SMs), with GQA, ragged tails, the causal mask and a packed batch whose short
sequences leave many units with no rows.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_grad, check_lse, check_o

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def one_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("onecta") / "libfa_onecta.so")
    build.build(force=True, extra_flags=["-DFA_DKDV_PERSIST_MAX_N=0", "-DFA_DKDV_PERSIST_MAX_N_CAUSAL=0",
                                         "-DFA_DKDV128_PERSIST_MAX_N=0", "-DFA_DKDV128_PERSIST_MAX_N_CAUSAL=0",
                                         "-DFA_DQ_PERSIST_MAX_N=0", "-DFA_DQ_PERSIST_MAX_N_CAUSAL=0",
                                         "-DFA_DQ128_PERSIST_MAX_N=0", "-DFA_DQ128_PERSIST_MAX_N_CAUSAL=0",
                                         "-DFA_FWD_PAIR_PERSIST_MAX_N=0", "-DFA_FWD_PAIR_PERSIST_MAX_N_CAUSAL=0"],
                lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_fwd_varlen", "fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_varlen",
                 "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


CASES = [
    # B, N, H, Hkv, causal: (N / 128 rounded up) * B * Hkv key-tile units, * B * H query-tile units
    (8, 333, 8, 8, False),   # 192 units, ragged last tile
    (8, 333, 16, 8, True),   # 192 units, GQA groups of two, causal
    (16, 640, 4, 2, True),   # 160 units of 1-5 query tiles each
    (1, 1, 1, 1, True),      # one row, one unit
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES)
def test_persistent_and_one_cta_agree_and_match_oracle(oracle_mod, one_lib, B, N, H, Hkv, causal, d):
    seed = 7300 + N + H + causal + d
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    pers = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    nb = one_lib.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    one = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = one_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                        one[0].data_ptr(), one[1].data_ptr(), one[2].data_ptr(), B, H, Hkv, N, d, scale, int(causal),
                        ws.data_ptr(), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert one_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), scale, causal)
    what = f"B{B} N{N} H{H}/{Hkv} causal={causal}"
    for name, a, b, r in zip(("dQ", "dK", "dV"), pers, one, ref):
        check_grad(a.cpu(), r, f"persistent {what} {name}")
        check_grad(b.cpu(), r, f"one CTA per unit {what} {name}")
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what} {name}: persistent and one-CTA differ"


@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False)])
def test_persistent_packed_batch_matches_one_cta(oracle_mod, one_lib, d, causal):
    lens = [(37 * i * i + 11 * i) % 300 for i in range(40)]  # 0-276 rows: 240 units, many past their sequence
    H, Hkv = 4, 2
    total = sum(lens)
    q = inputs.random_bf16((total, H, d), 7400 + d, "cuda")
    k = inputs.random_bf16((total, Hkv, d), 7401 + d, "cuda")
    v = inputs.random_bf16((total, Hkv, d), 7402 + d, "cuda")
    dO = inputs.random_bf16((total, H, d), 7403 + d, "cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal)
    pers = fa.attention_bwd_varlen(q, k, v, o, lse, dO, cu, max(lens), scale=scale, causal=causal)
    nb = one_lib.fa_bwd_workspace_bytes(len(lens), H, Hkv, max(lens), d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    one = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = one_lib.fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                               one[0].data_ptr(), one[1].data_ptr(), one[2].data_ptr(), cu.data_ptr(), len(lens),
                               max(lens), total, H, Hkv, d, scale, int(causal), ws.data_ptr(), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert one_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd_varlen(q, k, v, dO, cu, scale, causal)
    for name, a, b, r in zip(("dQ", "dK", "dV"), pers, one, ref):
        check_grad(a, r, f"packed persistent d{d} causal={causal} {name}")
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), \
            f"packed d{d} causal={causal} {name}: persistent and one-CTA differ"


PAIR_FWD_CASES = [
    # B, N, H, Hkv, causal: (N / 256 rounded up) * B * H units on at most 76 clusters
    (4, 640, 8, 4, False),  # 96 units; the last pair's second tile half empty
    (4, 640, 8, 4, True),
    (1, 1, 1, 1, True),
]


@pytest.mark.parametrize("B,N,H,Hkv,causal", PAIR_FWD_CASES)
def test_persistent_pair_forward_matches_one_cluster_per_unit(oracle_mod, one_lib, B, N, H, Hkv, causal):
    d = 256
    seed = 7700 + N + H + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    o1, lse1 = torch.empty_like(o), torch.empty_like(lse)
    assert one_lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), lse1.data_ptr(), B, H, Hkv, N, d,
                          scale, int(causal), None) == fa.FA_OK
    torch.cuda.synchronize()
    assert one_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    what = f"d256 B{B} N{N} H{H}/{Hkv} causal={causal}"
    assert torch.equal(o.view(torch.int16), o1.view(torch.int16)), f"{what}: O differs"
    assert torch.equal(lse, lse1), f"{what}: LSE differs"
    o_ref, lse_ref = oracle_mod.attention_fwd(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    check_o(o, o_ref, what)
    check_lse(lse, lse_ref, what)


@pytest.mark.parametrize("causal", [False, True])
def test_persistent_pair_forward_packed_batch(oracle_mod, one_lib, causal):
    lens = [(37 * i * i + 11 * i) % 700 for i in range(40)]  # 0-698 rows: 240 units, many past their sequence
    H, Hkv, d = 2, 1, 256
    total = sum(lens)
    q = inputs.random_bf16((total, H, d), 7800, "cuda")
    k = inputs.random_bf16((total, Hkv, d), 7801, "cuda")
    v = inputs.random_bf16((total, Hkv, d), 7802, "cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, max(lens), scale=scale, causal=causal)
    o1, lse1 = torch.empty_like(o), torch.empty_like(lse)
    assert one_lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), lse1.data_ptr(),
                                 cu.data_ptr(), len(lens), max(lens), total, H, Hkv, d, scale, int(causal),
                                 None) == fa.FA_OK
    torch.cuda.synchronize()
    assert one_lib.fa_last_device_status(None) == fa.FA_OK
    assert torch.equal(o.view(torch.int16), o1.view(torch.int16)), "packed d256: O differs"
    assert torch.equal(lse, lse1), "packed d256: LSE differs"
    o_ref, lse_ref = oracle_mod.attention_fwd_varlen(q, k, v, cu, scale, causal)
    check_o(o, o_ref, f"packed d256 causal={causal}")
    check_lse(lse, lse_ref, f"packed d256 causal={causal}")
