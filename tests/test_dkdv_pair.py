"""dK/dV on CTA pairs (tcgen05 cta_group::2) against dK/dV on single CTAs.

At head dim 128 the default library computes dK and dV with cluster pairs of
CTAs sharing one 256-row key tile, each M = 256 MMA reading half of its B
operand from each CTA (FlashAttention-4 paper summary, section 2.C), for
sequences longer than 2048 rows (4096 causal); shorter ones run the one-CTA
kernel, measured faster there.  The tests below use short shapes, so the
default library runs the one-CTA kernel and a build with both thresholds at 0
runs the pair; both must match the oracle, and they must give bitwise equal dK
and dV on shapes whose last key tile has no partner (odd tile counts), whose
partner lies wholly past the end of the sequence, under the causal mask (the
pair's second tile sees a query tile that it must mask whole) and with GQA.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_grad

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


PAIR_ALWAYS = ["-DFA_DKDV_PAIR_MIN_N=0", "-DFA_DKDV_PAIR_MIN_N_CAUSAL=0"]


@pytest.fixture(scope="module")
def pair_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("pair") / "libfa_dkdv2.so")
    build.build(force=True, extra_flags=PAIR_ALWAYS, lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_bwd_workspace_bytes", "fa_bwd", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


CASES = [
    # B, N, H, Hkv, causal
    (1, 128, 2, 2, False),   # one key tile: its partner holds no rows
    (1, 384, 2, 2, True),    # three tiles: the last pair is half empty
    (2, 640, 4, 2, True),    # GQA, causal, odd tile count
    (1, 1000, 2, 1, False),  # ragged tail inside the second tile of a pair
    (1, 1, 1, 1, True),      # a single row
]


@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES)
def test_pair_and_single_cta_dkdv_agree_and_match_oracle(oracle_mod, pair_lib, B, N, H, Hkv, causal):
    d = 128
    seed = 7100 + N + H + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    one = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)  # short: the one-CTA kernel
    nb = pair_lib.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    pair = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = pair_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                         pair[0].data_ptr(), pair[1].data_ptr(), pair[2].data_ptr(), B, H, Hkv, N, d, scale,
                         int(causal), ws.data_ptr(), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert pair_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), scale, causal)
    what = f"B{B} N{N} H{H}/{Hkv} causal={causal}"
    for name, a, b, r in zip(("dQ", "dK", "dV"), pair, one, ref):
        check_grad(a.cpu(), r, f"pair {what} {name}")
        check_grad(b.cpu(), r, f"single {what} {name}")
        # dQ: the same kernel in both builds; dK, dV: the same MMAs on the same
        # bf16 operands in the same K order, whichever SM holds which rows
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"{what} {name}: pair and single CTA differ"


@pytest.fixture(scope="module")
def cluster_scope_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("clscope") / "libfa_clscope.so")
    build.build(force=True, extra_flags=["-DFA_PAIR_SCOPE_CLUSTER=1"] + PAIR_ALWAYS, lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_bwd_workspace_bytes", "fa_bwd", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


@pytest.mark.parametrize("B,N,H,Hkv,causal", [(1, 640, 2, 2, True), (2, 512, 4, 2, False)])
def test_cluster_scope_build_gives_the_same_bits(cluster_scope_lib, B, N, H, Hkv, causal):
    # the pair kernels' waits and remote arrives with explicit cluster scope
    # (a slower build) order the same data: the results must not change
    d = 128
    seed = 7300 + N + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    # the default library runs the one-CTA kernel at these lengths, bitwise equal to the pair
    ref = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    nb = cluster_scope_lib.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    got = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    assert cluster_scope_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    dO.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), B, H, Hkv,
                                    N, d, scale, int(causal), ws.data_ptr(), nb, None) == fa.FA_OK
    torch.cuda.synchronize()
    assert cluster_scope_lib.fa_last_device_status(None) == fa.FA_OK
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


# ---------------------------------------------------------------- head dim 256
# The default library computes the head-dim-256 backward with CTA pairs: dK, dV
# with 64 keys per CTA (M = 128 pair MMAs, K in tensor memory, P^T and dS^T in
# shared memory) and dQ with 64 query rows per CTA (Q, dO in tensor memory).  A
# build with FA_DKDV256_PAIR=0 and FA_DQ256_PAIR=0 keeps one CTA per (key tile,
# head-dim half) and one CTA per query tile.
@pytest.fixture(scope="module")
def onecta256_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("one256") / "libfa_one256.so")
    build.build(force=True, extra_flags=["-DFA_DKDV256_PAIR=0", "-DFA_DQ256_PAIR=0"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_bwd_workspace_bytes", "fa_bwd", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


CASES_256 = [
    # B, N, H, Hkv, causal
    (1, 64, 1, 1, False),    # the pair's second CTA holds no keys
    (1, 200, 2, 1, True),    # ragged tail in the second CTA of the last pair, GQA
    (2, 384, 2, 2, True),    # diagonal tiles: the second CTA's keys hide half the queries
    (1, 1, 1, 1, True),      # a single row
]


@pytest.mark.parametrize("B,N,H,Hkv,causal", CASES_256)
def test_d256_pair_and_one_cta_match_oracle(oracle_mod, onecta256_lib, B, N, H, Hkv, causal):
    d = 256
    seed = 7900 + N + H + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    pair = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    nb = onecta256_lib.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    one = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = onecta256_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              dO.data_ptr(), one[0].data_ptr(), one[1].data_ptr(), one[2].data_ptr(), B, H, Hkv, N, d,
                              scale, int(causal), ws.data_ptr(), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert onecta256_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), scale, causal)
    what = f"d256 B{B} N{N} H{H}/{Hkv} causal={causal}"
    for name, a, b, r in zip(("dQ", "dK", "dV"), pair, one, ref):
        check_grad(a.cpu(), r, f"pair {what} {name}")
        check_grad(b.cpu(), r, f"one CTA {what} {name}")
