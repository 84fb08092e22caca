"""dK/dV on CTA pairs (tcgen05 cta_group::2) against dK/dV on single CTAs.

At head dim 128 the default library computes dK and dV with cluster pairs of
CTAs sharing one 256-row key tile, each M = 256 MMA reading half of its B
operand from each CTA (FlashAttention-4 paper summary, section 2.C).  A build
with FA_DKDV_PAIR=0 keeps the one-CTA kernel; both must match the oracle, and
they must agree with each other to the backward tolerance on shapes whose last
key tile has no partner (odd tile counts), whose partner lies wholly past the
end of the sequence, under the causal mask (the pair's second tile sees a
query tile that it must mask whole) and with GQA.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_grad, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def single_cta_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("single") / "libfa_dkdv1.so")
    build.build(force=True, extra_flags=["-DFA_DKDV_PAIR=0"], lib_path=path)
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
def test_pair_and_single_cta_dkdv_agree_and_match_oracle(oracle_mod, single_cta_lib, B, N, H, Hkv, causal):
    d = 128
    seed = 7100 + N + H + causal
    q = inputs.random_bf16((B, N, H, d), seed, "cuda")
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1, "cuda")
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2, "cuda")
    dO = inputs.random_bf16((B, N, H, d), seed + 3, "cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    pair = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    nb = single_cta_lib.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    one = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    st = single_cta_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                               one[0].data_ptr(), one[1].data_ptr(), one[2].data_ptr(), B, H, Hkv, N, d, scale,
                               int(causal), ws.data_ptr(), nb, None)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert single_cta_lib.fa_last_device_status(None) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), scale, causal)
    what = f"B{B} N{N} H{H}/{Hkv} causal={causal}"
    for name, a, b, r in zip(("dQ", "dK", "dV"), pair, one, ref):
        check_grad(a.cpu(), r, f"pair {what} {name}")
        check_grad(b.cpu(), r, f"single {what} {name}")
        if name == "dQ":  # the same dQ kernel in both builds
            assert torch.equal(a, b), f"{what} dQ"
        else:
            rn = b.float().cpu().numpy()
            if (rn != 0).any():
                assert rel_l2(a, rn) <= 1e-2, (what, name, rel_l2(a, rn))
            print(f"{what} {name}: pair vs single bitwise equal = {torch.equal(a, b)}")
