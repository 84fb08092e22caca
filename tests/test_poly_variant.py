"""The software exp2 mixed with MUFU.EX2 inside the kernels (FlashAttention-4
paper summary, section 2.B: part of the exponentials emulated on the FMA pipe).
The default build takes every exponential on MUFU (measured faster on this
part); a build with FA_FWD_POLY_PER16 = FA_BWD_POLY_PER16 = 6 takes 6 of every 16
columns through the polynomial in the forward and the dK/dV kernels, and must
still match the oracle within the same tolerances."""
import ctypes

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_grad, check_lse, check_o

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def poly_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("poly") / "libfa_poly6.so")
    build.build(force=True, extra_flags=["-DFA_FWD_POLY_PER16=6", "-DFA_BWD_POLY_PER16=6"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_bwd_workspace_bytes", "fa_bwd", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


@pytest.mark.parametrize("B,N,H,d,causal", [(1, 300, 2, 128, True), (2, 256, 2, 64, False), (1, 513, 1, 128, False)])
def test_mixed_exp2_build_matches_oracle(oracle_mod, poly_lib, B, N, H, d, causal):
    w = inputs.Workload("poly", B, H, H, N, d, causal, 4242 + N)
    x = inputs.make_inputs(w, device="cuda")
    q, k, v, dO = x["q"], x["k"], x["v"], x["dO"]
    o, lse = torch.empty_like(q), torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    assert poly_lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H, N, d,
                           w.sm_scale, int(causal), None) == fa.FA_OK
    nb = poly_lib.fa_bwd_workspace_bytes(B, H, H, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert poly_lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H, N, d, w.sm_scale, int(causal),
                           ws.data_ptr(), nb, None) == fa.FA_OK
    torch.cuda.synchronize()
    assert poly_lib.fa_last_device_status(None) == fa.FA_OK
    qc, kc, vc, dOc = (t.cpu() for t in (q, k, v, dO))
    o_ref, lse_ref = oracle_mod.attention_fwd(qc, kc, vc, w.sm_scale, causal)
    what = f"poly6 B{B} N{N} H{H} d{d} causal={causal}"
    check_o(o, o_ref, what)
    check_lse(lse, lse_ref, what)
    grads = oracle_mod.attention_bwd(qc, kc, vc, dOc, w.sm_scale, causal)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), grads):
        check_grad(g.cpu(), r, f"{what} {name}")
