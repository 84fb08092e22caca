"""The conditional O rescale (FlashAttention-4 paper summary, section 2.B) is
exact for any threshold tau: O and the row sum share the stale maximum, and
O / l and m + log2 l are what is stored.  A library built with tau = 0 (rescale
whenever the running maximum moves) must therefore give the default build's
O and LSE up to rounding, and both must match the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_lse, check_o, half_ulp_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def tau0_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("tau0") / "libfa_tau0.so")
    build.build(force=True, extra_flags=["-DFA_RESCALE_TAU=0.0f"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_rescale_count", "fa_last_device_status"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


@pytest.mark.parametrize("outliers,causal", [(True, True), (False, False)])
def test_tau_zero_build_agrees(oracle_mod, tau0_lib, outliers, causal):
    w = inputs.Workload("tau", 1, 2, 2, 1024, 128, causal, 11, outliers=outliers)
    x = inputs.make_inputs(w, device="cuda", with_dO=False)
    q, k, v = x["q"], x["k"], x["v"]
    fa.fa_rescale_count()
    o8, l8 = fa.attention_fwd(q, k, v, scale=w.sm_scale, causal=causal)
    n8 = fa.fa_rescale_count()
    o0, l0 = torch.empty_like(o8), torch.empty_like(l8)
    c = ctypes.c_uint(0)
    assert tau0_lib.fa_rescale_count(None, ctypes.addressof(c)) == fa.FA_OK
    assert tau0_lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o0.data_ptr(), l0.data_ptr(), 1, 2, 2, 1024, 128,
                           w.sm_scale, int(causal), None) == fa.FA_OK
    assert tau0_lib.fa_last_device_status(None) == fa.FA_OK
    assert tau0_lib.fa_rescale_count(None, ctypes.addressof(c)) == fa.FA_OK
    torch.cuda.synchronize()
    assert c.value > n8  # tau = 0 rescales at every move of the maximum
    a, b = o8.float().cpu().numpy().astype(np.float64), o0.float().cpu().numpy().astype(np.float64)
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), w.sm_scale, causal)
    o_abs, _ = oracle_mod.attention_fwd(x["q"].cpu(), x["k"].cpu(), x["v"].cpu().abs(), w.sm_scale, causal)
    # Each build rounds every P to bf16 (relative error <= 2^-9) against its own stale
    # maximum, and rounds O to bf16: the two differ by at most 2^-8 of sum_j P_j |v_j| / l
    # plus two half-ulps of O.
    bound = 2.0 ** -8 * o_abs + 2 * half_ulp_bf16(np.maximum(np.abs(a), np.abs(b))) + 1e-6
    assert (np.abs(a - b) <= bound).all(), f"worst excess {(np.abs(a - b) - bound).max():.3e}"
    assert np.abs(l8.cpu().numpy() - l0.cpu().numpy()).max() <= 1e-4
    for o, l, what in ((o8, l8, "tau 8"), (o0, l0, "tau 0")):
        check_o(o, o_ref, what)
        check_lse(l, lse_ref, what)
