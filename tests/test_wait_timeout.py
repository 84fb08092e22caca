"""Bounded waits, made to run out on the GPU.

Every wait inside the kernels is bounded; when one runs out the kernel sets
the library's status word, the other waits of the CTA give up, in-flight MMAs
and copies are drained, TMEM is freed and the kernel returns (include/fa.h,
fa_last_device_status).  A library built with -DFA_TEST_STALL and a 2 ms wait
limit lets a test make block 0 of one kernel skip one barrier arrival, a signal
that nothing else gives: the kernel must come back with FA_ERR_TIMEOUT and the
id of the wait that ran out, and the same process must then compute a correct
forward and backward pass.  Nothing here faults the GPU: the waits end by
themselves.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build, inputs
from helpers import check_grad, check_lse, check_o

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LIMIT_NS = 2_000_000  # 2 ms
# mode -> ids (include/fa.h) of the waits that can run out first in the stalled
# kernel: the one whose arrival was skipped (the MMA warp waiting on P or dS),
# or the producer's wait for a ring slot, which began earlier (the ring filled
# up before the first MMA) and is never released once the MMA warp stops.
MODES = {1: {4, 5}, 2: {16, 13}, 3: {17, 13}}


@pytest.fixture(scope="module")
def stall_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("stall") / "libfa_stall.so")
    # causal head-dim-128 shapes take the CTA-pair dK/dV kernel at every length in
    # this build, non-causal ones below 2048 rows the one-CTA kernel: mode 2 is
    # run both ways
    build.build(force=True, extra_flags=["-DFA_TEST_STALL", f"-DFA_WAIT_LIMIT_NS={LIMIT_NS}ull",
                                         "-DFA_DKDV_PAIR_MIN_N_CAUSAL=0"], lib_path=path)
    lib = ctypes.CDLL(path)
    for name in ("fa_fwd", "fa_bwd_workspace_bytes", "fa_bwd", "fa_last_device_status", "fa_last_device_status_site",
                 "fa_debug_stall"):
        res, args = fa.SIGNATURES[name]
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


def run(lib, x, B, H, N, d, causal):
    q, k, v, dO = x["q"], x["k"], x["v"], x["dO"]
    scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    assert lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H, N, d, scale,
                      int(causal), None) == fa.FA_OK
    nb = lib.fa_bwd_workspace_bytes(B, H, H, N, d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    g = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    assert lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                      g[0].data_ptr(), g[1].data_ptr(), g[2].data_ptr(), B, H, H, N, d, scale, int(causal),
                      ws.data_ptr(), nb, None) == fa.FA_OK
    return o, lse, g


def test_default_build_has_no_stall_hook():
    assert fa.lib().fa_debug_stall(1) == fa.FA_ERR_UNSUPPORTED


# (mode, causal, B, H, d).  The one-CTA dK/dV kernel and the dQ kernel are
# persistent: with 320 work units on at most one CTA per SM, block 0 runs
# several, and after the stall in its first unit it must still return (causal
# head-dim-128 dK/dV takes the CTA pairs in this build).
CASES = [(1, True, 1, 2, 128), (2, True, 1, 2, 128), (2, False, 1, 2, 128), (3, True, 1, 2, 128),
         (2, True, 4, 16, 64), (2, False, 4, 16, 64), (2, False, 4, 16, 128), (3, False, 4, 16, 64),
         (3, True, 4, 16, 128), (1, True, 4, 16, 128)]


@pytest.mark.parametrize("mode,causal,B,H,d", CASES)
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_correct(oracle_mod, stall_lib, mode, causal, B, H, d):
    N = 640
    w = inputs.Workload("stall", B, H, H, N, d, causal, 6100 + mode + d)
    x = inputs.make_inputs(w, device="cuda")
    site = ctypes.c_int(-1)
    assert stall_lib.fa_last_device_status_site(None, ctypes.byref(site)) == fa.FA_OK and site.value == 0
    assert stall_lib.fa_debug_stall(mode) == fa.FA_OK
    try:
        run(stall_lib, x, B, H, N, d, causal)  # the stalled kernel returns after its waits run out
        st = stall_lib.fa_last_device_status_site(None, ctypes.byref(site))
    finally:
        assert stall_lib.fa_debug_stall(0) == fa.FA_OK
    assert st == fa.FA_ERR_TIMEOUT
    assert site.value in MODES[mode], site.value
    assert stall_lib.fa_last_device_status_site(None, ctypes.byref(site)) == fa.FA_OK and site.value == 0  # cleared
    # the context is still usable: the same process computes a correct pass
    o, lse, g = run(stall_lib, x, B, H, N, d, causal)
    torch.cuda.synchronize()
    assert stall_lib.fa_last_device_status(None) == fa.FA_OK
    xc = {n: t.cpu() for n, t in x.items()}
    o_ref, lse_ref = oracle_mod.attention_fwd(xc["q"], xc["k"], xc["v"], w.sm_scale, causal)
    check_o(o, o_ref, f"after stall mode {mode}")
    check_lse(lse, lse_ref, f"after stall mode {mode}")
    refs = oracle_mod.attention_bwd(xc["q"], xc["k"], xc["v"], xc["dO"], w.sm_scale, causal)
    for name, a, r in zip(("dQ", "dK", "dV"), g, refs):
        check_grad(a.cpu(), r, f"after stall mode {mode} {name}")
