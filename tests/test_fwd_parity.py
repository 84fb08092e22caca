"""Forward parity: the CUDA library (through its C ABI) against the fp64 oracle
on the same seeded bf16 inputs, element by element."""
import math

import numpy as np
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import inputs
from helpers import check_lse, check_o

pytestmark = pytest.mark.gpu


def run_fwd(q, k, v, scale, causal):
    o, lse = fa.attention_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    return o.cpu(), lse.cpu()


def test_tiny_workload_full(oracle_mod):
    w = inputs.tiny()
    x = inputs.make_inputs(w)
    o, lse = run_fwd(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    check_o(o, o_ref, w.name)
    check_lse(lse, lse_ref, w.name)


CASES = [
    # B, N, H, Hkv, d, causal
    (1, 128, 1, 1, 128, False),
    (1, 256, 2, 2, 128, False),
    (2, 640, 2, 2, 128, True),
    (1, 384, 4, 2, 128, False),
    (1, 512, 4, 1, 128, True),
    (1, 1, 2, 2, 128, False),
    (1, 77, 1, 1, 128, True),
    (2, 300, 2, 1, 128, False),
    (1, 513, 2, 2, 128, True),
    (1, 256, 2, 2, 64, False),
    (1, 395, 2, 2, 64, True),
    (1, 256, 2, 2, 256, False),
    (1, 333, 2, 1, 256, True),
]


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", CASES)
def test_small_shapes_full(oracle_mod, B, N, H, Hkv, d, causal):
    seed = 1000 + N + 7 * d + H + causal
    q = inputs.random_bf16((B, N, H, d), seed)
    k = inputs.random_bf16((B, N, Hkv, d), seed + 1)
    v = inputs.random_bf16((B, N, Hkv, d), seed + 2)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, scale, causal)
    o_ref, lse_ref = oracle_mod.attention_fwd(q, k, v, scale, causal)
    what = f"B{B} N{N} H{H}/{Hkv} d{d} causal={causal}"
    check_o(o, o_ref, what)
    check_lse(lse, lse_ref, what)


def test_outliers_force_rescale(oracle_mod):
    """x20 outliers in Q and K move row maxima by far more than the rescale threshold:
    the conditional rescale must fire (counter > 0) and the result stay exact."""
    w = inputs.Workload("outliers", 1, 2, 2, 1024, 128, True, 7, outliers=True)
    x = inputs.make_inputs(w)
    fa.fa_rescale_count()  # reset
    o, lse = run_fwd(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    assert fa.fa_rescale_count() > 0
    o_ref, lse_ref = oracle_mod.attention_fwd(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
    check_o(o, o_ref, w.name)
    check_lse(lse, lse_ref, w.name)


def test_deterministic_and_lse_optional():
    w = inputs.Workload("det", 1, 2, 2, 384, 128, False, 8)
    x = inputs.make_inputs(w, device="cuda")
    o1, l1 = fa.attention_fwd(x["q"], x["k"], x["v"], causal=False)
    o2 = torch.empty_like(o1)
    assert fa.fa_fwd(x["q"], x["k"], x["v"], o2, None, 1, 2, 2, 384, 128, w.sm_scale, 0) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
