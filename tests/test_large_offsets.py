"""Tensors past 2^31 elements (the ABI accepts up to 2^40): every element offset
the kernels form must be 64-bit.  B=4096, H=128, N=128, d=64 gives 2^32
elements per tensor (8.6 GB in bf16, about 70 GB for the forward and backward
together) at little arithmetic cost; (batch, head) slices at the far end of the
tensors, where 32-bit offsets would wrap, are checked against the oracle."""
import pytest
import torch

import exact_attention_blackwell_gb300 as fa
from helpers import check_grad, check_lse, check_o

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

B, H, N, D = 4096, 128, 128, 64


def test_forward_and_backward_past_2_to_the_31_elements(oracle_mod):
    assert B * N * H * D == 1 << 32
    free, _ = torch.cuda.mem_get_info()
    if free < 80 << 30:
        pytest.skip(f"needs ~72 GB of free device memory, {free >> 30} GB free")
    g = torch.Generator(device="cuda").manual_seed(31)
    q, k, v, dO = (torch.randn((B, N, H, D), device="cuda", generator=g, dtype=torch.bfloat16) for _ in range(4))
    scale = D ** -0.5
    causal = True
    o, lse = fa.attention_fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, dO, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    # first, middle and last slices; (B-1, H-1) holds the largest offsets
    for b, h in ((0, 0), (B // 2 + 1, 77), (B - 1, 0), (B - 1, H - 1)):
        sl = lambda t: t[b:b + 1, :, h:h + 1].cpu()
        qs, ks, vs, dOs = sl(q), sl(k), sl(v), sl(dO)
        o_ref, lse_ref = oracle_mod.attention_fwd(qs, ks, vs, scale, causal)
        what = f"(b={b}, h={h})"
        check_o(sl(o), o_ref, what)
        check_lse(lse[b:b + 1, h:h + 1].cpu(), lse_ref, what)
        grads = oracle_mod.attention_bwd(qs, ks, vs, dOs, scale, causal)
        for name, t, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), grads):
            check_grad(sl(t), r, f"{what} {name}")
