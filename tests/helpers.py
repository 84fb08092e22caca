"""Shared test helpers: tolerances and comparison against the oracle."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances (fixed by the target of this library):
#   forward O max-abs <= 1e-2, plus half a bf16 ulp of the reference value, since
#   O is stored in bf16 and |O| can exceed 4 when a softmax row is nearly one-hot
#   (half an ulp is then 0.0156 > 1e-2);
#   LSE max-abs <= 1e-3;  backward dQ, dK, dV relative L2 <= 1e-2.
O_ATOL = 1e-2
LSE_ATOL = 1e-3
GRAD_REL_L2 = 1e-2


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def check_o(o_gpu, o_ref, what=""):
    o = o_gpu.float().cpu().numpy().astype(np.float64) if isinstance(o_gpu, torch.Tensor) else o_gpu
    err = np.abs(o - o_ref)
    bound = O_ATOL + half_ulp_bf16(o_ref)
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{what}: O error {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst} "
                                  f"(gpu {o[worst]:.5f} ref {o_ref[worst]:.5f}); max-abs {err.max():.3e}")
    return float(err.max())


def check_lse(lse_gpu, lse_ref, what=""):
    l = lse_gpu.float().cpu().numpy().astype(np.float64) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    err = np.abs(l - lse_ref)
    assert np.isfinite(l).all(), f"{what}: non-finite LSE"
    assert err.max() <= LSE_ATOL, f"{what}: LSE max-abs {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    return float(err.max())


def rel_l2(x, ref) -> float:
    x = x.float().cpu().numpy().astype(np.float64) if isinstance(x, torch.Tensor) else x
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def check_grad(g_gpu, g_ref, what=""):
    if np.linalg.norm(g_ref) == 0.0:
        # exactly-zero gradients (one visible key: dS = P (dP - D) = 0): relative
        # error is undefined, require the result to be zero up to rounding noise
        g = g_gpu.float().cpu().numpy() if isinstance(g_gpu, torch.Tensor) else g_gpu
        assert np.abs(g).max() <= 1e-4, f"{what}: expected zeros, max |g| {np.abs(g).max():.3e}"
        return 0.0
    e = rel_l2(g_gpu, g_ref)
    assert np.isfinite(e) and e <= GRAD_REL_L2, f"{what}: relative L2 {e:.3e}"
    return e
