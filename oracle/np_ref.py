"""Second, independent restatement of exact attention in numpy matrix form (fp64).

TEST INFRASTRUCTURE ONLY, for tiny shapes: it exists to cross-check the C
oracle (``attn_oracle.c``), which is written as per-row loops.  Here the same
definition is written as whole-matrix operations, per head:

    S = scale * Q K^T, masked entries -> -inf (causal: key j visible iff j <= i)
    P = softmax_rows(S);  O = P V;  LSE = log(sum_j exp(S_ij))
    dV = P^T dO;  dP = dO V^T;  dS = P * (dP - rowsum(dO * O));
    dQ = scale dS K;  dK = scale dS^T Q

(FlashAttention-4 article, "Por que el enfoque estandar ya no funciona": S = QK^T
and O = PV with a softmax between them; the scale, mask and backward are the
plainest reading of the pages, stated in the C oracle's header.)
"""
from __future__ import annotations

import numpy as np


def _heads(x: np.ndarray) -> np.ndarray:
    # [B, N, Hx, d] -> [B, Hx, N, d]
    return np.transpose(np.asarray(x, dtype=np.float64), (0, 2, 1, 3))


def _expand_kv(x: np.ndarray, H: int) -> np.ndarray:
    # [B, Hkv, N, d] -> [B, H, N, d], query head h reads kv head h // (H // Hkv)
    g = H // x.shape[1]
    return np.repeat(x, g, axis=1)


def _scores(q, k, scale, causal):
    s = scale * np.einsum("bhic,bhjc->bhij", q, k)
    if causal:
        N = s.shape[-1]
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    return s


def fwd(q, k, v, scale: float, causal: bool):
    """Returns (O [B,N,H,d], LSE [B,H,N])."""
    H = np.asarray(q).shape[2]
    qh, kh, vh = _heads(q), _expand_kv(_heads(k), H), _expand_kv(_heads(v), H)
    s = _scores(qh, kh, scale, causal)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    p = e / l
    o = p @ vh
    lse = (m + np.log(l))[..., 0]
    return np.transpose(o, (0, 2, 1, 3)), lse


def bwd(q, k, v, dO, scale: float, causal: bool):
    """Returns (dQ [B,N,H,d], dK [B,N,Hkv,d], dV [B,N,Hkv,d])."""
    H = np.asarray(q).shape[2]
    Hkv = np.asarray(k).shape[2]
    qh, kh, vh = _heads(q), _expand_kv(_heads(k), H), _expand_kv(_heads(v), H)
    doh = _heads(dO)
    s = _scores(qh, kh, scale, causal)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=-1, keepdims=True)
    o = p @ vh
    dv = np.swapaxes(p, -1, -2) @ doh
    dp = doh @ np.swapaxes(vh, -1, -2)
    Dvec = (doh * o).sum(axis=-1, keepdims=True)
    ds = p * (dp - Dvec)
    dq = scale * (ds @ kh)
    dk = scale * (np.swapaxes(ds, -1, -2) @ qh)
    B, _, N, d = dk.shape
    g = H // Hkv
    dk = dk.reshape(B, Hkv, g, N, d).sum(axis=2)
    dv = dv.reshape(B, Hkv, g, N, d).sum(axis=2)
    t = lambda x: np.transpose(x, (0, 2, 1, 3))
    return t(dq), t(dk), t(dv)
