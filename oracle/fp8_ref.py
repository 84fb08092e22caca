"""FP8 (e4m3) forward with incoherent processing — TEST INFRASTRUCTURE ONLY.

The FlashAttention-3 page, section 3 ("Baja precision (FP8) con reduccion del
error de cuantizacion"), lists the method's steps: (1) multiply the query and
key feature vectors by a random orthogonal matrix (for example a Hadamard
matrix); (2) this spreads outlier coordinates over all coordinates; (3) then
quantize to FP8; (4) the orthogonal factor cancels in Q K^T.  It prints the
effect: about 2.6 times less attention error than plain FP8.

This module restates those steps in numpy (fp64 unless a step is an
FP8 rounding decision, which is taken from float32 values exactly as the CUDA
path takes it).  What the pages leave open is read as follows (the library
documents the same choices):
  * the orthogonal matrix is M = diag(signs) H_d / sqrt(d), H_d the Sylvester
    Hadamard matrix, signs a caller-supplied +-1 vector; rotated rows are x M;
  * FP8 is e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
    finite 448, smallest subnormal 2^-9), round to nearest even, saturating;
  * Q and K are scaled per block of 128 rows of one (batch, head) so that the
    block's largest magnitude maps to 448; V (not rotated: the pages rotate
    only Q and K) per (batch, kv head);
  * the probabilities P are also rounded to e4m3 before the P V product; the
    row sum uses the unrounded P.
:func:`attention_fwd_fp8_inputs` returns the dequantized tensors and
:func:`attention_fwd_fp8` the exact attention on them: the FP8 method up to
the rounding of P, which the tests bound separately.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """All finite non-negative e4m3 values, decoded from their bit patterns (0x00..0x7E)."""
    out = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        out.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(out)


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value, ties to even, magnitudes above 448 saturated to 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)  # below 2^-6 the spacing stays that of the smallest binade: 2^-9
    quantum = np.exp2(e - 3)
    r = np.minimum(np.round(a / quantum) * quantum, E4M3_MAX)  # np.round ties to even
    return np.copysign(r, x)


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), entries +-1."""
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    assert h.shape[0] == d
    return h


def rotation(signs) -> np.ndarray:
    s = np.asarray(signs, dtype=np.float64)
    return s[:, None] * hadamard(s.size) / np.sqrt(s.size)


def _quantize(block: np.ndarray):
    """One scaling block (float32 values): codes as float64 values and the float32 scale."""
    amax = np.float32(np.abs(block).max()) if block.size else np.float32(0)
    if amax == 0:
        return np.zeros(block.shape), np.float32(1.0)
    inv = np.float32(E4M3_MAX) / amax
    return e4m3_round(block.astype(np.float32) * inv), amax / np.float32(E4M3_MAX)


def quantize_row_blocks(x: np.ndarray, rows: int = 128):
    """x [B, N, Hx, d] float32 -> (dequantized float64, codes, scales [B, Hx, ceil(N/rows)])."""
    B, N, Hx, d = x.shape
    nt = (N + rows - 1) // rows
    codes = np.zeros(x.shape)
    scales = np.zeros((B, Hx, nt), np.float32)
    for b in range(B):
        for h in range(Hx):
            for t in range(nt):
                c, s = _quantize(x[b, t * rows:(t + 1) * rows, h, :])
                codes[b, t * rows:(t + 1) * rows, h, :] = c
                scales[b, h, t] = s
    deq = codes * np.repeat(scales.astype(np.float64), rows, axis=2)[:, :, :N].transpose(0, 2, 1)[..., None]
    return deq, codes, scales


def quantize_heads(x: np.ndarray):
    """x [B, N, Hx, d] float32, one scale per (batch, head) -> (dequantized, codes, scales [B, Hx])."""
    B, N, Hx, d = x.shape
    codes = np.zeros(x.shape)
    scales = np.zeros((B, Hx), np.float32)
    for b in range(B):
        for h in range(Hx):
            c, s = _quantize(x[b, :, h, :])
            codes[b, :, h, :] = c
            scales[b, h] = s
    return codes * scales.astype(np.float64)[:, None, :, None], codes, scales


def rotate(x, signs) -> np.ndarray:
    """Rows of x [..., d] times M, rounded to float32 (the CUDA path rotates in float32)."""
    x = np.asarray(x, dtype=np.float64)
    if signs is None:
        return x.astype(np.float32)
    return np.einsum("...i,ij->...j", x, rotation(signs)).astype(np.float32)


def attention_fwd_fp8_inputs(q, k, v, signs):
    """The dequantized rotated Q, K and dequantized V the FP8 path multiplies (fp64)."""
    from . import _f64

    q, k, v = _f64(q), _f64(k), _f64(v)
    qh, _, _ = quantize_row_blocks(rotate(q, signs))
    kh, _, _ = quantize_row_blocks(rotate(k, signs))
    vh, _, _ = quantize_heads(v.astype(np.float32))
    return qh, kh, vh


def attention_fwd_fp8(q, k, v, signs, scale: float, causal: bool):
    """Exact attention (fp64 oracle) on the FP8-quantized inputs: (O, LSE)."""
    from . import attention_fwd

    qh, kh, vh = attention_fwd_fp8_inputs(q, k, v, signs)
    return attention_fwd(qh, kh, vh, scale, causal)
