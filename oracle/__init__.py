"""fp64 CPU oracle for exact attention — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports it, and it imports nothing from the product.

Two independent statements of the same definition live here:

* ``attn_oracle.c`` — the primary oracle: plain loops in fp64, OpenMP over
  independent rows.  Built into ``liboracle.so`` by :func:`build`.
* ``np_ref.py`` — a second restatement in matrix form with numpy, used only on
  tiny shapes to cross-check the C oracle.

Both follow the definition of attention on the pages (FlashAttention-4 article,
"Por que el enfoque estandar ya no funciona": S = Q K^T, O = P V with a softmax
between; FlashAttention-3 page, "El problema del mecanismo de atencion") with the
scale, causal mask, natural-log LSE and chain-rule backward written out in the
header of ``attn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` with gcc + OpenMP."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.POINTER(ctypes.c_double)
        IP = ctypes.POINTER(ctypes.c_int)
        i, dbl = ctypes.c_int, ctypes.c_double
        lib.oracle_fwd_rows.argtypes = [P, P, P, i, i, i, i, i, dbl, i, IP, i, P, P]
        lib.oracle_fwd_rows.restype = None
        lib.oracle_bwd_rows.argtypes = [P, P, P, P, i, i, i, i, i, dbl, i, IP, i, IP, i, P, P, P]
        lib.oracle_bwd_rows.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = None
        _lib = lib
    return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 values convert exactly)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _rows(rows, N):
    if rows is None:
        return None, N
    r = np.ascontiguousarray(rows, dtype=np.int32)
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < N))
    return r, int(r.size)


def num_threads() -> int:
    """OpenMP threads one oracle call uses."""
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    """Sets the OpenMP threads of later oracle calls (timing only; results do not depend on it)."""
    _load().oracle_set_threads(int(n))


def attention_fwd(q, k, v, scale: float, causal: bool, rows=None):
    """Forward: returns (O, LSE) in fp64.

    q: [B, N, H, d]; k, v: [B, N, Hkv, d].  ``rows`` (optional) lists the query
    rows to compute; O is then [B, len(rows), H, d] and LSE [B, H, len(rows)].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, N, Hkv, d) and v.shape == k.shape and H % Hkv == 0
    r, nr = _rows(rows, N)
    o = np.empty((B, nr, H, d), np.float64)
    lse = np.empty((B, H, nr), np.float64)
    _load().oracle_fwd_rows(_dp(q), _dp(k), _dp(v), B, H, Hkv, N, d, float(scale), int(bool(causal)),
                            _ip(r), nr, _dp(o), _dp(lse))
    return o, lse


def attention_bwd(q, k, v, dO, scale: float, causal: bool, qrows=None, kvrows=None):
    """Backward of L = sum(dO * O): returns (dQ, dK, dV) in fp64.

    ``qrows`` selects rows of dQ ([B, len(qrows), H, d]); ``kvrows`` selects rows
    of dK and dV ([B, len(kvrows), Hkv, d]).  None means all rows.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    assert dO.shape == q.shape and k.shape == (B, N, Hkv, d) and v.shape == k.shape and H % Hkv == 0
    qr, nq = _rows(qrows, N)
    kr, nkv = _rows(kvrows, N)
    dq = np.empty((B, nq, H, d), np.float64)
    dk = np.empty((B, nkv, Hkv, d), np.float64)
    dv = np.empty((B, nkv, Hkv, d), np.float64)
    _load().oracle_bwd_rows(_dp(q), _dp(k), _dp(v), _dp(dO), B, H, Hkv, N, d, float(scale),
                            int(bool(causal)), _ip(qr), nq, _ip(kr), nkv, _dp(dq), _dp(dk), _dp(dv))
    return dq, dk, dv


def _seq_bounds(cu_seqlens):
    cu = np.asarray(cu_seqlens.detach().cpu() if hasattr(cu_seqlens, "detach") else cu_seqlens, dtype=np.int64)
    assert cu.ndim == 1 and cu.size >= 2 and cu[0] == 0 and (np.diff(cu) >= 0).all()
    return [(int(a), int(b)) for a, b in zip(cu[:-1], cu[1:])]


def attention_fwd_varlen(q, k, v, cu_seqlens, scale: float, causal: bool):
    """Packed variable-length forward: sequence b is rows [cu[b], cu[b+1]) of
    q [total, H, d] and k, v [total, Hkv, d], and is the single-sequence
    problem of :func:`attention_fwd` on those rows (the plain reading of the
    varlen variant the FlashAttention-4 paper summary names in section 5).
    Returns (O [total, H, d], LSE [H, total]) in fp64; rows of no sequence stay 0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    total, H, d = q.shape
    o = np.zeros((total, H, d), np.float64)
    lse = np.zeros((H, total), np.float64)
    for a, b in _seq_bounds(cu_seqlens):
        if b == a:
            continue
        ob, lb = attention_fwd(q[None, a:b], k[None, a:b], v[None, a:b], scale, causal)
        o[a:b] = ob[0]
        lse[:, a:b] = lb[0]
    return o, lse


def attention_bwd_varlen(q, k, v, dO, cu_seqlens, scale: float, causal: bool):
    """Packed variable-length backward, per sequence as in :func:`attention_fwd_varlen`.
    Returns (dQ [total, H, d], dK, dV [total, Hkv, d]) in fp64."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for a, b in _seq_bounds(cu_seqlens):
        if b == a:
            continue
        g = attention_bwd(q[None, a:b], k[None, a:b], v[None, a:b], dO[None, a:b], scale, causal)
        dq[a:b], dk[a:b], dv[a:b] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv
