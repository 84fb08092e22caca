"""Fused exact attention for NVIDIA GB300 (sm_103a): Python binding.

The compute lives in ``libfa_gb300.so`` (hand-written CUDA, C ABI declared in
``include/fa.h``).  This module only marshals arguments: every function with a
C name calls the C entry point of the same name and returns its status code;
the ``attention_*`` helpers allocate outputs with torch and raise
:class:`FaError` on a non-zero status.  There is no fallback: if the library is
missing the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_ALIGNMENT = -3
FA_ERR_WORKSPACE = -4
FA_ERR_CUDA = -5
FA_ERR_TIMEOUT = -6

# name -> (restype, argtypes) for every symbol include/fa.h declares
_P, _I, _F, _LL, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_fp8_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_bwd_fused_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_bwd_fused": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_bwd_prepare": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "fa_bwd_dkdv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_bwd_dq": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_noalloc_scratch_bytes": (_SZ, []),
    "fa_exp2_poly": (_I, [_P, _P, _LL, _P]),
    "fa_last_device_status": (_I, [_P]),
    "fa_last_device_status_site": (_I, [_P, _P]),
    "fa_debug_stall": (_I, [_I]),
    "fa_rescale_count": (_I, [_P, _P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
}

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Loads the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with exact_attention_blackwell_gb300.build.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


# ------------------------------------------------------------------ C names
def fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, stream=None) -> int:
    return lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d, float(scale),
                        int(bool(causal)), _stream(stream))


def fa_fwd_fp8_workspace_bytes(B, H, Hkv, N, d) -> int:
    return int(lib().fa_fwd_fp8_workspace_bytes(B, H, Hkv, N, d))


def fa_fwd_fp8(q, k, v, rot_signs, o, lse, B, H, Hkv, N, d, scale, causal, workspace, workspace_bytes,
               stream=None) -> int:
    return lib().fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(rot_signs), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                            float(scale), int(bool(causal)), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, max_seqlen, total, H, Hkv, d, scale, causal, stream=None) -> int:
    return lib().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), B, max_seqlen, total,
                               H, Hkv, d, float(scale), int(bool(causal)), _stream(stream))


def fa_bwd_workspace_bytes(B, H, Hkv, N, d) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, Hkv, N, d))


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, causal, workspace, workspace_bytes,
           stream=None) -> int:
    return lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), B,
                        H, Hkv, N, d, float(scale), int(bool(causal)), _ptr(workspace), int(workspace_bytes),
                        _stream(stream))


def fa_bwd_fused_workspace_bytes(B, H, Hkv, N, d) -> int:
    return int(lib().fa_bwd_fused_workspace_bytes(B, H, Hkv, N, d))


def fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, causal, workspace, workspace_bytes,
                 stream=None) -> int:
    return lib().fa_bwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, H, Hkv, N, d, float(scale), int(bool(causal)), _ptr(workspace), int(workspace_bytes),
                              _stream(stream))


def fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens, B, max_seqlen, total, H, Hkv, d, scale, causal,
                  workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(cu_seqlens), B, max_seqlen, total, H, Hkv, d, float(scale), int(bool(causal)),
                               _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_prepare(o, lse, dO, B, H, Hkv, N, d, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_prepare(_ptr(o), _ptr(lse), _ptr(dO), B, H, Hkv, N, d, _ptr(workspace),
                                int(workspace_bytes), _stream(stream))


def fa_bwd_dkdv(q, k, v, dO, dk, dv, B, H, Hkv, N, d, scale, causal, workspace, workspace_bytes,
                stream=None) -> int:
    return lib().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dk), _ptr(dv), B, H, Hkv, N, d,
                             float(scale), int(bool(causal)), _ptr(workspace), int(workspace_bytes),
                             _stream(stream))


def fa_bwd_dq(q, k, v, dO, dq, B, H, Hkv, N, d, scale, causal, workspace, workspace_bytes, stream=None) -> int:
    return lib().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), B, H, Hkv, N, d, float(scale),
                           int(bool(causal)), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, causal, stream=None) -> int:
    """fa_bwd without a workspace: for callers that cannot allocate device
    memory when they run the backward pass (see include/fa.h)."""
    return lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                                _ptr(dv), B, H, Hkv, N, d, float(scale), int(bool(causal)), _stream(stream))


def fa_bwd_noalloc_scratch_bytes() -> int:
    """Size of fa_bwd_noalloc's built-in scratch array, as the library was built."""
    return int(lib().fa_bwd_noalloc_scratch_bytes())


def fa_exp2_poly(x, y, n, stream=None) -> int:
    return lib().fa_exp2_poly(_ptr(x), _ptr(y), int(n), _stream(stream))


def fa_rescale_count(stream=None) -> int:
    """Rescales applied by the forward kernels since the last call (then reset)."""
    c = ctypes.c_uint(0)
    st = lib().fa_rescale_count(_stream(stream), ctypes.addressof(c))
    if st != FA_OK:
        raise FaError(st, "fa_rescale_count")
    return int(c.value)


def fa_last_device_status(stream=None) -> int:
    return lib().fa_last_device_status(_stream(stream))


# ------------------------------------------------------------------ torch helpers
def _check(name, t, dtype, shape):
    """Raise ValueError unless t has this dtype and shape and is contiguous (the C ABI reads dense
    memory and cannot tell); returns (name, t) for the device check that follows all of them."""
    if t is None:
        raise ValueError(f"{name} is None")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return name, t


def _on_cuda(*checked):
    for name, t in checked:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, N, H, d] and [B, N, Hkv, d]")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    return B, N, H, Hkv, d


def _check_fixed(q, k, v, o=None, lse=None, dO=None):
    import torch

    B, N, H, Hkv, d = _dims(q, k)
    c = [_check("q", q, torch.bfloat16, (B, N, H, d)), _check("k", k, torch.bfloat16, (B, N, Hkv, d)),
         _check("v", v, torch.bfloat16, (B, N, Hkv, d))]
    if o is not None:
        c.append(_check("o", o, torch.bfloat16, (B, N, H, d)))
    if dO is not None:
        c.append(_check("dO", dO, torch.bfloat16, (B, N, H, d)))
    if lse is not None:
        c.append(_check("lse", lse, torch.float32, (B, H, N)))
    _on_cuda(*c)
    return B, N, H, Hkv, d


def _check_packed(q, k, v, cu_seqlens, o=None, lse=None, dO=None):
    import torch

    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q and k must be [total, H, d] and [total, Hkv, d]")
    total, H, d = q.shape
    Hkv = k.shape[1]
    c = [_check("q", q, torch.bfloat16, (total, H, d)), _check("k", k, torch.bfloat16, (total, Hkv, d)),
         _check("v", v, torch.bfloat16, (total, Hkv, d))]
    if cu_seqlens is None or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor of B + 1 offsets")
    c.append(_check("cu_seqlens", cu_seqlens, torch.int32, (cu_seqlens.numel(),)))
    if o is not None:
        c.append(_check("o", o, torch.bfloat16, (total, H, d)))
    if dO is not None:
        c.append(_check("dO", dO, torch.bfloat16, (total, H, d)))
    if lse is not None:
        c.append(_check("lse", lse, torch.float32, (H, total)))
    _on_cuda(*c)
    return total, H, Hkv, d


def attention_fwd(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """q [B,N,H,d], k/v [B,N,Hkv,d] bf16 CUDA tensors -> (o bf16, lse fp32 [B,H,N])."""
    import torch

    B, N, H, Hkv, d = _check_fixed(q, k, v, o=out, lse=lse)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    st = fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, stream)
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return o, lse


def attention_fwd_fp8(q, k, v, rot_signs=None, scale=None, causal=False, workspace=None, stream=None):
    """FP8 forward (d = 128): q [B,N,H,128], k/v [B,N,Hkv,128] bf16, rot_signs a float32 CUDA tensor of
    +-1 [128] or None -> (o bf16, lse fp32 [B,H,N], workspace holding the e4m3 tensors and scales)."""
    import torch

    if rot_signs is not None:
        _check("rot_signs", rot_signs, torch.float32, (128,))
    B, N, H, Hkv, d = _check_fixed(q, k, v)
    if rot_signs is not None:
        _on_cuda(("rot_signs", rot_signs))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = fa_fwd_fp8_workspace_bytes(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa_fwd_fp8(q, k, v, rot_signs, o, lse, B, H, Hkv, N, d, scale, causal, workspace, workspace.numel(), stream)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")
    return o, lse, workspace


def attention_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, scale=None, causal=False, out=None, lse=None,
                         stream=None):
    """Packed batch: q [total,H,d], k/v [total,Hkv,d] bf16 CUDA tensors, cu_seqlens an int32
    CUDA tensor [B+1] -> (o bf16 [total,H,d], lse fp32 [H,total])."""
    import torch

    total, H, Hkv, d = _check_packed(q, k, v, cu_seqlens, o=out, lse=lse)
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device) if lse is None else lse
    st = fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, int(max_seqlen), total, H, Hkv, d, scale, causal, stream)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return o, lse


def attention_bwd_varlen(q, k, v, o, lse, dO, cu_seqlens, max_seqlen, scale=None, causal=False, stream=None):
    """Packed batch backward (layouts of :func:`attention_fwd_varlen`) -> (dq, dk, dv) bf16."""
    import torch

    total, H, Hkv, d = _check_packed(q, k, v, cu_seqlens, o=o, lse=lse, dO=dO)
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = fa_bwd_workspace_bytes(B, H, Hkv, int(max_seqlen), d)
    workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens, B, int(max_seqlen), total, H, Hkv, d, scale,
                       causal, workspace, nbytes, stream)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_varlen")
    return dq, dk, dv


def attention_bwd_fused(q, k, v, o, lse, dO, scale=None, causal=False, workspace=None, stream=None):
    """The fused CTA-pair backward (head dim 128): (dq, dk, dv) bf16, not bitwise reproducible."""
    import torch

    B, N, H, Hkv, d = _check_fixed(q, k, v, o=o, lse=lse, dO=dO)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = fa_bwd_fused_workspace_bytes(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = fa_bwd_fused(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, causal, workspace, workspace.numel(),
                      stream)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_fused")
    return dq, dk, dv


def attention_bwd(q, k, v, o, lse, dO, scale=None, causal=False, workspace=None, stream=None):
    """Returns (dq, dk, dv) bf16."""
    import torch

    B, N, H, Hkv, d = _check_fixed(q, k, v, o=o, lse=lse, dO=dO)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    st = fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, causal, workspace, workspace.numel(),
                stream)
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv
