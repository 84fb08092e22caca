"""The C ABI, without a GPU: the library loads, exports every entry point that
include/fa.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import exact_attention_blackwell_gb300 as fa
from exact_attention_blackwell_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.lib()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_prepare", "fa_bwd_dkdv", "fa_bwd_dq",
              "fa_exp2_poly", "fa_last_device_status", "fa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fa.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for code, name in [(0, "FA_OK"), (-1, "FA_ERR_INVALID_ARG"), (-2, "FA_ERR_UNSUPPORTED"),
                       (-3, "FA_ERR_ALIGNMENT"), (-4, "FA_ERR_WORKSPACE"), (-5, "FA_ERR_CUDA"),
                       (-6, "FA_ERR_TIMEOUT"), (7, "FA_ERR_UNKNOWN")]:
        assert fa.status_string(code) == name


A = 0x10000  # a 16-byte aligned fake device address: never dereferenced, calls fail validation first


@pytest.mark.parametrize("args,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=-5), fa.FA_ERR_INVALID_ARG),
    (dict(H=6, Hkv=4), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(B=65536), fa.FA_ERR_UNSUPPORTED),
    (dict(H=65536, Hkv=65536), fa.FA_ERR_UNSUPPORTED),
    (dict(B=65535, H=65535, Hkv=65535, N=4096), fa.FA_ERR_UNSUPPORTED),  # B*N*H*d beyond 2^40
    (dict(q=A + 8), fa.FA_ERR_ALIGNMENT),
    (dict(o=A + 2), fa.FA_ERR_ALIGNMENT),
    (dict(lse=A + 2), fa.FA_ERR_ALIGNMENT),
])
def test_fwd_rejects_bad_arguments(lib, args, code):
    a = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=2, Hkv=2, N=128, d=128, scale=0.125, causal=0)
    a.update(args)
    assert fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["N"], a["d"],
                     a["scale"], a["causal"], 0) == code


@pytest.mark.parametrize("args,code", [
    (dict(dq=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(H=3, Hkv=2), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dk=A + 4), fa.FA_ERR_ALIGNMENT),
    (dict(ws=None), fa.FA_ERR_WORKSPACE),
    (dict(ws_bytes=100), fa.FA_ERR_WORKSPACE),
    (dict(ws=A + 16), fa.FA_ERR_WORKSPACE),
])
def test_bwd_rejects_bad_arguments(lib, args, code):
    a = dict(q=A, k=A, v=A, o=A, lse=A, dO=A, dq=A, dk=A, dv=A, B=1, H=2, Hkv=2, N=256, d=128, scale=0.1,
             causal=1, ws=A, ws_bytes=None)
    a.update(args)
    nbytes = fa.fa_bwd_workspace_bytes(a["B"], a["H"], a["Hkv"], a["N"], 128)
    wsb = nbytes if a["ws_bytes"] is None else a["ws_bytes"]
    assert fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dO"], a["dq"], a["dk"], a["dv"], a["B"],
                     a["H"], a["Hkv"], a["N"], a["d"], a["scale"], a["causal"], a["ws"], wsb, 0) == code


def test_bwd_stages_reject_bad_arguments(lib):
    nb = fa.fa_bwd_workspace_bytes(1, 2, 2, 256, 128)
    assert fa.fa_bwd_prepare(None, A, A, 1, 2, 2, 256, 128, A, nb, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_prepare(A, A + 2, A, 1, 2, 2, 256, 128, A, nb, 0) == fa.FA_ERR_ALIGNMENT
    assert fa.fa_bwd_prepare(A, A, A, 1, 2, 2, 256, 128, A, nb - 4, 0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_dkdv(A, A, A, A, A, None, 1, 2, 2, 256, 128, 0.1, 0, A, nb, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_dkdv(A, A, A, A, A, A, 1, 2, 2, 256, 96, 0.1, 0, A, nb, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_dkdv(A, A, A, A, A + 8, A, 1, 2, 2, 256, 128, 0.1, 0, A, nb, 0) == fa.FA_ERR_ALIGNMENT
    assert fa.fa_bwd_dq(A, A, A, A, None, 1, 2, 2, 256, 128, 0.1, 0, A, nb, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_dq(A, A, A, A, A, 1, 2, 2, 256, 128, -0.1, 0, A, nb, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_dq(A, A, A, A, A, 1, 2, 2, 256, 128, 0.1, 0, None, nb, 0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd_dq(A, A, A, A + 4, A, 1, 2, 2, 256, 128, 0.1, 0, A, nb, 0) == fa.FA_ERR_ALIGNMENT


def test_workspace_size():
    B, H, Hkv, N, d = 2, 4, 2, 1000, 128
    up = lambda x: (x + 255) // 256 * 256
    Npad = (N + 127) // 128 * 128
    assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d) == 2 * up(B * H * Npad * 4)
    assert fa.fa_bwd_workspace_bytes(B, H, Hkv, N, 96) == 0
    assert fa.fa_bwd_workspace_bytes(0, H, Hkv, N, d) == 0


def test_exp2_rejects_bad_arguments(lib):
    assert fa.fa_exp2_poly(None, None, 5, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_exp2_poly(A, A, -1, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_exp2_poly(A + 1, A, 5, 0) == fa.FA_ERR_ALIGNMENT
    assert fa.fa_exp2_poly(None, None, 0, 0) == fa.FA_OK


def test_fwd_varlen_rejects_bad_arguments(lib):
    # q, k, v, o, lse, cu, B, max_seqlen, total, H, Hkv, d, scale, causal, stream
    ok = dict(q=A, k=A, v=A, o=A, lse=A, cu=A, B=2, L=300, total=400, H=4, Hkv=2, d=128, scale=0.1)

    def call(**kw):
        a = dict(ok, **kw)
        return fa.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["B"], a["L"], a["total"], a["H"],
                                a["Hkv"], a["d"], a["scale"], 0, 0)

    assert call(cu=None) == fa.FA_ERR_INVALID_ARG
    assert call(cu=A + 2) == fa.FA_ERR_INVALID_ARG  # the table must be 4-byte aligned
    assert call(total=-1) == fa.FA_ERR_INVALID_ARG
    assert call(L=0) == fa.FA_ERR_INVALID_ARG
    assert call(B=0) == fa.FA_ERR_INVALID_ARG
    assert call(H=3) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(q=A + 8) == fa.FA_ERR_ALIGNMENT


def test_bwd_varlen_rejects_bad_arguments(lib):
    nb = fa.fa_bwd_workspace_bytes(2, 4, 2, 300, 128)

    def call(cu=A, total=400, ws=A, wsb=nb, dq=A, L=300):
        return fa.fa_bwd_varlen(A, A, A, A, A, A, dq, A, A, cu, 2, L, total, 4, 2, 128, 0.1, 0, ws, wsb, 0)

    assert call(cu=None) == fa.FA_ERR_INVALID_ARG
    assert call(cu=A + 2) == fa.FA_ERR_INVALID_ARG
    assert call(total=-3) == fa.FA_ERR_INVALID_ARG
    assert call(dq=None) == fa.FA_ERR_INVALID_ARG
    assert call(ws=None) == fa.FA_ERR_WORKSPACE
    assert call(wsb=nb - 4) == fa.FA_ERR_WORKSPACE
    assert call(L=0) == fa.FA_ERR_INVALID_ARG


def test_fwd_fp8_rejects_bad_arguments(lib):
    nb = fa.fa_fwd_fp8_workspace_bytes(1, 2, 2, 256, 128)
    assert nb > 0 and fa.fa_fwd_fp8_workspace_bytes(1, 2, 2, 256, 64) == 0

    def call(d=128, ws=A, wsb=nb, q=A, signs=None):
        return fa.fa_fwd_fp8(q, A, A, signs, A, None, 1, 2, 2, 256, d, 0.1, 0, ws, wsb, 0)

    assert call(d=64) == fa.FA_ERR_UNSUPPORTED
    assert call(q=None) == fa.FA_ERR_INVALID_ARG
    assert call(ws=None) == fa.FA_ERR_WORKSPACE
    assert call(wsb=nb - 1) == fa.FA_ERR_WORKSPACE
    assert call(ws=A + 16) == fa.FA_ERR_WORKSPACE  # 256-byte alignment
    assert call(signs=A + 2) == fa.FA_ERR_ALIGNMENT


def test_noalloc_scratch_size_matches_the_header(lib):
    with open(HEADER) as f:
        m = re.search(r"#define\s+FA_BWD_NOALLOC_SCRATCH_BYTES\s+\((\d+)ull\s*<<\s*(\d+)\)", f.read())
    assert m, "FA_BWD_NOALLOC_SCRATCH_BYTES not found in include/fa.h"
    assert fa.fa_bwd_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_noalloc_rejects_bad_arguments_like_fa_bwd(lib):
    good = (1, 2, 2, 256, 128, 0.1, 1, 0)  # B, H, Hkv, N, d, scale, causal, stream
    p9 = (A,) * 9
    assert fa.fa_bwd_noalloc(A, A, A, A, A, A, None, A, A, *good) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_noalloc(*p9, 1, 2, 2, 256, 96, 0.1, 1, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_noalloc(*p9, 1, 3, 2, 256, 128, 0.1, 1, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_noalloc(A, A, A, A, A + 2, A, A, A, A, *good) == fa.FA_ERR_ALIGNMENT
    assert fa.fa_bwd_noalloc(A, A, A, A, A, A, A + 8, A, A, *good) == fa.FA_ERR_ALIGNMENT


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="valid arguments would launch on the GPU with fake addresses")
def test_noalloc_fails_like_fa_bwd_without_a_usable_device(lib):
    # arguments that pass every check: the device check decides, and both entry
    # points must report the same status (no GPU here: the CUDA error)
    B, H, Hkv, N, d = 1, 2, 2, 256, 128
    nb = fa.fa_bwd_workspace_bytes(B, H, Hkv, N, d)
    ws = 0x100000  # 256-byte aligned
    ref = fa.fa_bwd(A, A, A, A, A, A, A, A, A, B, H, Hkv, N, d, 0.1, 1, ws, nb, 0)
    got = fa.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, H, Hkv, N, d, 0.1, 1, 0)
    assert ref != fa.FA_OK and got == ref
