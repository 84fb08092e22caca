"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws numbers.  Both sides of
every parity check (the CUDA library and the CPU oracle) receive the same bf16
tensors made here.

Recipe (the pages print no dataset; every workload is synthetic):
  * ``torch.Generator().manual_seed(seed)`` on the CPU; Q, K, V, dO drawn in that
    order as iid N(0, 1) fp32, Q and dO with shape [B, N, H, d], K and V with
    shape [B, N, Hkv, d].
  * With ``outliers=True`` (the causal stress workload), after dO one uniform
    draw per Q element then per K element; an element whose draw is < 0.01 is
    multiplied by 20.
  * Everything is then rounded to bf16 (round-to-nearest-even, torch default).
  * Packed variable-length batches (``PackedWorkload``): sequence lengths from
    ``numpy.random.default_rng(seed)``, log-uniform between ``lo`` and ``hi``
    rows, drawn until ``total`` rows are covered (the last one cut to fit);
    then Q, K, V, dO as above with shapes [total, H, d] / [total, Hkv, d] from
    ``torch.Generator().manual_seed(seed)``.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    causal: bool
    seed: int
    outliers: bool = False
    backward: bool = True
    scale: float = field(default=float("nan"))

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.d) if math.isnan(self.scale) else self.scale

    def fwd_flops(self) -> float:
        """4 B H N^2 d, halved when causal (the metric's convention)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


def tiny() -> Workload:
    return Workload("tiny B1 H2 N128 d64", 1, 2, 2, 128, 64, False, 0)


def headline() -> Workload:
    return Workload("B4 H16 N8192 d128 non-causal", 4, 16, 16, 8192, 128, False, 1)


def causal_outliers() -> Workload:
    return Workload("causal B8 H16 N4096 d128 1% x20 outliers", 8, 16, 16, 4096, 128, True, 2,
                    outliers=True)


def long_gqa() -> Workload:
    return Workload("GQA B1 H32 Hkv8 N32768 d128 causal fwd", 1, 32, 8, 32768, 128, True, 3,
                    backward=False)


def sweep() -> list[Workload]:
    out = []
    k = 0
    for d in (64, 128, 256):
        for N in (1024, 4096, 16384):
            for causal in (False, True):
                B = 32768 // N
                out.append(Workload(f"sweep d{d} N{N} B{B} {'causal' if causal else 'non-causal'}",
                                    B, 16, 16, N, d, causal, 100 + k))
                k += 1
    return out


def make_inputs(w: Workload, device="cpu", with_dO: bool = True):
    """Returns dict(q, k, v, dO) of bf16 tensors on ``device`` (drawn on the CPU)."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.B, w.N, w.H, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.N, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.N, w.Hkv, w.d), generator=g, dtype=torch.float32)
    dO = torch.randn((w.B, w.N, w.H, w.d), generator=g, dtype=torch.float32) if with_dO or w.outliers else None
    if w.outliers:
        q = torch.where(torch.rand(q.shape, generator=g) < 0.01, q * 20.0, q)
        k = torch.where(torch.rand(k.shape, generator=g) < 0.01, k * 20.0, k)
    out = {"q": q, "k": k, "v": v, "dO": dO if with_dO else None}
    return {n: (t.to(torch.bfloat16).to(device) if t is not None else None) for n, t in out.items()}


def random_bf16(shape, seed: int, device="cpu"):
    """iid N(0,1) rounded to bf16, for ad-hoc shapes (edge-case tests)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(device)


@dataclass(frozen=True)
class PackedWorkload:
    """Sequences of different lengths packed back to back (cu_seqlens layout)."""
    name: str
    lens: tuple
    H: int
    Hkv: int
    d: int
    causal: bool
    seed: int
    backward: bool = True

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def total(self) -> int:
        return int(sum(self.lens))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lens))

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def cu_seqlens(self) -> list:
        return [0] + [int(x) for x in np.cumsum(self.lens)]

    def fwd_flops(self) -> float:
        """Sum over sequences of the single-sequence convention."""
        f = sum(4.0 * self.H * n * n * self.d for n in self.lens)
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()


def packed_lengths(total: int, lo: int, hi: int, seed: int) -> tuple:
    rng = np.random.default_rng(seed)
    lens, left = [], total
    while left > 0:
        n = int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        n = min(max(n, 1), left)
        lens.append(n)
        left -= n
    return tuple(lens)


def packed_causal() -> PackedWorkload:
    lens = packed_lengths(65536, 128, 16384, 4)
    return PackedWorkload(f"packed {len(lens)} seqs (128..16384 rows, 65536 total) H16 d128 causal", lens, 16, 16,
                          128, True, 4)


def make_packed_inputs(w: PackedWorkload, device="cpu", with_dO: bool = True):
    """Returns dict(q, k, v, dO, cu_seqlens) for a packed workload (drawn on the CPU)."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.total, w.H, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.total, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.total, w.Hkv, w.d), generator=g, dtype=torch.float32)
    dO = torch.randn((w.total, w.H, w.d), generator=g, dtype=torch.float32) if with_dO else None
    out = {n: (t.to(torch.bfloat16).to(device) if t is not None else None)
           for n, t in {"q": q, "k": k, "v": v, "dO": dO}.items()}
    out["cu_seqlens"] = torch.tensor(w.cu_seqlens(), dtype=torch.int32, device=device)
    return out


def input_sha256(x: dict) -> str:
    """SHA-256 over the bf16 bits of q, k, v and dO (when present), in that order:
    the bits the kernels and the oracle both read, logged beside every result."""
    h = hashlib.sha256()
    for n in ("q", "k", "v", "dO"):
        t = x.get(n)
        if t is not None:
            h.update(t.detach().contiguous().cpu().view(torch.int16).numpy().tobytes())
    return h.hexdigest()
