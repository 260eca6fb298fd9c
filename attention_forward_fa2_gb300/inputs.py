"""Seeded synthetic inputs for the attention forward pass.

This module only draws random numbers and arranges them in the layouts the
library takes; it holds none of the attention arithmetic, so both the CUDA path
and the CPU oracle may be fed from it.

Recipe (the input generator shown in "Flash Attention 2 Chapter2", section on
mapping attention tensors to mma operands): ``torch.manual_seed(seed)``, then
``q = randn`` and ``k``, ``v`` drawn the same way, in float32 on the CPU, laid
out ``[batch, seq, heads, d_head]`` and rounded to bf16 (round to nearest
even).  Drawing on the CPU means the GPU and the oracle see the same bf16 bits.

The variable-length recipe draws 32 lengths uniformly in [128, 4096] with
``numpy.random.default_rng(seed).integers(..., endpoint=True)`` and packs the
sequences as ``[total_tokens, heads, d_head]`` with ``cu_seqlens`` offsets.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic forward problem (shapes and seed only)."""
    name: str
    B: int
    Nq: int
    Nk: int
    H: int
    d: int
    seed: int
    lengths: Optional[tuple] = None  # variable-length form: per-sequence lengths
    note: str = field(default="", compare=False)

    @property
    def varlen(self) -> bool:
        return self.lengths is not None

    def flops(self, causal: bool = False) -> float:
        """Matmul FLOPs, 4 * B * H * Nq * Nk * d ("GPU 内核与 FlashAttention" §10);
        variable-length: sum over sequences of 4 * H * len^2 * d.  Causal: only the
        visible (query, key) pairs count, query i seeing keys j <= i + Nk - Nq."""
        def pairs(nq, nk):
            if not causal:
                return nq * nk
            off = nk - nq
            return sum(min(nk, max(0, i + off + 1)) for i in range(nq))
        if self.varlen:
            return float(sum(4 * self.H * pairs(n, n) * self.d for n in self.lengths))
        return 4.0 * self.B * self.H * pairs(self.Nq, self.Nk) * self.d

    def hbm_bytes(self) -> float:
        """Algorithmic HBM bytes: Q, K, V read once, O written once (bf16), LSE
        written once (fp32)."""
        if self.varlen:
            tot = sum(self.lengths)
            return float(4 * tot * self.H * self.d * 2 + tot * self.H * 4)
        q = self.B * self.Nq * self.H * self.d * 2
        kv = 2 * self.B * self.Nk * self.H * self.d * 2
        return float(2 * q + kv + self.B * self.H * self.Nq * 4)


def varlen_lengths(seed: int = 4, n: int = 32, lo: int = 128, hi: int = 4096) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi, size=n, endpoint=True))


def _sweep():
    out = []
    for d in (64, 128):
        for N in (512, 1024, 2048, 4096, 8192):
            seed = 100 + 10 * (d == 128) + int(math.log2(N // 512))
            out.append(Workload("sweep_d%d_n%d" % (d, N), 16, N, N, 16, d, seed))
    return tuple(out)


TINY = Workload("tiny", 1, 256, 256, 2, 128, 0, note="B1 H2 N256 d128")
SLICE = Workload("slice", 1, 64, 4096, 1, 128, 1, note="64 queries x 4096 keys, d128")
PAGE = Workload("page", 16, 4096, 4096, 16, 128, 2, note="B16 N4096 H16 d128")
SWEEP = _sweep()
VARLEN = Workload("varlen", 32, 4096, 4096, 16, 128, 4, lengths=varlen_lengths(4),
                  note="32 sequences, lengths U[128,4096], H16 d128")

WORKLOADS = {w.name: w for w in (TINY, SLICE, PAGE, VARLEN) + SWEEP}


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    """float32 N(0,1) on the CPU, rounded to bf16."""
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_dense(B: int, Nq: int, Nk: int, H: int, d: int, seed: int):
    """q [B, Nq, H, d], k and v [B, Nk, H, d], bf16 on the CPU."""
    gen = torch.Generator().manual_seed(seed)
    q = randn_bf16((B, Nq, H, d), gen)
    k = randn_bf16((B, Nk, H, d), gen)
    v = randn_bf16((B, Nk, H, d), gen)
    return q, k, v


def make_varlen(lengths, H: int, d: int, seed: int, lengths_k=None):
    """Packed q [sum(lengths), H, d], k/v [sum(lengths_k), H, d] and int32
    cu_seqlens for q and k (bf16 tensors on the CPU)."""
    lengths_k = lengths if lengths_k is None else lengths_k
    cu_q = np.concatenate([[0], np.cumsum(np.asarray(lengths, np.int64))]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(np.asarray(lengths_k, np.int64))]).astype(np.int32)
    gen = torch.Generator().manual_seed(seed)
    q = randn_bf16((int(cu_q[-1]), H, d), gen)
    k = randn_bf16((int(cu_k[-1]), H, d), gen)
    v = randn_bf16((int(cu_k[-1]), H, d), gen)
    return q, k, v, torch.from_numpy(cu_q), torch.from_numpy(cu_k)


def make(w: Workload):
    """Inputs of a named workload: (q, k, v, cu_q, cu_k); cu_* are None when dense."""
    if w.varlen:
        return make_varlen(w.lengths, w.H, w.d, w.seed)
    q, k, v = make_dense(w.B, w.Nq, w.Nk, w.H, w.d, w.seed)
    return q, k, v, None, None


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a CPU bf16 tensor (what the oracle takes)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bf16")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """Inverse of bf16_bits."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
