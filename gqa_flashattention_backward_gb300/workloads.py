"""Seeded synthetic workloads for the GQA attention backward.

This module only describes shapes and draws seeded random inputs; it holds none
of the attention arithmetic, so both the CUDA path's tests/benchmark and the
CPU oracle can take their inputs from it.

The five workloads follow the pages' own test shapes:

* ``tiny``          B=1, Hq=4, Hkv=1, S=128, D=64, fp16, causal (small enough
                    for the fp64 oracle in seconds).
* ``mha_causal``    B=4, Hq=Hkv=8, D=64, fp16, causal, N_CTX in 2048..32768:
                    the shape of the Triton fused-attention backward tables
                    (triton issue #4717, "fused-attention-batch4-head8-d64-bwd-causal").
* ``varlen``        Hq=32, Hkv=8, D=128, bf16, causal, 8 sequences packed
                    through cu_seqlens, lengths uniform in [512, 4096]
                    (tilelang PR #1093's varlen GQA example).
* ``sink_window``   B=2, Hq=64, Hkv=8, D=128, S=4096, fp16, causal, window
                    1024, per-head fp32 sink ~ N(0,1) (tilelang-ascend PR
                    #1638's golden shape, H=64 with 8 query heads per kv head).
* ``long_context``  B=1, Hq=32, Hkv=4, Dqk=192, Dv=128, S=32768, bf16,
                    causal, Q/K/V ~ N(0, 0.5^2), dO ~ N(0, 1).

Inputs are drawn in fp32 from a CPU ``torch.Generator`` seeded with
``1000 + index`` and then rounded to the workload's dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch


@dataclass
class Workload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    S: int                 # per-batch length, or total packed tokens when varlen
    Dqk: int
    Dv: int
    dtype: torch.dtype
    causal: bool = True
    window: int = 0
    sink: bool = False
    qkv_std: float = 1.0
    varlen_lengths: Optional[List[int]] = None
    scale: Optional[float] = None
    extra: dict = field(default_factory=dict)
    Sk: Optional[int] = None                      # key rows (or packed key tokens); None: S
    varlen_lengths_k: Optional[List[int]] = None  # per-sequence key counts; None: varlen_lengths
    window_right: int = 0                         # > 0 (not causal): right extent of a local window

    @property
    def key_len(self) -> int:
        return self.Sk if self.Sk is not None else self.S

    @property
    def cu_seqlens_k(self) -> Optional[List[int]]:
        if self.varlen_lengths_k is None:
            return None
        cu = [0]
        for n in self.varlen_lengths_k:
            cu.append(cu[-1] + n)
        return cu

    @property
    def max_seqlen_k(self) -> int:
        if self.varlen_lengths_k:
            return max(self.varlen_lengths_k)
        return self.max_seqlen if self.varlen_lengths else self.key_len

    @property
    def resolved_scale(self) -> float:
        return self.scale if self.scale is not None else self.Dqk ** -0.5

    @property
    def cu_seqlens(self) -> Optional[List[int]]:
        if self.varlen_lengths is None:
            return None
        cu = [0]
        for n in self.varlen_lengths:
            cu.append(cu[-1] + n)
        return cu

    @property
    def max_seqlen(self) -> int:
        return max(self.varlen_lengths) if self.varlen_lengths else self.S

    def pairs(self) -> int:
        """Allowed (query, key) pairs summed over every query head and batch."""
        lens = self.varlen_lengths if self.varlen_lengths else [self.S] * self.B
        return sum(_pairs_one(n, self.causal, self.window) for n in lens) * self.Hq

    def flops_exact(self) -> float:
        """Five GEMMs over the allowed pairs: 2 * pairs * (3*Dqk + 2*Dv)."""
        return 2.0 * self.pairs() * (3 * self.Dqk + 2 * self.Dv)

    def flops_convention(self) -> float:
        """2.5 x forward FLOPs with the causal half, the Triton tutorial's count."""
        lens = self.varlen_lengths if self.varlen_lengths else [self.S] * self.B
        fwd = sum(2.0 * self.Hq * n * n * (self.Dqk + self.Dv) for n in lens)
        if self.causal:
            fwd *= 0.5
        return 2.5 * fwd

    def describe(self) -> dict:
        d = dict(workload=self.name, B=self.B, Hq=self.Hq, Hkv=self.Hkv, S=self.S, Dqk=self.Dqk, Dv=self.Dv,
                 dtype=str(self.dtype).replace("torch.", ""), causal=self.causal, window=self.window,
                 sink=self.sink)
        if self.varlen_lengths:
            d["seqlens"] = list(self.varlen_lengths)
        return d


def _pairs_one(n: int, causal: bool, window: int) -> int:
    if not causal:
        return n * n
    if window <= 0 or window >= n:
        return n * (n + 1) // 2
    # rows i < window see i+1 keys, the rest see `window` keys
    return window * (window + 1) // 2 + (n - window) * window


def tiny() -> Workload:
    return Workload("tiny", 0, B=1, Hq=4, Hkv=1, S=128, Dqk=64, Dv=64, dtype=torch.float16, scale=0.125)


def mha_causal(n_ctx: int = 16384) -> Workload:
    return Workload(f"mha_causal_n{n_ctx}", 1, B=4, Hq=8, Hkv=8, S=n_ctx, Dqk=64, Dv=64, dtype=torch.float16)


MHA_SWEEP = (2048, 4096, 8192, 16384, 32768)


def varlen() -> Workload:
    g = torch.Generator().manual_seed(1002)
    lens = torch.randint(512, 4097, (8,), generator=g).tolist()
    return Workload("varlen", 2, B=1, Hq=32, Hkv=8, S=sum(lens), Dqk=128, Dv=128, dtype=torch.bfloat16,
                    varlen_lengths=lens)


def sink_window() -> Workload:
    return Workload("sink_window", 3, B=2, Hq=64, Hkv=8, S=4096, Dqk=128, Dv=128, dtype=torch.float16,
                    window=1024, sink=True)


def long_context() -> Workload:
    return Workload("long_context", 4, B=1, Hq=32, Hkv=4, S=32768, Dqk=192, Dv=128, dtype=torch.bfloat16,
                    qkv_std=0.5)


def all_workloads() -> List[Workload]:
    return [tiny(), mha_causal(), varlen(), sink_window(), long_context()]


def shrink(w: Workload, **kw) -> Workload:
    """Same workload structure at other sizes (for fast parity cases)."""
    return replace(w, **kw)


def make_inputs(w: Workload, seed: Optional[int] = None):
    """Seeded q, k, v, dout (workload dtype, CPU) and sink (fp32 CPU or None)."""
    g = torch.Generator().manual_seed(1000 + w.index if seed is None else seed)

    def draw(shape, std):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(w.dtype)

    q = draw((w.B, w.Hq, w.S, w.Dqk), w.qkv_std)
    k = draw((w.B, w.Hkv, w.key_len, w.Dqk), w.qkv_std)
    v = draw((w.B, w.Hkv, w.key_len, w.Dv), w.qkv_std)
    dout = draw((w.B, w.Hq, w.S, w.Dv), 1.0)
    sink = torch.randn((w.Hq,), generator=g, dtype=torch.float32) if w.sink else None
    return q, k, v, dout, sink
