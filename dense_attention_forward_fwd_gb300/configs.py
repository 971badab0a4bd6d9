"""The five dense, non-causal, d=128 BF16 attention workloads this library is measured on.

Shapes follow the pages: the RTX 5090 benchmark of "Flash Attention на 5090 в CUDA C++"
(bs=1, heads=8, q=4096, kv=8192) and the 4K/8K/16K sequence lengths of the B200 kernel
write-up ("Sıfırdan yazılan CUDA attention kerneli..."). Inputs are iid N(0,1) BF16 drawn
by :mod:`inputs`; the peaked workload multiplies Q and K by 3.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

__all__ = ["Workload", "WORKLOADS", "by_name"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int = 128
    qk_mult: float = 1.0
    seed: int = 0
    # query rows per head compared against the oracle at full size (None = every row); only
    # the 16K workload is sampled (64 rows per head): its full FP64 oracle would take minutes
    oracle_rows_per_head: int | None = None

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), rounded to float32 as the kernel receives it."""
        import numpy as np
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def flops(self) -> int:
        """Algorithmic work: two B*H*Nq*Nk*d multiply-add contractions = 4*B*H*Nq*Nk*d."""
        return 4 * self.B * self.H * self.Nq * self.Nk * self.d

    @property
    def exps(self) -> int:
        return self.B * self.H * self.Nq * self.Nk

    @property
    def hbm_bytes(self) -> int:
        """Compulsory traffic: read Q, K, V once, write O (BF16) and LSE (FP32) once."""
        bh = self.B * self.H
        return bh * (2 * self.Nq * self.d + 2 * 2 * self.Nk * self.d + 2 * self.Nq * self.d + 4 * self.Nq)

    def describe(self) -> str:
        s = f"B={self.B},H={self.H},Nq={self.Nq},Nk={self.Nk},d={self.d}"
        if self.qk_mult != 1.0:
            s += f",QKx{self.qk_mult:g}"
        return s


WORKLOADS = [
    Workload("tiny-256", 1, 1, 256, 256),
    Workload("rect-4k-8k", 1, 8, 4096, 8192),
    Workload("square-4k", 4, 16, 4096, 4096),
    Workload("peaked-8k", 2, 16, 8192, 8192, qk_mult=3.0),
    Workload("long-16k", 1, 16, 16384, 16384, oracle_rows_per_head=64),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(f"unknown workload {name!r}; known: {[w.name for w in WORKLOADS]}")
