"""Named decode-GEMM workloads and their seeded input recipes.

Each workload fixes M (tokens), N (weight rows / output features), K, L
(independent weight sets), the split-K cluster size, and how A and B are
drawn: A ~ N(0, 0.02^2), B ~ N(0, 1), optionally with a fraction of B
entries scaled (outlier activations), all through ``synthetic``.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import synthetic


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    L: int
    split_k: int
    seed: int
    sigma_a: float = 0.02
    sigma_b: float = 1.0
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    note: str = ""

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: A and B read once, C written once (bf16)."""
        return 2 * self.L * (self.N * self.K + self.M * self.K + self.M * self.N)

    @property
    def flops(self) -> int:
        return 2 * self.L * self.M * self.N * self.K

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)

    def make_a(self, threads=None, out=None) -> np.ndarray:
        return synthetic.normal_bf16((self.L, self.N, self.K), self.seed,
                                     synthetic.STREAM_A, self.sigma_a,
                                     threads=threads, out=out)

    def make_b(self, threads=None, out=None) -> np.ndarray:
        return synthetic.normal_bf16((self.L, self.M, self.K), self.seed,
                                     synthetic.STREAM_B, self.sigma_b,
                                     outlier_p=self.outlier_p,
                                     outlier_scale=self.outlier_scale,
                                     threads=threads, out=out)


TINY = Workload("tiny split-K GEMM", M=4, N=256, K=1024, L=1, split_k=4, seed=0)
DECODE_M1 = Workload("single-token decode projection", M=1, N=7168, K=2048, L=1,
                     split_k=4, seed=1, note="29 MB of weights, pure weight streaming")
DECODE_M16 = Workload("small-batch decode", M=16, N=4096, K=7168, L=1, split_k=8,
                      seed=2, outlier_p=0.01, outlier_scale=30.0,
                      note="1% of activations scaled x30")
WIDE_S2 = Workload("wide projection", M=64, N=18432, K=7168, L=1, split_k=2, seed=3,
                   note="264 MB of weights, past L2")
WIDE_S4 = WIDE_S2.with_(split_k=4)
SWEEP_M = (1, 2, 4, 8, 16, 32, 64, 128)
SWEEP_SPLITS = (1, 2, 4, 8)


def sweep(M: int, split_k: int) -> Workload:
    return Workload("sweep", M=M, N=7168, K=16384, L=2, split_k=split_k, seed=4,
                    note="L=2 independent weight sets")


ALL_FIXED = (TINY, DECODE_M1, DECODE_M16, WIDE_S2, WIDE_S4)


def all_sweep():
    return [sweep(m, s) for m in SWEEP_M for s in SWEEP_SPLITS]
