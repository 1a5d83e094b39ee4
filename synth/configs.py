"""The five synthetic workloads of the sampling pipeline.

Each is a stand-in, by shape and degree distribution, for the power-law graphs
(Papers100M, IGB, UK web graphs, Products-like) that the GARDEN page measures
on (Section VI-A, Table V); none of those datasets is used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional


@dataclass(frozen=True)
class Workload:
    name: str
    n_nodes: int
    mean_deg: float
    gamma: float
    wmax: float                   # largest expected degree of the Chung-Lu weights
    dim: int
    dtype: str                    # "f32" or "bf16"
    fanouts: List[int]            # hop order: fanouts[0] is the hop next to the seeds
    batch: int                    # seeds per mini-batch
    p_mask: float                 # share of nodes in the training mask (1.0: all)
    cache_bytes: Optional[int]    # HBM feature-cache budget; None: the whole table
    n_sub: int = 1                # mini-batches per super-batch
    offset_bits: int = 32         # CSR offset width the workload calls for
    rng_seed: int = 0
    host_features: bool = False   # full table in pinned host memory (misses read zero-copy)
    presample_batches: int = 64   # batches used to rank nodes for the cache
    notes: str = ""

    @property
    def n_hops(self) -> int:
        return len(self.fanouts)

    @property
    def row_bytes(self) -> int:
        return self.dim * (4 if self.dtype == "f32" else 2)

    @property
    def cache_rows(self) -> int:
        if self.cache_bytes is None:
            return self.n_nodes
        return min(self.n_nodes, self.cache_bytes // self.row_bytes)

    def sampler_seed(self, batch: int) -> int:
        """Hash seed of mini-batch (or super-batch) ``batch``."""
        return ((self.rng_seed & 0xFFFFFFFF) << 32) | (batch & 0x7FFFFFFF)

    def presample_seed(self, batch: int) -> int:
        """Hash seed of presampling batch ``batch`` (never a measured batch's)."""
        return ((self.rng_seed & 0xFFFFFFFF) << 32) | 0x80000000 | (batch & 0x7FFFFFFF)

    def scaled(self, n_nodes: int, **kw) -> "Workload":
        """Same recipe on fewer nodes (for oracle-sized parity cases)."""
        wmax = kw.pop("wmax", None)
        if wmax is None:
            wmax = min(self.wmax, math.sqrt(n_nodes * self.mean_deg))
        return replace(self, n_nodes=n_nodes, wmax=wmax, name=self.name + "@%d" % n_nodes, **kw)


def _sqrt_bound(n, mean):
    # Chung-Lu validity bound w_max^2 <= sum(w) where no maximum is given
    return math.sqrt(n * mean)


CONFIGS = {
    "tiny": Workload("tiny", 10_000, 10.0, 2.1, 500.0, 64, "f32", [10, 5], 256, 1.0, None,
                     notes="all features cached in HBM"),
    "mid": Workload("mid", 2_400_000, 26.0, 2.0, 20_000.0, 100, "f32", [15, 10, 5], 1024, 0.08,
                    2_400_000 * 400 // 2, host_features=True,
                    notes="cache = 50% of feature bytes, ranked by presampled access frequency"),
    "billion": Workload("billion", 111_000_000, 14.4, 2.2, _sqrt_bound(111_000_000, 14.4), 128, "f32",
                        [15, 10, 5], 1024, 0.01, 12 * 10**9, offset_bits=64, host_features=True,
                        notes="1.6B edges, int64 offsets, 12 GB cache"),
    "wide": Workload("wide", 30_000_000, 20.0, 2.1, _sqrt_bound(30_000_000, 20.0), 1024, "bf16",
                     [25, 10], 4096, 1.0, 16 * 10**9, host_features=True,
                     notes="bf16 features, 16 GB cache"),
}
for _g in (1.8, 2.0, 2.3, 2.6):
    for _b in (512, 4096):
        _k = "skew_g%.1f_b%d" % (_g, _b)
        CONFIGS[_k] = Workload(_k, 10_000_000, 20.0, _g, _sqrt_bound(10_000_000, 20.0), 256, "f32",
                               [20, 10], _b, 1.0, None, n_sub=8,
                               notes="super-batch of 8, cache = 100% HBM")


def workload(name: str) -> Workload:
    return CONFIGS[name]
