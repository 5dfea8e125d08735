"""The five synthetic workloads, as seeded descriptions.

Each workload restates one of the shapes the pages measure (production shards that are not
public) as seeded synthetic input with the stated table sizes, widths, dtypes, bag-length
and id distributions.  The recipe for each is spelled out below; every random draw is made
from ``seed`` by ``synth.gen``.

Bag lengths are per (table, bag); ids follow a per-table distribution:
  * ``uniform``: ids uniform in [0, E).
  * ``zipf``: a truncated Zipf-Mandelbrot law, density proportional to (x + 1 + q)^-s on
    [0, E), floored to an integer rank k, then scattered over the table by the bijection
    id = (a*k + c) mod E (gcd(a, E) = 1) so that hot rows are not adjacent.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class LengthSpec:
    kind: str                 # "fixed" | "poisson" | "lognormal"
    value: float = 0.0        # fixed length, Poisson mean, or lognormal mu
    sigma: float = 0.0        # lognormal sigma
    min_len: int = 0          # lengths below this are raised to it
    empty_frac: float = 0.0   # fraction of bags forced to length 0 (drawn independently)


@dataclass(frozen=True)
class IdSpec:
    kind: str                 # "uniform" | "zipf"
    s: float = 0.0
    q: float = 0.0


@dataclass(frozen=True)
class TableSpec:
    E: int
    D: int
    lengths: LengthSpec
    ids: IdSpec
    histogram: bool = False   # caller's declaration that the table suits the counts x table path


@dataclass(frozen=True)
class TBEConfig:
    name: str
    description: str
    B: int
    tables: tuple
    wdtype: str               # "f32" | "f16" | "bf16"
    itype: str                # "i32" | "i64"
    weighted: bool
    optimizer: str            # "sgd" | "adagrad"
    lr: float
    eps: float
    w_scale: float            # weights ~ U(-w_scale, w_scale)
    bad_id_frac: float        # fraction of ids replaced by out-of-range values
    seed: int
    meta: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def T(self) -> int:
        return len(self.tables)

    @property
    def D(self) -> np.ndarray:
        return np.array([t.D for t in self.tables], dtype=np.int32)

    @property
    def E(self) -> np.ndarray:
        return np.array([t.E for t in self.tables], dtype=np.int64)

    @property
    def total_D(self) -> int:
        return int(self.D.sum())

    @property
    def total_rows(self) -> int:
        return int(self.E.sum())

    @property
    def elem_offsets(self) -> np.ndarray:
        """First weight element of each table in the packed layout, [T+1]."""
        return np.concatenate([[0], np.cumsum(self.E * self.D.astype(np.int64))]).astype(np.int64)

    @property
    def histogram_tables(self) -> tuple:
        return tuple(i for i, t in enumerate(self.tables) if t.histogram)

    def shrink(self, B: int | None = None, E_div: int = 1, T: int | None = None,
               name: str | None = None) -> "TBEConfig":
        """A smaller workload of the same kind: fewer bags, fewer tables, fewer rows per table
        (rows divided by E_div, at least 8; tables marked for the counts x table path keep E)."""
        tables = self.tables[: (T or self.T)]
        tables = tuple(t if t.histogram else dataclasses.replace(t, E=max(8, t.E // E_div))
                       for t in tables)
        B = B or self.B
        return dataclasses.replace(
            self, name=name or f"{self.name}[B={B},T={len(tables)},E/{E_div}]", B=B, tables=tables)


def _log_uniform_ints(rng: np.random.Generator, lo: int, hi: int, n: int) -> list:
    return [int(round(math.exp(v))) for v in rng.uniform(math.log(lo), math.log(hi), n)]


def _c1() -> TBEConfig:
    L = LengthSpec("fixed", 8)
    ids = IdSpec("uniform")
    return TBEConfig(
        name="c1_tiny",
        description="T=2, E=1000, D=64, fp32 ~U(-0.1,0.1), B=32, L=8, uniform int64 ids, "
                    "unweighted, SGD lr=0.01, grads ~N(0,1)",
        B=32, tables=tuple(TableSpec(1000, 64, L, ids) for _ in range(2)), wdtype="f32",
        itype="i64", weighted=False, optimizer="sgd", lr=0.01, eps=1e-8, w_scale=0.1,
        bad_id_frac=0.0, seed=0)


def _c2() -> TBEConfig:
    rng = np.random.default_rng(np.random.SeedSequence([1, 0xE]))
    Es = _log_uniform_ints(rng, 100_000, 1_000_000, 26)
    L = LengthSpec("poisson", 20.0, min_len=1)
    ids = IdSpec("zipf", s=1.05, q=0.0)
    return TBEConfig(
        name="c2_mid",
        description="T=26, E log-uniform 100k-1M, D=128 fp16 ~U(-0.01,0.01), B=8192, "
                    "L~Poisson(20) min 1, Zipf(s=1.05) ids, int32 indices/offsets, "
                    "row-wise Adagrad lr=0.01 eps=1e-8",
        B=8192, tables=tuple(TableSpec(E, 128, L, ids) for E in Es), wdtype="f16", itype="i32",
        weighted=False, optimizer="adagrad", lr=0.01, eps=1e-8, w_scale=0.01, bad_id_frac=0.0,
        seed=1)


# Zipf-Mandelbrot parameters of the large-skew workload, chosen so that the closed-form
# expectations of this sampler give ~3.0M distinct rows over the batch and ~125K hits on the
# hottest row of each table (the batch statistic 83M / 3M / 125K); checked by
# tests/test_synth.py against synth.gen.expected_stats.
C3_ZIPF_S = 1.4135
C3_ZIPF_Q = 7.01


def _c3() -> TBEConfig:
    L = LengthSpec("lognormal", math.log(20.0) - 0.5, sigma=1.0, min_len=1)
    ids = IdSpec("zipf", s=C3_ZIPF_S, q=C3_ZIPF_Q)
    return TBEConfig(
        name="c3_stress",
        description="T=32, E=4M, D=128 fp16 ~U(-0.01,0.01), B=131072 (T*B=4.19M bags), "
                    "L=max(1,round(lognormal(ln20-0.5, 1))) (mean 20, ~83.9M lookups), "
                    f"Zipf-Mandelbrot(s={C3_ZIPF_S}, q={C3_ZIPF_Q}) ids (~3M distinct rows, "
                    "hottest ~125K hits), int64, row-wise Adagrad lr=0.01 eps=1e-8",
        B=131072, tables=tuple(TableSpec(4_000_000, 128, L, ids) for _ in range(32)),
        wdtype="f16", itype="i64", weighted=False, optimizer="adagrad", lr=0.01, eps=1e-8,
        w_scale=0.01, bad_id_frac=0.0, seed=2)


def _c4() -> TBEConfig:
    hist = TableSpec(64, 128, LengthSpec("fixed", 256), IdSpec("uniform"), histogram=True)
    companion = TableSpec(1_000_000, 128, LengthSpec("poisson", 10.0), IdSpec("uniform"))
    return TBEConfig(
        name="c4_hist",
        description="feature 0: E=64, D=128 fp16, L=256, uniform ids (counts x table path); "
                    "feature 1: E=1M, D=128 fp16, L~Poisson(10), uniform ids (gather); "
                    "B=65536, unweighted, int64, row-wise Adagrad lr=0.01 eps=1e-8",
        B=65536, tables=(hist, companion), wdtype="f16", itype="i64", weighted=False,
        optimizer="adagrad", lr=0.01, eps=1e-8, w_scale=0.01, bad_id_frac=0.0, seed=3)


def _c5() -> TBEConfig:
    rng = np.random.default_rng(np.random.SeedSequence([4, 0xE]))
    Es = _log_uniform_ints(rng, 50_000, 2_000_000, 64)
    Ds = [int(d) for d in rng.choice(np.array([32, 64, 128, 256]), size=64)]
    L = LengthSpec("poisson", 30.0, empty_frac=0.05)
    ids = IdSpec("zipf", s=1.1, q=0.0)
    return TBEConfig(
        name="c5_mixed",
        description="T=64, D uniform over {32,64,128,256}, E log-uniform 50k-2M, bf16 "
                    "~U(-0.01,0.01), B=16384, L~Poisson(30) with 5% of bags empty, psw~U(0,1), "
                    "Zipf(s=1.1) ids with 0.1% out of range, int64, row-wise Adagrad",
        B=16384, tables=tuple(TableSpec(E, D, L, ids) for E, D in zip(Es, Ds)), wdtype="bf16",
        itype="i64", weighted=True, optimizer="adagrad", lr=0.01, eps=1e-8, w_scale=0.01,
        bad_id_frac=0.001, seed=4)


CONFIGS = {c.name: c for c in (_c1(), _c2(), _c3(), _c4(), _c5())}


def get_config(name: str) -> TBEConfig:
    for key, cfg in CONFIGS.items():
        if key == name or key.split("_")[0] == name:
            return cfg
    raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
