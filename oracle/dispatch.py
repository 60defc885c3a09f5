"""Shape- and error-driven variant selection (LoKA Dispatch).

TEST INFRASTRUCTURE ONLY (see the package docstring).

LoKA page, section III-C "Library and Recipe Selection": for each GEMM the
candidate implementations are first filtered by the expected error from the
probe (typically MERE < 0.2) and by the speedup over the high-precision path
(typically > 1.05x); from the survivors the one with the highest measured
throughput is chosen.  Section VI "Limitations": when no candidate qualifies,
low precision is disabled for that layer (the BF16 path runs).

Readings (the pages leave these open):
  * Table rows are measured (problem, variant, time, rel_err, mere) records.
    A query matches rows with the same N, K and norm; among those the rows
    whose M is nearest in log2 (ties: larger M) and whose outlier fraction is
    nearest (ties: larger fraction) form the candidate set.
  * Filters: rel_err <= max_rel_err; mere < max_mere when max_mere >= 0;
    t_bf16 / t > min_speedup when min_speedup >= 0 and a BF16 row exists
    (without a BF16 row the speedup filter rejects every FP8 candidate).
  * Among survivors: smallest time; ties -> smaller rel_err -> smaller
    variant id.  No survivor, or no matching row -> BF16 (variant 3).
"""
from __future__ import annotations

import math
from typing import Iterable, List, NamedTuple

BF16_VARIANT = 3


class Entry(NamedTuple):
    M: int
    N: int
    K: int
    norm: int
    outlier_frac: float
    variant: int
    time_us: float
    rel_err: float
    mere: float


class Policy(NamedTuple):
    max_rel_err: float = 1e-2
    max_mere: float = 0.2
    min_speedup: float = -1.0


def candidates(table: Iterable[Entry], M: int, N: int, K: int, norm: int, outlier_frac: float) -> List[Entry]:
    rows = [e for e in table if e.N == N and e.K == K and e.norm == norm]
    if not rows:
        return []
    dm = min(abs(math.log2(e.M) - math.log2(M)) for e in rows)
    rows = [e for e in rows if abs(math.log2(e.M) - math.log2(M)) == dm]
    best_m = max(e.M for e in rows)
    rows = [e for e in rows if e.M == best_m]
    do = min(abs(e.outlier_frac - outlier_frac) for e in rows)
    rows = [e for e in rows if abs(e.outlier_frac - outlier_frac) == do]
    best_o = max(e.outlier_frac for e in rows)
    return [e for e in rows if e.outlier_frac == best_o]


def select(table: Iterable[Entry], M: int, N: int, K: int, norm: int, outlier_frac: float,
           policy: Policy = Policy()) -> int:
    rows = candidates(table, M, N, K, norm, outlier_frac)
    if not rows:
        return BF16_VARIANT
    bf16 = [e for e in rows if e.variant == BF16_VARIANT]
    t_ref = min(e.time_us for e in bf16) if bf16 else None
    keep = []
    for e in rows:
        if not e.rel_err <= policy.max_rel_err:
            continue
        if policy.max_mere >= 0 and not e.mere < policy.max_mere:
            continue
        if policy.min_speedup >= 0 and e.variant != BF16_VARIANT:
            if t_ref is None or not (t_ref / e.time_us > policy.min_speedup):
                continue
        keep.append(e)
    if not keep:
        return BF16_VARIANT
    keep.sort(key=lambda e: (e.time_us, e.rel_err, e.variant))
    return keep[0].variant
