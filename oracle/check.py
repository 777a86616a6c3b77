"""Parity checker (test infrastructure).

The acceptance rule for a fast implementation against the fp64 oracle:
  * each histogram sums to exactly the oracle's total (n1 * n2);
  * each bin equals the oracle's bin exactly, except that pairs whose fp64 theta lies within
    1e-6 rad of a bin edge may land in the bin on the other side of that edge.

Given only histograms, the rule is checked through cumulative counts. Let C(K) = sum_{k<=K} h[k].
A pair can cross the edge between bins K and K+1 only if it is in that edge's window, so the
net flow D(K) = C_oracle(K) - C_fast(K) across the edge must satisfy
    -near_above[K+1] <= D(K) <= near_below[K+1].
With bins wider than twice the tolerance no pair is near two edges, so this is equivalent to the
rule. When both windows of every edge are empty the histograms must be equal bin for bin.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class ParityReport:
    ok: bool
    sum_fast: int
    sum_oracle: int
    bins_differing: int
    moved_pairs: int                      # sum over edges of |net flow|
    violations: list = field(default_factory=list)   # (edge K, net flow, -near_above, near_below)

    def __str__(self) -> str:
        s = "ok" if self.ok else "FAIL"
        return (f"{s}: sums fast={self.sum_fast} oracle={self.sum_oracle}, bins differing={self.bins_differing}, "
                f"net moved pairs={self.moved_pairs}, violations={self.violations[:5]}")


def edge_flux(fast_hist, oracle_hist, near_below, near_above) -> ParityReport:
    f = np.asarray(fast_hist, dtype=np.uint64).astype(object)
    o = np.asarray(oracle_hist, dtype=np.uint64).astype(object)
    lo = np.asarray(near_below, dtype=np.uint64).astype(object)
    hi = np.asarray(near_above, dtype=np.uint64).astype(object)
    nb = len(o)
    assert len(f) == nb and len(lo) == nb + 1 and len(hi) == nb + 1
    sf, so = int(sum(f)), int(sum(o))
    viol = []
    moved = 0
    cf = co = 0
    for k in range(nb - 1):
        cf += int(f[k])
        co += int(o[k])
        d = co - cf
        moved += abs(d)
        if d > int(lo[k + 1]) or d < -int(hi[k + 1]):
            viol.append((k + 1, d, -int(hi[k + 1]), int(lo[k + 1])))
    differing = int(sum(1 for a, b in zip(f, o) if a != b))
    ok = (sf == so) and not viol
    return ParityReport(ok, sf, so, differing, moved, viol)


def omega_close(omega_a, omega_b, rel: float = 1e-12) -> bool:
    """Two omega vectors agree to ``rel`` relative (NaN where both are NaN)."""
    a = np.asarray(omega_a, dtype=np.float64)
    b = np.asarray(omega_b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    na, nb = np.isnan(a), np.isnan(b)
    if not np.array_equal(na, nb):
        return False
    m = ~na
    return bool(np.all(np.abs(a[m] - b[m]) <= rel * np.maximum(np.abs(b[m]), 1e-300) + 1e-300))
