"""ORACLE -- test infrastructure, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import, call or execute anything under ``oracle/``. This module shares no
code with the library's stage solver.

The memory-balancing stage plan by brute force (ninfer pipeline-stages.md,
"How it works": solve_stage_plan, "maximum page groups every stage can hold,
then least-full stage", and "Verification": the solver checked against a
brute-force partition enumeration). Every contiguous plan of n_layers layers
into n_stages non-empty stages is enumerated; a plan's capacity is the largest
number of units P in [0, max_units] at which every stage s fits,

    fixed[s] + sum(layer_bytes of s) + P * sum(layer_unit_bytes of s) <= free[s],

or -1 when some stage does not fit at P = 0. The answer is the plan with the
largest capacity; among those the smallest fullest-stage fraction
max_s(used_s / free[s]) at that capacity (exact rationals); among those the
first in lexicographic order of the cuts. When no plan fits at all, the even
split (cut s = s * n_layers / n_stages) and capacity -1.

Pins: ``tests/pins.py`` (hand-worked cases).
"""
from __future__ import annotations

import itertools
from fractions import Fraction


def stage_capacity(free: int, fixed: int, weights: int, unit: int, max_units: int) -> int:
    """The largest P in [0, max_units] with fixed + weights + P * unit <= free, or -1."""
    room = free - fixed - weights
    if room < 0:
        return -1
    if unit == 0:
        return max_units
    return min(max_units, room // unit)


def plan_capacity(fence, layer_bytes, layer_unit_bytes, stage_free, stage_fixed, max_units) -> int:
    caps = []
    for s in range(len(fence) - 1):
        w = sum(layer_bytes[fence[s]:fence[s + 1]])
        u = sum(layer_unit_bytes[fence[s]:fence[s + 1]])
        caps.append(stage_capacity(stage_free[s], stage_fixed[s], w, u, max_units))
    return min(caps)


def fullest_fraction(fence, P, layer_bytes, layer_unit_bytes, stage_free, stage_fixed) -> Fraction:
    worst = Fraction(0)
    for s in range(len(fence) - 1):
        used = stage_fixed[s] + sum(layer_bytes[fence[s]:fence[s + 1]]) + P * sum(layer_unit_bytes[fence[s]:fence[s + 1]])
        worst = max(worst, Fraction(used, stage_free[s]))
    return worst


def solve(layer_bytes, layer_unit_bytes, stage_free, stage_fixed=None, max_units: int = 1 << 40):
    """(cuts, units) by enumerating every plan (small cases only)."""
    L, N = len(layer_bytes), len(stage_free)
    fixed = list(stage_fixed) if stage_fixed is not None else [0] * N
    best = None  # (capacity, fraction, cuts)
    for cuts in itertools.combinations(range(1, L), N - 1):  # lexicographic order
        fence = (0, *cuts, L)
        cap = plan_capacity(fence, layer_bytes, layer_unit_bytes, stage_free, fixed, max_units)
        if cap < 0:
            continue
        frac = fullest_fraction(fence, cap, layer_bytes, layer_unit_bytes, stage_free, fixed)
        if best is None or cap > best[0] or (cap == best[0] and frac < best[1]):
            best = (cap, frac, list(cuts))
    if best is None:
        return [s * L // N for s in range(1, N)], -1
    return best[2], best[0]
