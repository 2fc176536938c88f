"""Memory-balancing stage solver: the brute-force oracle against hand-worked
cases, then the library's exact solver against the oracle (CPU only).

The pages describe the solver (ninfer pipeline-stages.md, "How it works":
solve_stage_plan, "maximum page groups every stage can hold, then least-full
stage"; if nothing fits, the layers dealt evenly) and how it was checked
("Verification": against a brute-force partition enumeration) and what the
default split does ("Verification": the head stage gets fewer layers, a device
with twice the memory gets more). They print no worked numbers, so the pins
below are small cases solved by hand.
"""
import random

import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
from oracle import stage_solver as orc

# ---------------------------------------------------------------------------
# pins: the oracle against hand-worked cases (each takes the oracle module, so
# that the mutant test below can run them on planted mistakes too)
# ---------------------------------------------------------------------------


def pin_one_stage_closed_form(mod):
    # one stage: P = floor((free - fixed - sum W) / sum U) = floor((1000 - 100 - 60) / 7) = 120
    assert mod.solve([10, 20, 30], [1, 2, 4], [1000], [100]) == ([], 120)


def pin_even_layers_even_split(mod):
    # 4 layers of 10 B + 1 B per unit, two stages of 100 B: the 2/2 split gives
    # 20 + 2P <= 100 -> P = 40; 1/3 gives 30 + 3P <= 100 -> P = 23
    assert mod.solve([10] * 4, [1] * 4, [100, 100]) == ([2], 40)


def pin_twice_the_memory_gets_more_layers(mod):
    # 6 layers of 10 B + 1 B per unit; stage 1 has twice the memory.
    # cuts 2: min((100-20)/2, (200-40)/4) = min(40, 40) = 40; cuts 3: min(70/3=23, 170/3=56) = 23;
    # cuts 1: min(90, 150/5=30) = 30 -> cut 2, the bigger stage holds 4 of 6
    cuts, units = mod.solve([10] * 6, [1] * 6, [100, 200])
    assert (cuts, units) == ([2], 40)
    assert 6 - cuts[0] > cuts[0]


def pin_head_stage_gets_fewer_layers(mod):
    # 8 layers of 10 B + 1 B per unit, two stages of 100 B, the last one also holding a
    # 30 B head. Cut c: stage 0 allows (100 - 10c) / c units, stage 1 (10c - 10) / (8 - c).
    # c = 4: min(15, 7) = 7; c = 5: min(10, 13) = 10; c = 6: min(6, 25) = 6 -> c = 5,
    # the head stage holds 3 of the 8 layers
    assert mod.solve([10] * 8, [1] * 8, [100, 100], [0, 30]) == ([5], 10)


def pin_nothing_fits_deals_evenly(mod):
    # 5 layers of 10 B over two stages of 15 B: some stage holds at least three layers
    # (30 B), so nothing fits; the even split of 5 layers over 2 stages is cut 1 * 5 // 2 = 2
    assert mod.solve([10] * 5, [0] * 5, [15, 15]) == ([2], -1)
    # 7 layers over 3 stages: cuts 7 // 3 = 2 and 14 // 3 = 4
    assert mod.solve([10] * 7, [0] * 7, [5, 5, 5]) == ([2, 4], -1)


def pin_small_stage_between_large_layers(mod):
    # layers 1, 1, 9, 1 over stages of 2, 1, 10 bytes: the only plan that fits
    # gives stage 1 exactly layer 1 (cuts 1, 2); stage 0 taking both small
    # layers would leave stage 1 the 9-byte layer
    assert mod.solve([1, 1, 9, 1], [0, 0, 0, 0], [2, 1, 10], max_units=50) == ([1, 2], 50)


def pin_fraction_breaks_capacity_ties(mod):
    # zero unit bytes: every fitting plan has capacity max_units; the fullest
    # stage decides. layers 5, 5, 5, 5, stages 40 and 10: cuts 3 -> max(15/40, 5/10) = 1/2,
    # cuts 2 -> max(10/40, 10/10) = 1 (fits exactly), cuts 1 -> 15/10 does not fit
    assert mod.solve([5] * 4, [0] * 4, [40, 10], max_units=9) == ([3], 9)


def pin_fraction_counts_the_units(mod):
    # the fullest stage is judged at the solved capacity, units included: layers 10, 10, 10,
    # unit bytes 0, 0, 5, stages of 100 and 100, max 4 units. Cuts 1: stage 1 holds 20 + 4*5 = 40;
    # cuts 2: stage 0 holds 20, stage 1 holds 10 + 20 = 30 -> max(20/100, 30/100) beats
    # max(10/100, 40/100): cuts 2 (without the units cuts 1 and 2 would both be 20/100)
    assert mod.solve([10, 10, 10], [0, 0, 5], [100, 100], max_units=4) == ([2], 4)


def pin_lexicographic_among_equals(mod):
    # two identical stages, 3 equal layers, no unit bytes: cuts 1 and 2 are mirror
    # images with the same fullest fraction (20/30); the first in lexicographic order wins
    assert mod.solve([10] * 3, [0] * 3, [30, 30], max_units=5) == ([1], 5)


def pin_capacity_capped(mod):
    assert mod.stage_capacity(100, 0, 0, 0, 77) == 77
    assert mod.stage_capacity(100, 10, 20, 7, 1000) == 10
    assert mod.stage_capacity(100, 90, 20, 1, 1000) == -1
    assert mod.stage_capacity(100, 10, 20, 7, 5) == 5


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc)


# plausible mistakes planted in copies of the oracle: every one must fail a pin
MUTANTS = {
    "capacity_off_by_one": ("return min(max_units, room // unit)", "return min(max_units, room // unit + 1)"),
    "fixed_bytes_ignored": ("room = free - fixed - weights", "room = free - weights"),
    "capacity_not_capped": ("return min(max_units, room // unit)", "return room // unit"),
    "one_layer_unit_bytes": ("u = sum(layer_unit_bytes[fence[s]:fence[s + 1]])", "u = layer_unit_bytes[fence[s]]"),
    "plan_capacity_max": ("return min(caps)", "return max(caps)"),
    "fullest_without_units": ("+ P * sum(layer_unit_bytes[fence[s]:fence[s + 1]])", ""),
    "fraction_reversed": ("frac < best[1]", "frac > best[1]"),
    "last_of_equals": ("(cap == best[0] and frac < best[1])", "(cap == best[0] and frac <= best[1])"),
    "even_split_shifted": ("[s * L // N for s in range(1, N)]", "[(s * L + N - 1) // N for s in range(1, N)]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    import types
    old, new = MUTANTS[name]
    src = open(orc.__file__).read()
    assert src.count(old) == 1, f"mutant {name}: snippet not found once"
    mod = types.ModuleType(f"stage_solver_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the mutant {name}"


# ---------------------------------------------------------------------------
# the library's solver against the oracle
# ---------------------------------------------------------------------------


def _random_case(rng):
    L = rng.randint(1, 9)
    N = rng.randint(1, min(L, 4))
    lb = [rng.choice([0, 1, 2, 5, 10, 17, 40]) * rng.randint(1, 4) for _ in range(L)]
    lu = [rng.choice([0, 0, 1, 2, 3, 8]) for _ in range(L)]
    total = sum(lb) + 1
    free = [rng.randint(max(1, total // (2 * N)), 2 * total) for _ in range(N)]
    fixed = [rng.choice([0, 0, 1, 7, total // 4]) for _ in range(N)] if rng.random() < 0.6 else None
    max_units = rng.choice([0, 3, 64, 1 << 20])
    return lb, lu, free, fixed, max_units


def test_library_matches_brute_force_on_random_cases():
    rng = random.Random(20261202)
    for _ in range(3000):
        lb, lu, free, fixed, mu = _random_case(rng)
        want = orc.solve(lb, lu, free, fixed, mu)
        got = lps.stage_plan_solve(lb, lu, free, fixed, mu)
        assert got == want, (lb, lu, free, fixed, mu, got, want)


def test_library_matches_brute_force_on_larger_cases():
    # up to 14 layers over 5 stages (1001 plans each), layer sizes of two orders of magnitude
    rng = random.Random(77)
    for _ in range(150):
        L = rng.randint(8, 14)
        N = rng.randint(2, 5)
        lb = [rng.choice([100, 150, 900, 1000, 1100]) for _ in range(L)]
        lu = [rng.choice([1, 2, 3]) for _ in range(L)]
        free = [rng.randint(sum(lb) // N, 2 * sum(lb) // N + 500) for _ in range(N)]
        fixed = [rng.choice([0, 50, 400]) for _ in range(N)]
        assert lps.stage_plan_solve(lb, lu, free, fixed, 10**6) == orc.solve(lb, lu, free, fixed, 10**6)


def test_library_matches_brute_force_on_pins():
    cases = [([10, 20, 30], [1, 2, 4], [1000], [100], 1 << 40), ([10] * 8, [1] * 8, [100, 100], [0, 30], 1 << 40),
             ([1, 1, 9, 1], [0] * 4, [2, 1, 10], None, 50), ([10] * 5, [0] * 5, [15, 15], None, 9),
             ([5] * 4, [0] * 4, [40, 10], None, 9), ([10] * 3, [0] * 3, [30, 30], None, 5),
             ([10, 10, 10], [0, 0, 5], [100, 100], None, 4), ([10] * 7, [0] * 7, [5, 5, 5], None, 3)]
    for lb, lu, free, fixed, mu in cases:
        assert lps.stage_plan_solve(lb, lu, free, fixed, mu) == orc.solve(lb, lu, free, fixed, mu)


def test_library_handles_large_byte_counts():
    # 64-bit byte counts and a large unit count: the exact 128-bit arithmetic
    lb = [2**40] * 6
    lu = [2**20] * 6
    free = [2**43, 2**44, 2**43]
    got = lps.stage_plan_solve(lb, lu, free, None, 2**40)
    assert got == orc.solve(lb, lu, free, None, 2**40)


def test_library_refuses_bad_arguments():
    with pytest.raises(lps.LpsError):
        lps.stage_plan_solve([1, 2], [0, 0], [10, 10, 10])  # more stages than layers
    with pytest.raises(lps.LpsError):
        lps.stage_plan_solve([1, 2], [0, 0], [10, 0])  # a stage with no memory
    with pytest.raises(lps.LpsError):
        lps.stage_plan_solve([1, 2], [0, 0], [10, 10], max_units=-1)


# ---------------------------------------------------------------------------
# the byte model of a bound model, and a plan that stage_plan_create accepts
# ---------------------------------------------------------------------------

DESC_8B = dict(n_layers=32, n_embd=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn=14336, vocab=128256,
               weight_dtype=0, kv_dtype=0, max_ctx=8448, batch=1, pending_depth=4, rope_theta=10000.0,
               rms_eps=1e-5, flags=0)


def test_model_stage_bytes_8b():
    b = lps.model_stage_bytes(DESC_8B)
    # QKV 6144 x 4096, o 4096 x 4096, gate + up 2 x 14336 x 4096, down 4096 x 14336, bf16; two f32 norms
    w = (6144 * 4096 + 4096 * 4096 + 2 * 14336 * 4096 + 4096 * 14336) * 2 + 2 * 4096 * 4
    assert b["layer_bytes"].tolist() == [w] * 32
    assert b["layer_unit_bytes"].tolist() == [1 * 8 * 128 * 2 * 2] * 32  # K and V rows, bf16
    assert b["first_stage_bytes"] == 128256 * 4096 * 2
    assert b["last_stage_bytes"] >= 128256 * 4096 * 2 + 5 * 128256 * 4


def test_model_stage_bytes_int8_scales():
    d = dict(DESC_8B, weight_dtype=1, batch=8)
    b = lps.model_stage_bytes(d)
    rows = 6144 + 4096 + 2 * 14336 + 4096
    w = (6144 * 4096 + 4096 * 4096 + 2 * 14336 * 4096 + 4096 * 14336) + rows * 4 + 2 * 4096 * 4
    assert b["layer_bytes"][0] == w
    assert b["layer_unit_bytes"][0] == 8 * 8 * 128 * 2 * 2


def test_solved_plan_for_the_8b_shape():
    b = lps.model_stage_bytes(DESC_8B)
    every = b["every_stage_bytes"]
    fixed = [every + b["first_stage_bytes"], every, every, every + b["last_stage_bytes"]]
    # four stages sharing one device's 80 GB: 20 GB each
    free = [20 * 10**9] * 4
    cuts, units = lps.stage_plan_solve(b["layer_bytes"], b["layer_unit_bytes"], free, fixed, max_units=1 << 30)
    assert units > 0
    plan = lps.stage_plan_create(32, cuts)
    counts = np.diff(plan.fence)
    # the stages with the embedding and the head hold fewer layers than the middle ones
    assert counts[0] <= counts[1] and counts[3] <= counts[2]
    # and the capacity is the largest the per-stage budget allows for that split
    assert units == min(
        (free[s] - fixed[s] - int(counts[s]) * int(b["layer_bytes"][0])) // (int(counts[s]) * int(b["layer_unit_bytes"][0]))
        for s in range(4))
