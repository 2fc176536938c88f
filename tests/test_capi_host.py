"""The C-ABI library on the CPU: it loads, exports every declared entry point,
and its host-only stage-plan logic matches the plans printed on the pages.
No compute calls are made here."""
import json
import os
import re

import pytest

import layer_pipeline_staged_gb300 as lps
from layer_pipeline_staged_gb300 import _capi
from layer_pipeline_staged_gb300 import build as lps_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    lps_build.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "lps.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = [ln for ln in src.splitlines() if not ln.lstrip().startswith("typedef")]
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:long\s+)?\w+\s*\*?\s*(\w+)\s*\(", "\n".join(lines), flags=re.M)))


def test_exports_every_declared_symbol():
    L = lps.load()
    declared = _declared()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(_capi.EXPORTS) == declared


def test_golden_stage_plans():
    data = json.load(open(os.path.join(ROOT, "tests", "golden", "stage_plans.json")))
    for g in data["plans"]:
        if "counts" in g:
            plan = lps.stage_plan_from_counts(g["counts"])
            cuts_plan = lps.stage_plan_create(g["n_layers"], cuts=g["fence"][1:-1])
            assert cuts_plan.fence == tuple(g["fence"])
        else:
            plan = lps.stage_plan_create(g["n_layers"], n_stages=g["even_stages"])
        assert plan.fence == tuple(g["fence"]), g["source"]
        for il, s in g["stage_of"].items():
            assert plan.stage_of(int(il)) == s, (g["source"], il)


@pytest.mark.parametrize("n_layers,cuts", [(4, [0]), (4, [4]), (4, [2, 2]), (4, [3, 1]), (4, [-1]), (8, [1, 9])])
def test_bad_cuts_refused(n_layers, cuts):
    with pytest.raises(lps.LpsError) as e:
        lps.stage_plan_create(n_layers, cuts=cuts)
    assert e.value.code == lps.LPS_EINVAL
    assert "stage_plan_create" in str(e.value)


def test_even_split_matches_formula():
    for n_layers in range(1, 40):
        for N in range(1, n_layers + 1):
            plan = lps.stage_plan_create(n_layers, n_stages=N)
            assert plan.fence == tuple([s * n_layers // N for s in range(N)] + [n_layers])
            owners = [plan.stage_of(il) for il in range(n_layers)]
            assert owners == sorted(owners) and len(set(owners)) == N


def test_counts_refuse_empty_stage_and_stage_of_range():
    with pytest.raises(lps.LpsError):
        lps.stage_plan_from_counts([3, 0, 2])
    plan = lps.stage_plan_from_counts([1, 2])
    with pytest.raises(lps.LpsError):
        plan.stage_of(3)
    with pytest.raises(lps.LpsError):
        plan.stage_of(-1)
    assert plan.n_stages == 2
