"""The launch trace (model_trace_*): one record per launch in launch order, with
device start/end times, and no change to the results."""
import numpy as np
import pytest

import synth
from workloads import bind

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["tiny"]


def test_trace_records_every_launch_in_order():
    w = synth.make_weights(TINY)
    toks = synth.make_tokens(TINY, 3)
    plain = bind(TINY, w)
    ref = [plain.decode_step(toks[t], t) for t in range(3)]

    m = bind(TINY, w)
    m.trace_enable(1024)
    got = [m.decode_step(toks[t], t) for t in range(3)]
    recs, dropped = m.trace_read()
    assert dropped == 0
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)  # tracing changes no result

    fence = TINY.fence
    per_step = ["embed"] + ["qkv", "attn", "oproj", "gateup", "down"] * TINY.n_layers + ["head"]
    assert len(recs) == 3 * len(per_step)
    steps = sorted({r["step"] for r in recs})
    assert len(steps) == 3 and steps == list(range(steps[0], steps[0] + 3))
    for t in range(3):
        rs = [r for r in recs if r["step"] == steps[t]]
        assert [r["kind"] for r in rs] == per_step
        layers = [r["layer"] for r in rs[1:-1]]
        assert layers == [l for l in range(TINY.n_layers) for _ in range(5)]
        for r in rs[1:-1]:
            assert fence[r["stage"]] <= r["layer"] < fence[r["stage"] + 1]
        assert rs[0]["stage"] == 0 and rs[-1]["stage"] == len(fence) - 2
        for r in rs:
            assert 0 < r["start_ns"] <= r["end_ns"]
        for s in range(len(fence) - 1):  # one stream per stage: its launches start in order
            starts = [r["start_ns"] for r in rs if r["stage"] == s]
            assert starts == sorted(starts)


def test_trace_capacity_counts_dropped_launches():
    w = synth.make_weights(TINY)
    m = bind(TINY, w)
    m.trace_enable(5)
    m.decode_step(synth.make_tokens(TINY, 1)[0], 0)
    recs, dropped = m.trace_read()
    assert len(recs) == 5 and dropped == 2 + 5 * TINY.n_layers - 5
    m.trace_disable()
