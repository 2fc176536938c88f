"""The launch trace (model_trace_*): one record per launch in launch order, with
device start/end times, and no change to the results."""
import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import synth
from workloads import bind

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["tiny"]


def _per_step(persistent: bool):
    """Records of one step: one per launch (chained kernels) or one per phase of
    the persistent stage kernels (with the merge of the attention chunks)."""
    layer = ["qkv", "attn", "merge", "oproj", "gateup", "down"] if persistent else ["qkv", "attn", "oproj",
                                                                                     "gateup", "down"]
    return ["embed"] + layer * TINY.n_layers + ["head"], len(layer)


@pytest.mark.parametrize("flags", [lps.LPS_FLAG_PERSISTENT, 0], ids=["persistent", "chained"])
def test_trace_records_every_launch_in_order(flags):
    w = synth.make_weights(TINY)
    toks = synth.make_tokens(TINY, 3)
    plain = bind(TINY, w, flags=flags)
    ref = [plain.decode_step(toks[t], t) for t in range(3)]

    m = bind(TINY, w, flags=flags)
    m.trace_enable(1024)
    got = [m.decode_step(toks[t], t) for t in range(3)]
    recs, dropped = m.trace_read()
    assert dropped == 0
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)  # tracing changes no result

    fence = TINY.fence
    per_step, nl = _per_step(flags != 0)
    assert len(recs) == 3 * len(per_step)
    steps = sorted({r["step"] for r in recs})
    assert len(steps) == 3 and steps == list(range(steps[0], steps[0] + 3))
    for t in range(3):
        rs = [r for r in recs if r["step"] == steps[t]]
        assert [r["kind"] for r in rs] == per_step
        layers = [r["layer"] for r in rs[1:-1]]
        assert layers == [l for l in range(TINY.n_layers) for _ in range(nl)]
        for r in rs[1:-1]:
            assert fence[r["stage"]] <= r["layer"] < fence[r["stage"] + 1]
        assert rs[0]["stage"] == 0 and rs[-1]["stage"] == len(fence) - 2
        for r in rs:
            assert 0 < r["start_ns"] <= r["end_ns"]
        for s in range(len(fence) - 1):  # a stage's launches (or phases) start in order
            starts = [r["start_ns"] for r in rs if r["stage"] == s]
            assert starts == sorted(starts)
        if flags:
            # phases of one persistent launch are separated by grid barriers: no
            # phase starts before the previous one has ended on every CTA
            for a, b in zip(rs, rs[1:]):
                if a["stage"] == b["stage"]:
                    assert b["start_ns"] >= a["end_ns"], (a, b)


@pytest.mark.parametrize("flags", [lps.LPS_FLAG_PERSISTENT, 0], ids=["persistent", "chained"])
def test_trace_capacity_counts_dropped_launches(flags):
    w = synth.make_weights(TINY)
    m = bind(TINY, w, flags=flags)
    per_step, _ = _per_step(flags != 0)
    # the persistent kernel records a launch's phases together or not at all:
    # room for stage 0's launch only
    cap = 1 + 6 * TINY.fence[1] + 2 if flags else 5
    m.trace_enable(cap)
    m.decode_step(synth.make_tokens(TINY, 1)[0], 0)
    recs, dropped = m.trace_read()
    kept = 1 + 6 * TINY.fence[1] if flags else 5
    assert len(recs) == kept and dropped == len(per_step) - kept
    m.trace_disable()


def test_trace_records_prefill_chunks_through_the_stages():
    """A 3-chunk prefill on 2 stages: every launch recorded with its chunk
    number; per chunk, stage 0 runs the embedding and its layers, stage 1 its
    layers (split, QKV GEMM, chunk attention, merge, o-proj GEMM, split, gate/up
    GEMM, down GEMM per layer), the last chunk ends with the LM head; stage 1
    starts chunk c only after stage 0 has finished it (the boundary slot's
    event). Tracing changes no result."""
    w = synth.make_weights(TINY)
    toks = synth.make_tokens(TINY, 48)
    plain = bind(TINY, w, max_ctx=48).prefill(toks, chunk=16)
    m = bind(TINY, w, max_ctx=48)
    m.prefill(toks[:16], chunk=16)  # the first call allocates the prefill buffers
    m.trace_enable(4096)
    got = m.prefill(toks, chunk=16)
    recs, dropped = m.trace_read()
    assert dropped == 0 and np.array_equal(got, plain)
    layer = ["pf_split", "pf_gemm", "pf_attn", "pf_merge", "pf_gemm", "pf_split", "pf_gemm", "pf_gemm"]
    fence = TINY.fence
    chunks = sorted({r["step"] for r in recs})
    assert len(chunks) == 3
    for i, c in enumerate(chunks):
        for s in range(len(fence) - 1):
            rs = [r for r in recs if r["step"] == c and r["stage"] == s and r["kind"] != "head"]
            want = (["embed"] if s == 0 else []) + layer * (fence[s + 1] - fence[s])
            assert [r["kind"] for r in rs] == want, (c, s)
            assert all(0 < r["start_ns"] <= r["end_ns"] for r in rs)
        s0 = [r for r in recs if r["step"] == c and r["stage"] == 0]
        s1 = [r for r in recs if r["step"] == c and r["stage"] == 1 and r["kind"] != "head"]
        assert min(r["start_ns"] for r in s1) >= max(r["end_ns"] for r in s0), c
    heads = [r for r in recs if r["kind"] == "head"]
    assert len(heads) == 1 and heads[0]["step"] == chunks[-1]
    # report how much of stage 1's chunk c ran while stage 0 ran chunk c + 1
    for a, b in zip(chunks, chunks[1:]):
        s1 = [r for r in recs if r["step"] == a and r["stage"] == 1 and r["kind"] != "head"]
        s0 = [r for r in recs if r["step"] == b and r["stage"] == 0]
        lo = max(min(r["start_ns"] for r in s1), min(r["start_ns"] for r in s0))
        hi = min(max(r["end_ns"] for r in s1), max(r["end_ns"] for r in s0))
        print(f"chunks {a}/{b}: stage 1 and stage 0 overlap for {max(0, hi - lo) / 1e3:.1f} us")
    m.trace_disable()
