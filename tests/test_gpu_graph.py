"""Whole-step CUDA graph (LPS_FLAG_GRAPH): each step captured from stage 0's
stream with the other stages forked and joined through the boundary events
(ninfer pipeline-stages.md, "StageLink": the decode pass as one graph), the
instantiated graph updated in place for the next position. The replayed steps
give the bits of the stream path."""
import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from workloads import assert_close, bind

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["tiny"]


def _eager(m, toks, pos0=0):
    return np.stack([m.decode_step(toks[t], pos0 + t) for t in range(len(toks))])


def _deferred(m, toks, pos0=0):
    pend, got = [], []
    for t in range(len(toks)):
        pend.append(m.decode_step_deferred(toks[t], pos0 + t))
        if len(pend) == 3:
            p = pend.pop(0)
            got.append(p.wait())
            p.free()
    for p in pend:
        got.append(p.wait())
        p.free()
    return np.stack(got)


@pytest.mark.parametrize("fence,flags", [((0, 1, 3, 4), 0), ((0, 4), 0), ((0, 2, 4), lps.LPS_FLAG_SINGLE_STREAM),
                                         ((0, 1, 2, 3, 4), lps.LPS_FLAG_SERIAL_STEPS)],
                         ids=["3-stages", "1-stage", "single-stream", "serial"])
def test_graph_steps_bit_identical_to_streams(fence, flags):
    w = synth.make_weights(TINY)
    toks = synth.make_tokens(TINY, 12)
    ref = _eager(bind(TINY, w, fence=fence, max_ctx=16, flags=flags), toks)
    g = bind(TINY, w, fence=fence, max_ctx=16, flags=flags | lps.LPS_FLAG_GRAPH, pending_depth=4)
    assert np.array_equal(_eager(g, toks), ref)
    # deferred replays, rewinding to position 0
    assert np.array_equal(_deferred(g, toks), ref)
    orc = oracle.Oracle(TINY, w, max_ctx=16)
    for t in range(3):
        assert_close(ref[t], orc.step(toks[t], t), TINY, f"step {t}")


def test_graph_1b_and_batch2_and_prefill():
    """The 1B shape on 4 stages (16 steps), a batch-2 model on the skinny GEMM,
    and graph steps after a prefill: each the stream path's bits."""
    cfg = synth.CONFIGS["1b"]
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, 16)
    ref = _eager(bind(cfg, w, max_ctx=16), toks)
    assert np.array_equal(_deferred(bind(cfg, w, max_ctx=16, flags=lps.LPS_FLAG_GRAPH, pending_depth=4), toks), ref)

    b2 = TINY.replace(name="tiny_b2", batch=2)
    w2 = synth.make_weights(b2)
    t2 = synth.make_tokens(b2, 8)
    r2 = _eager(bind(b2, w2, max_ctx=8), t2)
    assert np.array_equal(_eager(bind(b2, w2, max_ctx=8, flags=lps.LPS_FLAG_GRAPH), t2), r2)

    wt = synth.make_weights(TINY)
    tt = synth.make_tokens(TINY, 40)
    plain = bind(TINY, wt, max_ctx=40)
    graph = bind(TINY, wt, max_ctx=40, flags=lps.LPS_FLAG_GRAPH)
    for m in (plain, graph):
        m.prefill(tt[:32], chunk=16)
    assert np.array_equal(_eager(graph, tt[32:], 32), _eager(plain, tt[32:], 32))


def test_graph_refuses_the_persistent_kernel():
    w = synth.make_weights(TINY)
    with pytest.raises(lps.LpsError) as ei:
        bind(TINY, w, max_ctx=8, flags=lps.LPS_FLAG_GRAPH | lps.LPS_FLAG_PERSISTENT)
    assert ei.value.code == lps.LPS_EINVAL
