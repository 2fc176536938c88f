"""The decoder workloads at their own shapes, on the GPU, against the oracle.

- zero-padded heads (48 q / 12 kv over a 32/8 model, GQA 4 kept): dummy heads'
  attention outputs are exactly zero; padded logits match the unpadded
  model's within tolerance; both match the oracle;
- the 1B-shape decoder over its whole teacher-forced sequence (1024 + 128);
- full contexts (8B at 8192 with 4 stages and deferred readback, 8B-q8 at
  32768 with batch 1 and 8): a state transplant -- the same cache rows are
  imported into both sides -- then decode steps in the launch configuration
  the benchmark times, compared at every sequence.
"""
import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from workloads import assert_close, bind, iter_random_kv

pytestmark = pytest.mark.gpu


def _deferred_steps(m, toks, pos0, depth=4):
    pend, got = [], []
    for t in range(len(toks)):
        pend.append(m.decode_step_deferred(toks[t], pos0 + t))
        if len(pend) == depth:
            p = pend.pop(0)
            got.append(p.wait())
            p.free()
    for p in pend:
        got.append(p.wait())
        p.free()
    return np.stack(got)


@pytest.fixture(scope="module")
def padded():
    cfg = synth.CONFIGS["padded"]
    return cfg, synth.make_weights(cfg), synth.make_weights(cfg.base())


def test_padded_dummy_heads_zero_and_match_unpadded(padded):
    cfg, wp, wb = padded
    T = 8
    toks = synth.make_tokens(cfg, T)
    mp = bind(cfg, wp, max_ctx=T, flags=lps.LPS_FLAG_KEEP_ATTN_OUT)
    mb = bind(cfg.base(), wb, max_ctx=T)
    orc = oracle.Oracle(cfg, wp, max_ctx=T)
    for t in range(T):
        lp = mp.decode_step(toks[t], t)
        lb = mb.decode_step(toks[t], t)
        ref = orc.step(toks[t], t)
        assert_close(lp, ref, cfg, f"padded vs oracle, step {t}")
        assert_close(lp, lb, cfg, f"padded vs unpadded, step {t}")
    for l in (0, 5, 6, 14, 15, 23):  # layers on every stage
        for b in range(cfg.batch):
            o = mp.attn_out(l, b)
            assert np.all(o[cfg.n_q_heads:] == 0.0), (l, b)
            assert np.all(np.abs(o[:cfg.n_q_heads]).sum(axis=1) > 0), (l, b)
    assert mp.stats()["fence"] == (0, 6, 15, 24)


def test_padded_full_context_transplant(padded):
    cfg, wp, _ = padded
    P = cfg.ctx
    max_ctx = P + 4
    m = bind(cfg, wp, max_ctx=max_ctx)
    orc = oracle.Oracle(cfg, wp, max_ctx=max_ctx)
    for (l, b), (k, v) in iter_random_kv(cfg, 41, cfg.n_layers, max_ctx, P):
        m.kv_import(l, b, k, v, P)
        orc.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(cfg, 2, seed=cfg.seed_t + 3)
    got = _deferred_steps(m, toks, P)
    for t in range(2):
        assert_close(got[t], orc.step(toks[t], P + t), cfg, f"step {t}")


def test_1b_whole_sequence():
    cfg = synth.CONFIGS["1b"]
    T = cfg.ctx + cfg.steps
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, T)
    orc = oracle.Oracle(cfg, w, max_ctx=T)
    m4 = bind(cfg, w, max_ctx=T)
    got = _deferred_steps(m4, toks, 0)
    worst = 0.0
    for t in range(T):
        worst = max(worst, assert_close(got[t], orc.step(toks[t], t), cfg, f"step {t}"))
    m1 = bind(cfg, w, max_ctx=T, fence=(0, cfg.n_layers))
    assert np.array_equal(np.stack([m1.decode_step(toks[t], t) for t in range(T)]), got)
    st = m4.stats()
    assert st["boundary_crossings"] == 3 * T and st["deferred_steps"] == T


@pytest.mark.parametrize("name", ["8b", "8b_q8", "8b_q8_b8"])
def test_full_context_transplant(name):
    cfg = synth.CONFIGS[name]
    P = cfg.ctx
    max_ctx = P + 2
    w = synth.make_weights(cfg)
    m = bind(cfg, w, max_ctx=max_ctx, pending_depth=4)
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    for (l, b), (k, v) in iter_random_kv(cfg, 43, cfg.n_layers, max_ctx, P):
        m.kv_import(l, b, k, v, P)
        orc.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(cfg, 2, seed=cfg.seed_t + 5)
    got = _deferred_steps(m, toks, P)
    for t in range(2):
        assert_close(got[t], orc.step(toks[t], P + t), cfg, f"{name} step {t}")
    # the rows this step wrote: the GPU's and the oracle's agree within one bf16 rounding
    for l in (0, cfg.n_layers - 1):
        kg, vg = m.kv_export(l, 0)
        ko, vo = orc.kv_export(l, 0)
        for g_, o_ in ((kg, ko), (vg, vo)):
            a = synth.bf16_to_f32(g_[:, P:P + 2]).astype(np.float64)
            b = synth.bf16_to_f32(o_[:, P:P + 2]).astype(np.float64)
            scale = np.max(np.abs(b), axis=2, keepdims=True)
            assert np.all(np.abs(a - b) <= np.abs(b) * 2 ** -7 + 1e-4 * scale)
            assert np.array_equal(g_[:, :P], o_[:, :P])
