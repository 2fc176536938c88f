"""Chunked prefill through the stages (memra_engine::pp, prime_pp_on /
prime_pipe_on; ninfer pipeline-stages.md, "Prefill micro-chunk overlap"):
model_prefill against the oracle's decode of the same prompt, bit-identity
across stage plans and stream arms, and the argument checks."""
import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from workloads import assert_close, bind, random_kv

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["tiny"]


TINY_Q8 = TINY.replace(name="tiny_q8", index=97, weight_dtype="int8")


@pytest.fixture(scope="module")
def tiny():
    w = synth.make_weights(TINY)
    T = 80  # a 64-token prompt and 16 decode steps
    toks = synth.make_tokens(TINY, T)
    orc = oracle.Oracle(TINY, w, max_ctx=T)
    ref = np.stack([orc.step(toks[t], t) for t in range(T)])
    kv = [orc.kv_export(l, 0) for l in range(TINY.n_layers)]
    orc.close()
    return w, toks, ref, kv


def _kv_close(m, kv, layers, upto):
    """The cache rows [0, upto) the prefill wrote are the oracle's within a few bf16 roundings."""
    for l in layers:
        kg, vg = m.kv_export(l, 0)
        for g_, o_ in ((kg, kv[l][0]), (vg, kv[l][1])):
            a = synth.bf16_to_f32(g_[:, :upto]).astype(np.float64)
            b = synth.bf16_to_f32(o_[:, :upto]).astype(np.float64)
            scale = np.max(np.abs(b))
            assert np.max(np.abs(a - b)) <= 2e-2 * scale, (l, np.max(np.abs(a - b)) / scale)


def test_tiny_prefill_every_position(tiny):
    """Segments of 1 to 22 tokens (chunks of 16 inside a segment), each call
    returning its last token's logits: together every prompt position."""
    w, toks, ref, kv = tiny
    m = bind(TINY, w, max_ctx=80)
    pos, i = 0, 0
    lens = (1, 5, 16, 3, 17, 22)
    while pos < 64:
        n = min(lens[i % len(lens)], 64 - pos)
        lg = m.prefill(toks[pos:pos + n], pos0=pos, chunk=16)
        assert_close(lg, ref[pos + n - 1], TINY, f"prefill ending at position {pos + n - 1}")
        pos += n
        i += 1
    _kv_close(m, kv, range(TINY.n_layers), 64)
    # decode continues from the prefilled cache
    for t in range(64, 80):
        assert_close(m.decode_step(toks[t], t), ref[t], TINY, f"decode step {t} after prefill")


@pytest.mark.parametrize("chunk", [0, 16, 7])
def test_tiny_prefill_then_decode(tiny, chunk):
    w, toks, ref, _ = tiny
    m = bind(TINY, w, max_ctx=80)
    assert_close(m.prefill(toks[:64], chunk=chunk), ref[63], TINY, f"prefill (chunk {chunk})")
    for t in range(64, 80):
        assert_close(m.decode_step(toks[t], t), ref[t], TINY, f"decode step {t} (chunk {chunk})")


def _prefill_run(cfg, w, toks, P, steps, fence=None, flags=0, chunk=16):
    m = bind(cfg, w, fence=fence, max_ctx=P + steps, flags=flags)
    lg = m.prefill(toks[:P], chunk=chunk)
    kv = [m.kv_export(l, 0) for l in range(cfg.n_layers)]
    dec = np.stack([m.decode_step(toks[t], t) for t in range(P, P + steps)]) if steps else None
    m.close()
    return lg, kv, dec


def test_tiny_prefill_stage_plans_bit_identical(tiny):
    """The same prefill (and the decode after it) is the same bits under every
    cut of the 4 layers, with chunks overlapping across the stages."""
    w, toks, _, _ = tiny
    base = _prefill_run(TINY, w, toks, 64, 16, fence=(0, 4))
    for fence in ((0, 2, 4), (0, 1, 2, 3, 4), (0, 3, 4), (0, 1, 4)):
        got = _prefill_run(TINY, w, toks, 64, 16, fence=fence)
        assert np.array_equal(got[0], base[0]), fence
        for (kg, vg), (kb, vb) in zip(got[1], base[1]):
            assert np.array_equal(kg, kb) and np.array_equal(vg, vb), fence
        assert np.array_equal(got[2], base[2]), fence


def test_tiny_prefill_stream_arms(tiny):
    """The prefill kernels give the same bits on the single-stream arm and on
    a model that decodes on the persistent stage kernel."""
    w, toks, _, _ = tiny
    base = _prefill_run(TINY, w, toks, 64, 0)
    for flags in (lps.LPS_FLAG_SINGLE_STREAM, lps.LPS_FLAG_PERSISTENT, lps.LPS_FLAG_SERIAL_STEPS):
        got = _prefill_run(TINY, w, toks, 64, 0, flags=flags)
        assert np.array_equal(got[0], base[0]), flags
        for (kg, vg), (kb, vb) in zip(got[1], base[1]):
            assert np.array_equal(kg, kb) and np.array_equal(vg, vb), flags


def test_1b_prefill_context_then_decode():
    """The 1B shape: its 1024-token context prefilled in chunks of 128 through 4
    stages, then 32 decode steps, against the oracle's decode of the whole
    sequence; 4 stages bit-identical to 1 stage."""
    cfg = synth.CONFIGS["1b"]
    P, D = cfg.ctx, 32
    T = P + D
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, T)
    orc = oracle.Oracle(cfg, w, max_ctx=T)
    ref = np.stack([orc.step(toks[t], t) for t in range(T)])
    orc.close()
    got4 = _prefill_run(cfg, w, toks, P, D, chunk=0)
    assert_close(got4[0], ref[P - 1], cfg, "1B prefill, last prompt token")
    worst = 0.0
    for i in range(D):
        worst = max(worst, assert_close(got4[2][i], ref[P + i], cfg, f"1B decode step {P + i} after prefill"))
    print(f"1B prefill + decode: worst error {worst:.3e} x max|logit|")
    got1 = _prefill_run(cfg, w, toks, P, D, fence=(0, cfg.n_layers), chunk=0)
    assert np.array_equal(got1[0], got4[0])
    for (kg, vg), (kb, vb) in zip(got1[1], got4[1]):
        assert np.array_equal(kg, kb) and np.array_equal(vg, vb)
    assert np.array_equal(got1[2], got4[2])


def test_8b_prefill_over_oracle_cache():
    """The 8B shape (32 layers, 4 stages at cuts 8/16/24): over the oracle's own
    cache rows [0, t), a one-token prefill at position t matches the oracle's
    step t; a 256-token prefill in chunks of 128 on 4 stages is bit-identical
    to 1 stage, and so are the 16 deferred decode steps after it."""
    cfg = synth.CONFIGS["8b"]
    P, D = 256, 16
    T = P + D
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, T)
    orc = oracle.Oracle(cfg, w, max_ctx=T)
    ref = np.stack([orc.step(toks[t], t) for t in range(P)])
    kv = [orc.kv_export(l, 0) for l in range(cfg.n_layers)]
    orc.close()
    m = bind(cfg, w, max_ctx=T)
    for t in (0, 1, 77, 128, P - 1):
        for l in range(cfg.n_layers):
            m.kv_import(l, 0, kv[l][0], kv[l][1], t)
        assert_close(m.prefill(toks[t:t + 1], pos0=t), ref[t], cfg, f"8B one-token prefill at {t}")
    m.close()
    m4 = bind(cfg, w, max_ctx=T, pending_depth=4)
    m1 = bind(cfg, w, max_ctx=T, fence=(0, cfg.n_layers))
    lg4, lg1 = m4.prefill(toks[:P]), m1.prefill(toks[:P])
    assert np.array_equal(lg4, lg1)
    for l in (0, 7, 8, 31):
        for a, b in zip(m4.kv_export(l, 0), m1.kv_export(l, 0)):
            assert np.array_equal(a, b), l
    pend, dec4 = [], []
    for t in range(P, T):
        pend.append(m4.decode_step_deferred(toks[t], t))
        if len(pend) == 4 or t == T - 1:
            for p in pend:
                dec4.append(p.wait())
                p.free()
            pend = []
    dec4 = np.stack(dec4)
    dec1 = np.stack([m1.decode_step(toks[t], t) for t in range(P, T)])
    assert np.array_equal(dec4, dec1)


@pytest.fixture(scope="module")
def tiny_q8():
    w = synth.make_weights(TINY_Q8)
    T = 80
    toks = synth.make_tokens(TINY_Q8, T)
    orc = oracle.Oracle(TINY_Q8, w, max_ctx=T)
    ref = np.stack([orc.step(toks[t], t) for t in range(T)])
    orc.close()
    return w, toks, ref


def test_tiny_q8_prefill_every_position_and_plans(tiny_q8):
    """int8 row-scale weights (widened to bf16 in shared memory, the row scale
    on the accumulator): every prompt position against the oracle at the int8
    tolerance, decode after the prefill, and bit-identity across stage plans."""
    w, toks, ref = tiny_q8
    m = bind(TINY_Q8, w, max_ctx=80)
    pos, i = 0, 0
    lens = (3, 16, 1, 21, 7, 16)
    while pos < 64:
        n = min(lens[i % len(lens)], 64 - pos)
        assert_close(m.prefill(toks[pos:pos + n], pos0=pos, chunk=16), ref[pos + n - 1], TINY_Q8,
                     f"int8 prefill ending at position {pos + n - 1}")
        pos += n
        i += 1
    for t in range(64, 80):
        assert_close(m.decode_step(toks[t], t), ref[t], TINY_Q8, f"int8 decode step {t} after prefill")
    base = _prefill_run(TINY_Q8, w, toks, 64, 8, fence=(0, 4))
    for fence in ((0, 2, 4), (0, 1, 2, 3, 4)):
        got = _prefill_run(TINY_Q8, w, toks, 64, 8, fence=fence)
        assert np.array_equal(got[0], base[0]), fence
        for (kg, vg), (kb, vb) in zip(got[1], base[1]):
            assert np.array_equal(kg, kb) and np.array_equal(vg, vb), fence
        assert np.array_equal(got[2], base[2]), fence


def test_8b_q8_prefill_over_oracle_cache():
    """The 8B shape with int8 weights (2 stages, cut 16): one-token prefills over
    the oracle's own cache rows against the oracle's steps, and a 256-token
    prefill on 2 stages bit-identical to 1 stage."""
    cfg = synth.CONFIGS["8b_q8"]
    P = 128
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, P)
    orc = oracle.Oracle(cfg, w, max_ctx=P)
    ref = np.stack([orc.step(toks[t], t) for t in range(P)])
    kv = [orc.kv_export(l, 0) for l in range(cfg.n_layers)]
    orc.close()
    m = bind(cfg, w, max_ctx=P)
    for t in (0, 5, 64, P - 1):
        for l in range(cfg.n_layers):
            m.kv_import(l, 0, kv[l][0], kv[l][1], t)
        assert_close(m.prefill(toks[t:t + 1], pos0=t), ref[t], cfg, f"8B int8 one-token prefill at {t}")
    m.close()
    lg2 = _prefill_run(cfg, w, toks, P, 0, chunk=0)
    lg1 = _prefill_run(cfg, w, toks, P, 0, fence=(0, cfg.n_layers), chunk=0)
    assert np.array_equal(lg2[0], lg1[0])
    for (kg, vg), (kb, vb) in zip(lg2[1], lg1[1]):
        assert np.array_equal(kg, kb) and np.array_equal(vg, vb)


def test_prefill_argument_checks(tiny):
    w, toks, _, _ = tiny
    m = bind(TINY, w, max_ctx=80)
    bad = [
        dict(tokens=toks[:4], pos0=1),                      # skips row 0
        dict(tokens=toks[:4], pos0=78),                     # past max_ctx
        dict(tokens=toks[:4], pos0=0, chunk=129),           # chunk too large
        dict(tokens=np.array([0, TINY.vocab], np.int32)),   # token out of range
        dict(tokens=np.zeros(0, np.int32)),                 # empty
        dict(tokens=toks[:4], b=1),                         # no such sequence
    ]
    for kw in bad:
        with pytest.raises(lps.LpsError) as ei:
            m.prefill(**kw)
        assert ei.value.code == lps.LPS_EINVAL, kw
    m.prefill(toks[:4])  # the model is still usable
    vm = bind(TINY.replace(name="tiny_v2", batch=2), w, max_ctx=16, flags=lps.LPS_FLAG_VERIFY)
    with pytest.raises(lps.LpsError) as ei:
        vm.prefill(toks[:4])
    assert ei.value.code == lps.LPS_EINVAL and "verify" in str(ei.value)
    b2 = TINY.replace(name="tiny_b2", batch=2)
    mb = bind(b2, synth.make_weights(b2), max_ctx=16)
    with pytest.raises(lps.LpsError) as ei:
        mb.prefill(toks[:4])
    assert ei.value.code == lps.LPS_EINVAL and "row-major" in str(ei.value)


def test_prefill_interleaved_with_deferred_steps(tiny):
    """Prefill calls enqueued while deferred decode steps are still in flight
    (stream order keeps them apart): a prompt prefilled, deferred steps, a second
    prompt segment appended by prefill, more deferred steps -- the same bits at
    every position as the same schedule run eagerly on another model."""
    w, toks, _, _ = tiny
    seq = [("p", 0, 24), ("d", 24, 6), ("p", 30, 20), ("d", 50, 10)]

    def run(deferred):
        m = bind(TINY, w, max_ctx=80, pending_depth=4)
        out, pend = {}, []
        for kind, p0, n in seq:
            if kind == "p":
                out[p0 + n - 1] = m.prefill(toks[p0:p0 + n], pos0=p0, chunk=16)
                continue
            for t in range(p0, p0 + n):
                if not deferred:
                    out[t] = m.decode_step(toks[t], t)
                    continue
                pend.append((t, m.decode_step_deferred(toks[t], t)))
                if len(pend) == 4:
                    tp, p = pend.pop(0)
                    out[tp] = p.wait()
                    p.free()
        for tp, p in pend:
            out[tp] = p.wait()
            p.free()
        m.close()
        return out

    eager, deferred = run(False), run(True)
    assert sorted(eager) == sorted(deferred)
    for t in eager:
        assert np.array_equal(eager[t], deferred[t]), t


MID = synth.ModelConfig("mid_prefill", 93, 3, 512, 32, 8, 128, 512, 1000, "bf16", 1, 0, 0, (1, 2))


@pytest.mark.parametrize("chunk", [16, 0])
def test_prefill_after_long_imported_context(chunk):
    """Cache rows [0, 5000) imported into both sides, then 40 prompt tokens
    prefilled in calls of 17, 1 and 22 tokens: the chunk attention runs over
    many key chunks per 16-token block, with the causal mask inside the chunk;
    each call's last logits against the oracle's step at that position, and
    the cache rows the prefill wrote against the oracle's."""
    cfg, P = MID, 5000
    w = synth.make_weights(cfg)
    max_ctx = P + 40
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    m = bind(cfg, w, max_ctx=max_ctx)
    for (l, b), (k, v) in random_kv(cfg, 19, cfg.n_layers, max_ctx, P).items():
        m.kv_import(l, b, k, v, P)
        orc.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(cfg, 40, seed=61)[:, 0]
    ref = [orc.step(toks[j:j + 1], P + j)[0] for j in range(40)]
    pos = 0
    for n in (17, 1, 22):
        got = m.prefill(toks[pos:pos + n], pos0=P + pos, chunk=chunk)
        assert_close(got, ref[pos + n - 1], cfg, f"prefill ending at {P + pos + n - 1}")
        pos += n
    for l in range(cfg.n_layers):
        for a, b in zip(m.kv_export(l, 0), orc.kv_export(l, 0)):
            assert np.array_equal(a[:, :P], b[:, :P])
            rg = synth.bf16_to_f32(a[:, P:P + 40]).astype(np.float64)
            ro = synth.bf16_to_f32(b[:, P:P + 40]).astype(np.float64)
            scale = np.max(np.abs(ro), axis=2, keepdims=True)
            assert np.all(np.abs(rg - ro) <= np.abs(ro) * 2 ** -6 + 1e-3 * scale), f"layer {l}"


G8 = synth.ModelConfig("g8_prefill", 88, 2, 512, 16, 2, 64, 512, 1000, "bf16", 1, 0, 0, (1,))
G1 = synth.ModelConfig("g1_prefill", 89, 2, 512, 4, 4, 128, 512, 1000, "bf16", 1, 0, 0, (1,))


@pytest.mark.parametrize("cfg", [G8, G1], ids=lambda c: c.name)
def test_prefill_group_sizes(cfg):
    """The chunk attention at the GQA extremes: eight q heads per kv head (one
    16-token group per CTA, eight warps) and one (eight 16-token groups per
    CTA), after 700 imported cache rows; each call's last logits against the
    oracle, and two stage plans bit-identical."""
    P = 700
    w = synth.make_weights(cfg)
    max_ctx = P + 40
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    kv = random_kv(cfg, 23, cfg.n_layers, max_ctx, P)
    toks = synth.make_tokens(cfg, 40, seed=62)[:, 0]
    for (l, b), (k, v) in kv.items():
        orc.kv_import(l, b, k, v, P)
    ref = [orc.step(toks[j:j + 1], P + j)[0] for j in range(40)]
    outs = []
    for fence in ((0, 1, 2), (0, 2)):
        m = bind(cfg, w, fence=fence, max_ctx=max_ctx)
        for (l, b), (k, v) in kv.items():
            m.kv_import(l, b, k, v, P)
        got, pos = [], 0
        for n in (17, 1, 22):
            lg = m.prefill(toks[pos:pos + n], pos0=P + pos, chunk=0)
            assert_close(lg, ref[pos + n - 1], cfg, f"{cfg.name} prefill ending at {P + pos + n - 1}")
            got.append(lg)
            pos += n
        outs.append(got)
        m.close()
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
