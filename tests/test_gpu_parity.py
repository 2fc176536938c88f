"""GPU path (through the C ABI) against the CPU oracle on seeded inputs.

Bit-exact between GPU arms (stage plans, eager vs deferred readback, the
single-stream seam, replays); within the stated tolerance against the oracle
(max-abs error <= 2e-3 x max|logit| for bf16 weights, 5e-3 for int8), at every
teacher-forced position.
"""
import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from workloads import assert_close, bind, random_kv

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["tiny"]
# small shapes that reach the multi-chunk, multi-sub-tile attention paths
MID = synth.ModelConfig("mid", 95, 2, 512, 32, 8, 128, 512, 1000, "bf16", 1, 0, 0, (1,))
MID64 = synth.ModelConfig("mid64", 96, 2, 256, 16, 4, 64, 352, 500, "bf16", 2, 0, 0, (1,))
MID_Q8 = MID.replace(name="mid_q8", index=97, weight_dtype="int8")
# the 8B-shape layer (n_embd 4096, 32/8 heads of 128, ffn 14336) with a 50k vocabulary: every GEMV
# streams many ring buffers per CTA, as at full size
WIDE = synth.ModelConfig("wide", 98, 2, 4096, 32, 8, 128, 14336, 50000, "bf16", 1, 0, 0, (1,))
WIDE_Q8 = WIDE.replace(name="wide_q8", index=99, weight_dtype="int8")


@pytest.mark.parametrize("cfg", [WIDE, WIDE_Q8], ids=lambda c: c.name)
def test_full_width_layers_match_oracle(cfg):
    """Both batch-1 paths at the 8B layer width, against the oracle."""
    w = synth.make_weights(cfg)
    T = 6
    toks = synth.make_tokens(cfg, T)
    orc = oracle.Oracle(cfg, w, max_ctx=T)
    ref = [orc.step(toks[t], t) for t in range(T)]
    for flags in (0, lps.LPS_FLAG_PERSISTENT):
        m = bind(cfg, w, max_ctx=T, flags=flags)
        assert m.stats()["persistent"] == (flags != 0)
        for t in range(T):
            assert_close(m.decode_step(toks[t], t), ref[t], cfg, f"step {t} (flags {flags})")
        m.close()


@pytest.fixture(scope="module")
def tiny():
    w = synth.make_weights(TINY)
    T = TINY.max_ctx
    toks = synth.make_tokens(TINY, T)
    orc = oracle.Oracle(TINY, w, max_ctx=T)
    ref = np.stack([orc.step(toks[t], t) for t in range(T)])
    return w, toks, ref, orc


def run_eager(m, toks, start=0):
    return np.stack([m.decode_step(toks[t], start + t) for t in range(len(toks))])


# the two batch-1 paths: the chained per-projection kernels (default) and the persistent stage kernel
ARMS = {"chained": 0, "persistent": lps.LPS_FLAG_PERSISTENT}


@pytest.mark.parametrize("arm", ARMS)
def test_tiny_matches_oracle_every_position(tiny, arm):
    w, toks, ref, _ = tiny
    m = bind(TINY, w, flags=ARMS[arm])
    got = run_eager(m, toks)
    assert_close(got, ref, TINY, f"tiny N=2 ({arm})")
    st = m.stats()
    assert st["persistent"] == (arm == "persistent")
    assert st["stage_walks"] == 2 * len(toks) and st["boundary_crossings"] == len(toks)
    assert st["fence"] == (0, 2, 4)
    assert st["kernel_launches"] == len(toks) * (2 if arm == "persistent" else 2 + 5 * TINY.n_layers)


@pytest.mark.parametrize("arm", ARMS)
def test_tiny_stage_plans_bit_identical(tiny, arm):
    w, toks, _, _ = tiny
    base = run_eager(bind(TINY, w, fence=(0, 4), flags=ARMS[arm]), toks)
    for fence in ((0, 2, 4), (0, 1, 2, 3, 4), (0, 3, 4), (0, 1, 4)):
        m = bind(TINY, w, fence=fence, flags=ARMS[arm])
        assert np.array_equal(run_eager(m, toks), base), fence
        assert m.stats()["boundary_crossings"] == (len(fence) - 2) * len(toks)
    if arm == "chained":
        # the single-stream seam (two plain copies per boundary) runs the chained kernels
        single = bind(TINY, w, fence=(0, 1, 3, 4), flags=lps.LPS_FLAG_SINGLE_STREAM)
        assert not single.stats()["persistent"]
        assert np.array_equal(run_eager(single, toks), base)


def test_tiny_deferred_pipelined_bit_identical(tiny):
    w, toks, ref, _ = tiny
    eager = run_eager(bind(TINY, w), toks)
    m = bind(TINY, w, pending_depth=4)
    pend, got = [], []
    for t in range(len(toks)):
        pend.append(m.decode_step_deferred(toks[t], t))
        if len(pend) == 4:
            p = pend.pop(0)
            got.append(p.wait())
            p.free()
    for p in pend:
        got.append(p.wait())
        p.free()
    assert np.array_equal(np.stack(got), eager)
    st = m.stats()
    assert st["deferred_steps"] == len(toks) and st["pending_drains"] == len(toks)


def test_tiny_random_gains():
    w = synth.make_weights(TINY, random_gains=True)
    T = 20
    toks = synth.make_tokens(TINY, T)
    orc = oracle.Oracle(TINY, w, max_ctx=T)
    m = bind(TINY, w, max_ctx=T)
    for t in range(T):
        assert_close(m.decode_step(toks[t], t), orc.step(toks[t], t), TINY, f"step {t}")


def test_kv_rows_match_oracle_and_plans(tiny):
    w, toks, _, orc = tiny
    T = len(toks)
    m2, m1 = bind(TINY, w), bind(TINY, w, fence=(0, 4))
    run_eager(m2, toks)
    run_eager(m1, toks)
    for l in range(TINY.n_layers):
        k2, v2 = m2.kv_export(l, 0)
        k1, v1 = m1.kv_export(l, 0)
        assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
        ko, vo = orc.kv_export(l, 0)
        for g, o in ((k2, ko), (v2, vo)):
            assert not g[:, T:].any()
            a = synth.bf16_to_f32(g[:, :T]).astype(np.float64)
            b = synth.bf16_to_f32(o[:, :T]).astype(np.float64)
            # rows hold the same values up to one bf16 rounding of slightly different fp32/fp64 sums;
            # near-zero entries carry the sums' absolute error (cancellation), hence the scaled term
            scale = np.max(np.abs(b), axis=2, keepdims=True)
            assert np.all(np.abs(a - b) <= np.abs(b) * 2 ** -7 + 1e-4 * scale)
            assert np.mean(a == b) > 0.95


def test_kv_import_export_roundtrip():
    w = synth.make_weights(MID64)
    m = bind(MID64, w, max_ctx=300)
    kv = random_kv(MID64, 5, MID64.n_layers, 300, 257)
    for (l, b), (k, v) in kv.items():
        m.kv_import(l, b, k, v, 257)
    for (l, b), (k, v) in kv.items():
        k2, v2 = m.kv_export(l, b)
        assert np.array_equal(k, k2) and np.array_equal(v, v2)


def test_rewind_rewrites_the_same_row(tiny):
    w, toks, _, _ = tiny
    m = bind(TINY, w)
    run_eager(m, toks[:30])
    before = [m.kv_export(l, 0) for l in range(TINY.n_layers)]
    alt = (toks[20] + 1) % TINY.vocab
    got = m.decode_step(alt, 20)
    fresh = bind(TINY, w)
    run_eager(fresh, toks[:20])
    assert np.array_equal(got, fresh.decode_step(alt, 20))
    for l in range(TINY.n_layers):
        k, v = m.kv_export(l, 0)
        assert np.array_equal(k[:, :20], before[l][0][:, :20])
        assert not np.array_equal(k[:, 20], before[l][0][:, 20])
        assert np.array_equal(k[:, 21:30], before[l][0][:, 21:30])  # stale rows stay; only [0, pos] is read


@pytest.mark.parametrize("cfg", [MID, MID64, MID_Q8], ids=lambda c: c.name)
@pytest.mark.parametrize("P", [0, 63, 64, 65, 127, 129, 2431, 2433, 5001])
def test_attention_long_context_synthetic_cache(cfg, P):
    """Cache rows [0, P) imported into both sides; the next steps attend over
    P+1.. rows: ragged sub-tiles, several chunks, several sub-tiles per chunk."""
    w = synth.make_weights(cfg)
    max_ctx = P + 3
    m = bind(cfg, w, max_ctx=max_ctx)
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    if P:
        for (l, b), (k, v) in random_kv(cfg, 11 + P, cfg.n_layers, max_ctx, P).items():
            m.kv_import(l, b, k, v, P)
            orc.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(cfg, 3, seed=77)
    for t in range(3):
        assert_close(m.decode_step(toks[t], P + t), orc.step(toks[t], P + t), cfg, f"P={P} step {t}")


@pytest.mark.parametrize("cfg", [MID, MID64], ids=lambda c: c.name)
def test_attention_very_long_context_combine(cfg):
    """40k cached rows: hundreds of chunks per (sequence, kv head), so the last
    CTA merges the partials in several staged pieces."""
    P = 40000
    w = synth.make_weights(cfg)
    max_ctx = P + 2
    m = bind(cfg, w, max_ctx=max_ctx)
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    for (l, b), (k, v) in random_kv(cfg, 123, cfg.n_layers, max_ctx, P).items():
        m.kv_import(l, b, k, v, P)
        orc.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(cfg, 2, seed=78)
    for t in range(2):
        assert_close(m.decode_step(toks[t], P + t), orc.step(toks[t], P + t), cfg, f"step {t}")


def test_refusals_leave_state_unchanged(tiny):
    w, toks, ref, _ = tiny
    m = bind(TINY, w)
    run_eager(m, toks[:5])
    for tok, pos, what in ((TINY.vocab, 5, "token"), (-1, 5, "token"), (toks[5], 7, "skips"),
                           (toks[5], TINY.max_ctx, "max_ctx")):
        with pytest.raises(lps.LpsError) as e:
            m.decode_step(tok, pos)
        assert e.value.code == lps.LPS_EINVAL and "decode_step" in str(e.value) and what in str(e.value)
    got = run_eager(m, toks[5:10], start=5)
    assert np.array_equal(got, run_eager(bind(TINY, w), toks[:10])[5:])


def test_pending_ring_busy_and_free_without_wait(tiny):
    w, toks, _, _ = tiny
    m = bind(TINY, w, pending_depth=2)
    a = m.decode_step_deferred(toks[0], 0)
    b = m.decode_step_deferred(toks[1], 1)
    with pytest.raises(lps.LpsError) as e:
        m.decode_step_deferred(toks[2], 2)
    assert e.value.code == lps.LPS_EBUSY
    a.free()  # dropped without waiting
    c = m.decode_step_deferred(toks[2], 2)
    eager = run_eager(bind(TINY, w), toks[:3])
    assert np.array_equal(b.wait(), eager[1]) and np.array_equal(c.wait(), eager[2])
    assert np.array_equal(c.wait(), eager[2])  # waiting twice is allowed
    b.free()
    c.free()


def test_device_resident_step(tiny):
    import torch
    w, toks, _, _ = tiny
    m = bind(TINY, w)
    eager = run_eager(bind(TINY, w), toks[:6])
    tok_dev = torch.tensor(toks[:6, 0], dtype=torch.int32, device="cuda")
    out = torch.empty((6, TINY.vocab), dtype=torch.float32, device="cuda")
    for t in range(6):
        m.decode_step_device(tok_dev[t:t + 1].data_ptr(), t, out[t].data_ptr())
    m.synchronize()
    assert np.array_equal(out.cpu().numpy(), eager[:, 0])


def test_soak_deferred_replays_bit_identical():
    """20 replays of a pipelined deferred run (teacher forced, rewound to 0):
    every step of every replay equals the eager run bit for bit."""
    cfg = MID64
    w = synth.make_weights(cfg)
    T = 48
    toks = synth.make_tokens(cfg, T)
    eager = run_eager(bind(cfg, w, max_ctx=T, fence=(0, 1, 2)), toks)
    m = bind(cfg, w, max_ctx=T, fence=(0, 1, 2), pending_depth=4)
    for rep in range(20):
        pend, got = [], []
        for t in range(T):
            pend.append(m.decode_step_deferred(toks[t], t))
            if len(pend) == 4:
                p = pend.pop(0)
                got.append(p.wait())
                p.free()
        for p in pend:
            got.append(p.wait())
            p.free()
        assert np.array_equal(np.stack(got), eager), f"replay {rep}"


@pytest.mark.parametrize("flags", [0, lps.LPS_FLAG_SERIAL_STEPS], ids=["overlap", "serial"])
def test_soak_full_width_deferred(flags):
    """Many pipelined deferred steps at full layer width (four stages, ring
    wrap-around in every GEMV), stages of consecutive steps overlapping or
    not: no device-side error, every step equal to the eager run."""
    cfg = WIDE.replace(n_layers=4, cuts=(1, 2, 3))
    w = synth.make_weights(cfg)
    T = 96
    toks = synth.make_tokens(cfg, T)
    eager = run_eager(bind(cfg, w, max_ctx=T), toks)
    m = bind(cfg, w, max_ctx=T, pending_depth=4, flags=flags)
    pend, got = [], []
    for t in range(T):
        pend.append(m.decode_step_deferred(toks[t], t))
        if len(pend) == 4:
            p = pend.pop(0)
            got.append(p.wait())
            p.free()
    for p in pend:
        got.append(p.wait())
        p.free()
    m.synchronize()
    assert np.array_equal(np.stack(got), eager)
