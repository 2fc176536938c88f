"""Speculative-verify rows through the stages (LPS_FLAG_VERIFY): the batch's M
rows are M consecutive positions of one sequence with one cache (memra_engine::pp,
spec_pp_on: the verify forward takes the stage split). The oracle runs the same
tokens as ordinary one-row decode steps; every verify row must give that
position's logits, and the cache rows the step writes must be the ones M
single steps write.
"""
import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from workloads import TOL_BF16, assert_close, bind, rel_err, random_kv

pytestmark = pytest.mark.gpu

# one sequence; the verify model binds it with batch = M rows
MID = synth.ModelConfig("mid_verify", 93, 3, 512, 32, 8, 128, 512, 1000, "bf16", 1, 0, 0, (1, 2))
MID_Q8 = MID.replace(name="mid_verify_q8", index=94, weight_dtype="int8")


def _verify_model(cfg, w, M, max_ctx, fence=None):
    return bind(cfg.replace(batch=M), w, fence=fence, max_ctx=max_ctx, flags=lps.LPS_FLAG_VERIFY)


@pytest.mark.parametrize("cfg", [MID, MID_Q8], ids=lambda c: c.name)
@pytest.mark.parametrize("M", [2, 4, 8])
def test_verify_rows_match_single_steps(cfg, M):
    """Fill the sequence M tokens per verify step from position 0 (the rows of a
    step attend to the rows before them in the same step); compare every row
    with the oracle's one-row decode step at that position."""
    w = synth.make_weights(cfg)
    steps = 3
    T = M * steps
    max_ctx = T + 1
    toks = synth.make_tokens(cfg, T, seed=55)[:, 0]
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    ref = np.stack([orc.step(toks[t:t + 1], t)[0] for t in range(T)])
    m = _verify_model(cfg, w, M, max_ctx)
    for s in range(steps):
        got = m.decode_step(toks[s * M:(s + 1) * M], s * M)
        assert_close(got, ref[s * M:(s + 1) * M], cfg, f"M={M} step {s}")


def test_verify_after_long_context_and_cache_rows():
    """Rows [0, P) imported into both sides; a verify step at P..P+M-1 attends
    over several chunks per kv head, and writes the M cache rows an oracle
    running M single steps writes (the KV-row criterion of the one-row tests)."""
    cfg, M, P = MID, 4, 2500
    w = synth.make_weights(cfg)
    max_ctx = P + M + 1
    orc = oracle.Oracle(cfg, w, max_ctx=max_ctx)
    m = _verify_model(cfg, w, M, max_ctx)
    for (l, b), (k, v) in random_kv(cfg, 17, cfg.n_layers, max_ctx, P).items():
        m.kv_import(l, b, k, v, P)
        orc.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(cfg, M, seed=56)[:, 0]
    ref = np.stack([orc.step(toks[j:j + 1], P + j)[0] for j in range(M)])
    got = m.decode_step(toks, P)
    assert_close(got, ref, cfg, "verify at P")
    for l in range(cfg.n_layers):
        gk, gv = m.kv_export(l, 0)
        ok, ov = orc.kv_export(l, 0)
        for a, b in ((gk, ok), (gv, ov)):
            assert np.array_equal(a[:, :P], b[:, :P])
            # new rows: the same values up to one bf16 rounding of slightly different sums; entries
            # near zero carry the sums' absolute error (cancellation), hence the row-scaled term
            rg = synth.bf16_to_f32(a[:, P:P + M]).astype(np.float64)
            ro = synth.bf16_to_f32(b[:, P:P + M]).astype(np.float64)
            scale = np.max(np.abs(ro), axis=2, keepdims=True)
            assert np.all(np.abs(rg - ro) <= np.abs(ro) * 2 ** -7 + 1e-4 * scale), f"layer {l}"
            assert np.mean(rg == ro) > 0.95


def test_verify_stage_plans_bit_identical():
    cfg, M = MID, 4
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, 2 * M, seed=57)[:, 0]
    outs = []
    for fence in ((0, 3), (0, 1, 3), (0, 1, 2, 3)):
        m = _verify_model(cfg, w, M, 2 * M + 1, fence=fence)
        outs.append([m.decode_step(toks[s * M:(s + 1) * M], s * M) for s in range(2)])
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)


def test_verify_matches_library_single_steps():
    """The same tokens through the library's own one-row path (the batch-1 GEMV
    kernels) and through verify rows (the tensor-core skinny GEMM)."""
    cfg, M = MID, 4
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, 2 * M, seed=58)[:, 0]
    one = bind(cfg, w, max_ctx=2 * M + 1)
    ref = np.stack([one.decode_step(toks[t:t + 1], t)[0] for t in range(2 * M)])
    m = _verify_model(cfg, w, M, 2 * M + 1)
    got = np.concatenate([m.decode_step(toks[s * M:(s + 1) * M], s * M) for s in range(2)])
    assert np.all(rel_err(got, ref) <= TOL_BF16)


def test_verify_refuses_non_consecutive_rows():
    cfg, M = MID, 4
    w = synth.make_weights(cfg)
    m = _verify_model(cfg, w, M, 16)
    toks = np.zeros(M, np.int32)
    with pytest.raises(lps.LpsError):
        m.decode_step(toks, [0, 1, 3, 4])  # not consecutive
    with pytest.raises(lps.LpsError):
        m.decode_step(toks, 1)  # starts past the filled rows
    with pytest.raises(lps.LpsError):
        m.decode_step(toks, 13)  # the last row would be at max_ctx
    m.decode_step(toks, 0)
    m.decode_step(toks, 4)  # continues right after the rows written
    with pytest.raises(lps.LpsError):
        m.kv_export(0, 1)  # one sequence
