"""The seeded workload generator: deterministic, order free, right moments."""
import numpy as np

import synth


def test_counter_based_and_order_free():
    a = synth.normal_bf16(1, 7, (1000,))
    b = synth.normal_bf16(1, 7, (3000,))[:1000]  # a prefix of a longer draw is the same draw
    assert np.array_equal(a, b)
    synth.lib().synth_set_threads(1)
    try:
        c = synth.normal_bf16(1, 7, (200_000,))
    finally:
        synth.lib().synth_set_threads(0)
    assert np.array_equal(c, synth.normal_bf16(1, 7, (200_000,)))
    assert not np.array_equal(a, synth.normal_bf16(1, 8, (1000,)))
    assert not np.array_equal(a, synth.normal_bf16(2, 7, (1000,)))


def test_normal_moments():
    x = synth.bf16_to_f32(synth.normal_bf16(3, 1, (400_000,))).astype(np.float64)
    assert abs(x.mean()) < 2e-4 and abs(x.std() - 0.02) < 2e-4
    z = x / 0.02
    assert abs(np.mean(z ** 4) - 3.0) < 0.05  # Gaussian kurtosis


def test_q8_rows_roundtrip():
    q, s = synth.normal_q8_rows(4, 2, 64, 300)
    w = synth.normal_f32(4, 2, (64, 300))
    assert np.array_equal(np.abs(q).max(axis=1), np.full(64, 127))
    err = np.abs(w.astype(np.float64) - q.astype(np.float64) * s[:, None])
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))


def test_tokens_uniform_range():
    t = synth.tokens(5, 0, 4096, 100_000)
    assert t.min() >= 0 and t.max() < 4096
    counts = np.bincount(t, minlength=4096)
    assert counts.min() > 0 and abs(counts.mean() - 100_000 / 4096) < 1e-9


def test_padded_weights_share_real_weights():
    cfg = synth.CONFIGS["padded"].replace(n_layers=1, n_embd=64, ffn=32, vocab=16, head_dim=8)
    base = synth.make_weights(cfg.base())
    pad = synth.make_weights(cfg)
    hd = cfg.head_dim
    for k in ("wq", "wk", "wv"):
        n = base["layers"][0][k].shape[0]
        assert np.array_equal(pad["layers"][0][k][:n], base["layers"][0][k])
        assert not pad["layers"][0][k][n:].any()
    assert pad["layers"][0]["wq"].shape[0] == 48 * hd and pad["layers"][0]["wk"].shape[0] == 12 * hd
    wo = pad["layers"][0]["wo"]
    assert np.array_equal(wo[:, :32 * hd], base["layers"][0]["wo"]) and not wo[:, 32 * hd:].any()


def test_step_bytes_match_hand_count():
    c = synth.CONFIGS["8b"]
    # 32 layers x (6144 + 4096 + 2 * 14336 + 4096 rows x 4096 ... ) bf16, plus head, norms, one embed row
    per_layer = (6144 * 4096 + 4096 * 4096 + 2 * 14336 * 4096 + 4096 * 14336) * 2 + 2 * 4096 * 4
    assert c.weight_bytes() == 32 * per_layer + 128256 * 4096 * 2 + 4096 * 4 + 4096 * 2
    assert abs(c.weight_bytes() / 1e9 - 15.009) < 0.01
    assert c.kv_bytes(8191) == 32 * 2 * 8 * 128 * 2 * 8193
