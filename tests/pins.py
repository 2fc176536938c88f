"""Pins for the oracle: each checks it against something other than itself.

Every pin is a function ``pin_*(lib)`` that raises AssertionError on failure;
``lib`` selects a build of the oracle library (None = the committed source).
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
plants mistakes in copies of the oracle and checks that some pin fails.

What pins what:
- the whole decoder: a second implementation in matrix form over all
  positions, with no cache and a causal mask (numpy, fp64), RoPE done with
  complex numbers and bf16 rounding done on the fp64 bit pattern;
- building blocks: torch's CPU library routines in fp64 (rms_norm,
  scaled_dot_product_attention), numpy matmul, closed forms (RoPE at pos 0 and
  at pos 1 with head_dim 4, RMSNorm of a constant vector, softmax of q = 0,
  attention at pos 0);
- structure: N-stage equals 1-stage bit for bit; zero-padded dummy heads give
  exactly zero attention outputs and leave logits bit for bit unchanged (the
  numerical chain of "TP3 support via zero-padded dummy heads", Weight-padding
  design: zero q/k -> zero scores -> uniform softmax over zero V -> 0).
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

# ---------------------------------------------------------------------------
# small workloads
# ---------------------------------------------------------------------------

MICRO = synth.ModelConfig("micro", 90, 3, 64, 4, 2, 16, 96, 160, "bf16", 2, 12, 0, (1,))
MICRO_Q8 = MICRO.replace(name="micro_q8", index=91, weight_dtype="int8")


def _weights(cfg, random_gains=True):
    return synth.make_weights(cfg, random_gains=random_gains)


def _deq(m) -> np.ndarray:
    if isinstance(m, tuple):
        q, s = m
        return q.astype(np.float64) * s.astype(np.float64)[:, None]
    return synth.bf16_to_f32(m).astype(np.float64)


def _bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even) by integer rounding of the fp64
    bit pattern: keep sign, exponent and the top 7 of 52 fraction bits."""
    u = np.ascontiguousarray(x, np.float64).view(np.uint64)
    drop = np.uint64(45)
    lsb = (u >> drop) & np.uint64(1)
    u = (u + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb) & ~((np.uint64(1) << drop) - np.uint64(1))
    return u.view(np.float64)


def _rope_complex(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """x [..., T, hd]: pair (i, i + hd/2) as the complex number x_i + j x_{i+hd/2},
    turned by exp(j * pos * theta^(-2i/hd))."""
    hd = x.shape[-1]
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = theta ** (-2.0 * np.arange(half) / hd)
    z = z * np.exp(1j * pos[:, None] * freq[None, :])
    return np.concatenate([z.real, z.imag], axis=-1)


def _rms_rows(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    h = h.astype(np.float64)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * g.astype(np.float64)


def brute_force_sequence(cfg, w, toks: np.ndarray, return_kv: bool = False):
    """Logits [T, V] of one sequence for tokens at positions 0..T-1, computed
    layer by layer over all positions at once with a causal mask and no cache."""
    T = len(toks)
    hd, nq, nkv = cfg.head_dim, cfg.q_heads, cfg.kv_heads
    G = nq // nkv
    pos = np.arange(T, dtype=np.float64)
    h = _deq(w["embed"])[toks].astype(np.float32)
    kv = []
    for lw in w["layers"]:
        xn = _rms_rows(h, lw["attn_norm"], cfg.rms_eps)
        Q = (xn @ _deq(lw["wq"]).T).reshape(T, nq, hd).transpose(1, 0, 2)
        K = (xn @ _deq(lw["wk"]).T).reshape(T, nkv, hd).transpose(1, 0, 2)
        V = (xn @ _deq(lw["wv"]).T).reshape(T, nkv, hd).transpose(1, 0, 2)
        Q = _rope_complex(Q, pos, cfg.rope_theta)
        K = _bf16_round_bits(_rope_complex(K, pos, cfg.rope_theta))
        V = _bf16_round_bits(V)
        kv.append((K, V))
        mask = np.triu(np.ones((T, T), bool), 1)
        O = np.empty((nq, T, hd))
        for hh in range(nq):
            S = Q[hh] @ K[hh // G].T / np.sqrt(hd)
            S[mask] = -np.inf
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            O[hh] = P @ V[hh // G]
        O = O.transpose(1, 0, 2).reshape(T, nq * hd)
        h = (h.astype(np.float64) + O @ _deq(lw["wo"]).T).astype(np.float32)
        xn = _rms_rows(h, lw["ffn_norm"], cfg.rms_eps)
        a = xn @ _deq(lw["w_gate"]).T
        a = a / (1.0 + np.exp(-a)) * (xn @ _deq(lw["w_up"]).T)
        h = (h.astype(np.float64) + a @ _deq(lw["w_down"]).T).astype(np.float32)
    logits = _rms_rows(h, w["out_norm"], cfg.rms_eps) @ _deq(w["lm_head"]).T
    return (logits, kv) if return_kv else logits


def run_oracle(cfg, w, toks: np.ndarray, fence=None, lib=None):
    """Teacher-forced steps at positions 0..T-1; toks [T, B] -> logits [T, B, V]."""
    orc = oracle.Oracle(cfg, w, fence=fence, max_ctx=toks.shape[0], lib=lib)
    out = np.stack([orc.step(toks[t], t) for t in range(toks.shape[0])])
    return out, orc


def _rel(a, b):
    return float(np.max(np.abs(a.astype(np.float64) - b.astype(np.float64))) / np.max(np.abs(b)))


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_decoder_matches_brute_force(lib=None):
    """Cached step-by-step decode == no-cache matrix form, bf16 and int8, B=2."""
    for cfg in (MICRO, MICRO_Q8):
        w = _weights(cfg)
        toks = synth.make_tokens(cfg, 12)
        got, orc = run_oracle(cfg, w, toks, lib=lib)
        for b in range(cfg.batch):
            ref, kv = brute_force_sequence(cfg, w, toks[:, b], return_kv=True)
            ref = ref.astype(np.float32)  # logits are returned as f32
            assert _rel(got[:, b], ref) < 1e-9, (cfg.name, b, _rel(got[:, b], ref))
            for l, (K, V) in enumerate(kv):  # cache rows == bf16(RoPE(k)) / bf16(v), per position
                k, v = orc.kv_export(l, b)
                kk = synth.bf16_to_f32(k[:, :12]).astype(np.float64)
                vv = synth.bf16_to_f32(v[:, :12]).astype(np.float64)
                assert np.mean(kk != K) < 1e-3 and np.mean(vv != V) < 1e-3
                assert np.allclose(kk, K, rtol=2 ** -7, atol=0) and np.allclose(vv, V, rtol=2 ** -7, atol=0)


def pin_sequences_independent(lib=None):
    """Sequence b's logits do not depend on the other sequences of the batch."""
    w = _weights(MICRO)
    toks = synth.make_tokens(MICRO, 8)
    got, _ = run_oracle(MICRO, w, toks, lib=lib)
    one = MICRO.replace(batch=1)
    solo, _ = run_oracle(one, w, toks[:, 1:2], lib=lib)
    assert np.array_equal(got[:, 1], solo[:, 0])


def pin_n_stage_equals_one_stage(lib=None):
    """The split changes scheduling, not math: every plan gives the same bits."""
    w = _weights(MICRO)
    toks = synth.make_tokens(MICRO, 6)
    ref, _ = run_oracle(MICRO, w, toks, fence=(0, 3), lib=lib)
    for fence in ((0, 1, 3), (0, 2, 3), (0, 1, 2, 3)):
        got, _ = run_oracle(MICRO, w, toks, fence=fence, lib=lib)
        assert np.array_equal(got, ref), fence


def pin_padded_heads_exact(lib=None):
    """Zero-padded dummy heads (GQA kept, appended at the end of each head axis):
    dummy attention outputs are exactly 0 and logits equal the unpadded model's."""
    base = MICRO.replace(index=92, n_q_heads=4, n_kv_heads=2)
    padded = base.replace(pad_q_heads=6, pad_kv_heads=3)
    wb = synth.make_weights(base, random_gains=True)
    wp = synth.make_weights(padded, random_gains=True)
    toks = synth.make_tokens(base, 6)
    ref, _ = run_oracle(base, wb, toks, lib=lib)
    got, orc = run_oracle(padded, wp, toks, lib=lib)
    assert np.array_equal(got, ref)
    for l in range(base.n_layers):
        for b in range(base.batch):
            o = orc.attn_out(l, b)
            assert np.all(o[4:] == 0.0), (l, b)
            assert np.all(np.abs(o[:4]).sum(axis=1) > 0)


def pin_zero_sublayers(lib=None):
    """With W_o = W_d = 0 every layer adds nothing: logits = W_head . rmsnorm(E[tok])."""
    for cfg in (MICRO, MICRO_Q8):
        w = _weights(cfg)
        for lw in w["layers"]:
            for key in ("wo", "w_down"):
                m = lw[key]
                lw[key] = (np.zeros_like(m[0]), m[1]) if isinstance(m, tuple) else np.zeros_like(m)
        toks = synth.make_tokens(cfg, 3)
        got, _ = run_oracle(cfg, w, toks, lib=lib)
        E, H = _deq(w["embed"]), _deq(w["lm_head"])
        for t in range(3):
            for b in range(cfg.batch):
                x = E[toks[t, b]].astype(np.float32).astype(np.float64)
                xn = x / np.sqrt(np.mean(x * x) + cfg.rms_eps) * w["out_norm"]
                assert _rel(got[t, b], (H @ xn).astype(np.float32)) < 1e-12


def pin_uniform_softmax_when_q_zero(lib=None):
    """W_q = 0 makes q = 0, scores 0 and the softmax uniform: the attention
    output of every head is the mean of its kv head's cached V rows."""
    w = _weights(MICRO)
    for lw in w["layers"]:
        lw["wq"] = np.zeros_like(lw["wq"])
    toks = synth.make_tokens(MICRO, 5)
    _, orc = run_oracle(MICRO, w, toks, lib=lib)
    G = MICRO.q_heads // MICRO.kv_heads
    for l in range(MICRO.n_layers):
        for b in range(MICRO.batch):
            _, v = orc.kv_export(l, b)
            o = orc.attn_out(l, b)
            for hh in range(MICRO.q_heads):
                mean = synth.bf16_to_f32(v[hh // G, :5]).astype(np.float64).mean(axis=0)
                assert np.allclose(o[hh], mean, rtol=1e-12, atol=1e-15)


def pin_rope_closed_forms(lib=None):
    """Rotate-half RoPE, angle pos * theta^(-2i/hd): identity at pos 0; at pos 1
    with hd 4 the pairs (0, 2) and (1, 3) turn by 1 and 10000^(-1/2) rad; norms
    of pairs kept; dot products depend only on the position difference."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(8)
    assert np.array_equal(oracle.rope(x, 0, lib=lib), x)
    got = oracle.rope(np.array([1.0, 2.0, 0.0, 0.0]), 1, lib=lib)
    want = np.array([np.cos(1.0), 2 * np.cos(0.01), np.sin(1.0), 2 * np.sin(0.01)])
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15)
    y = oracle.rope(x, 37, lib=lib)
    assert np.allclose(y[:4] ** 2 + y[4:] ** 2, x[:4] ** 2 + x[4:] ** 2, rtol=1e-12)
    k = rng.standard_normal(8)
    d1 = oracle.rope(x, 9, lib=lib) @ oracle.rope(k, 4, lib=lib)
    d2 = oracle.rope(x, 105, lib=lib) @ oracle.rope(k, 100, lib=lib)
    assert abs(d1 - d2) < 1e-12


def pin_rmsnorm_library(lib=None):
    """RMSNorm against torch's rms_norm in fp64, and the constant-vector closed form."""
    import torch
    rng = np.random.default_rng(6)
    h = rng.standard_normal(96).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(96)).astype(np.float32)
    got = oracle.rmsnorm(h, g, 1e-5, lib=lib)
    want = torch.nn.functional.rms_norm(torch.from_numpy(h.astype(np.float64)), (96,),
                                        weight=torch.from_numpy(g.astype(np.float64)), eps=1e-5).numpy()
    assert np.allclose(got, want, rtol=1e-13, atol=0)
    c = np.full(32, -0.25, np.float32)
    got = oracle.rmsnorm(c, np.full(32, 2.0, np.float32), 1e-5, lib=lib)
    assert np.allclose(got, -0.25 / np.sqrt(0.0625 + 1e-5) * 2.0, rtol=1e-14)


def pin_attention_library(lib=None):
    """One head over cache rows [0, pos] against torch's scaled_dot_product_attention
    in fp64; pos 0 returns v_0; q = 0 returns the mean of the V rows."""
    import torch
    rng = np.random.default_rng(7)
    hd, n = 16, 40
    K = synth.normal_bf16(7, 1, (n, hd), stddev=1.0)
    V = synth.normal_bf16(7, 2, (n, hd), stddev=1.0)
    q = rng.standard_normal(hd)
    for pos in (0, 1, 17, n - 1):
        got = oracle.attend_head(q, K, V, pos, lib=lib)
        Kt = torch.from_numpy(synth.bf16_to_f32(K[:pos + 1]).astype(np.float64))[None, None]
        Vt = torch.from_numpy(synth.bf16_to_f32(V[:pos + 1]).astype(np.float64))[None, None]
        want = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[None, None, None], Kt, Vt)
        assert np.allclose(got, want.numpy().reshape(-1), rtol=1e-12, atol=1e-14), pos
    assert np.array_equal(oracle.attend_head(q, K, V, 0, lib=lib), synth.bf16_to_f32(V[0]).astype(np.float64))
    got = oracle.attend_head(np.zeros(hd), K, V, 9, lib=lib)
    assert np.allclose(got, synth.bf16_to_f32(V[:10]).astype(np.float64).mean(axis=0), rtol=1e-13)


def pin_matvec_library(lib=None):
    """bf16 and int8-row-scale matvec against numpy fp64 matmul of the dequantised matrix."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal(72)
    wb = synth.normal_bf16(8, 1, (33, 72))
    assert _rel(oracle.matvec(wb, x, lib=lib), _deq(wb) @ x) < 1e-14
    q, s = synth.normal_q8_rows(8, 2, 33, 72)
    assert _rel(oracle.matvec((q, s), x, lib=lib), (q.astype(np.float64) * s[:, None].astype(np.float64)) @ x) < 1e-14


def pin_bf16_rounding(lib=None):
    """Rounding to bf16 against torch's float32 -> bfloat16 conversion (round to
    nearest even) on float32-representable values, plus the ties at 1 + 2^-8 and
    1 + 3 * 2^-8."""
    import torch
    x = np.random.default_rng(9).standard_normal(2000).astype(np.float32) * 0.03
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_round(float(v), lib=lib) for v in x], np.uint16)
    assert np.array_equal(got, want)
    assert oracle.bf16_round(1.0 + 2 ** -8, lib=lib) == 0x3F80
    assert oracle.bf16_round(1.0 + 3 * 2 ** -8, lib=lib) == 0x3F82
    assert oracle.bf16_round(-2.0, lib=lib) == 0xC000


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
