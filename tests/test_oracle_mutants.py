"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one: a dropped term, a wrong sign or index, a swapped
operand. Each mutant replaces one exact snippet of ``oracle/oracle.c``."""
import os
import subprocess

import pytest

import oracle
import pins

MUTANTS = {
    "rope_sign": ("x[i] = a * c - b * s;", "x[i] = a * c + b * s;"),
    "rope_freq": ("pow(theta, -2.0 * i / hd)", "pow(theta, -1.0 * i / hd)"),
    "rope_pos_off_by_one": ("double ang = (double)pos *", "double ang = (double)(pos + 1) *"),
    "norm_gain_dropped": ("xn[i] = (double)h[i] * inv * (double)g[i];", "xn[i] = (double)h[i] * inv;"),
    "norm_mean_dropped": ("sqrt(ss / n + eps)", "sqrt(ss + eps)"),
    "attn_scale_dropped": ("s[t] = acc * scale;", "s[t] = acc;"),
    "attn_current_row_excluded": ("for (int t = 0; t <= pos; ++t) {\n    double acc = 0.0;",
                                  "for (int t = 0; t <= pos; ++t) {\n    double acc = (t == pos) ? -1e30 : 0.0;"),
    "gqa_mapping": ("int kh = hh / group;", "int kh = hh % nkv;"),
    "silu_sign": ("z / (1.0 + exp(-z))", "z / (1.0 + exp(z))"),
    "swiglu_swapped": ("g[i] = silu(g[i]) * u[i];", "g[i] = g[i] * silu(u[i]);"),
    "mlp_residual_dropped": ("orc_matvec(&L->wd, int8, g, y);\n  for (int i = 0; i < E; ++i) h[i] = (float)((double)h[i] + y[i]);",
                             "orc_matvec(&L->wd, int8, g, y);\n  for (int i = 0; i < E; ++i) h[i] = (float)(y[i]);"),
    "v_stores_k": ("= orc_bf16_round(v[(size_t)kh * hd + i]);", "= orc_bf16_round(k[(size_t)kh * hd + i]);"),
    "int8_scale_dropped": ("* (double)m->s[r];", ";"),
    "bf16_truncates": ("nearbyint(ldexp(m, 8))", "trunc(ldexp(m, 8))"),
    "final_norm_wrong_gain": ("orc_rmsnorm(h, m->out_norm,", "orc_rmsnorm(h, m->layers[0].ffn_norm,"),
    "k_not_rotated": ("for (int kh = 0; kh < nkv; ++kh) orc_rope(", "for (int kh = 0; kh < 0; ++kh) orc_rope("),
    "softmax_not_normalised": ("for (int i = 0; i < hd; ++i) o[i] /= l;", ""),
    "boundary_in_f16_like": ("memcpy(hs, h, sizeof(float) * E);",
                             "memcpy(hs, h, sizeof(float) * E); if (s > 0) for (int i = 0; i < E; ++i) hs[i] = (float)(_Float16)hs[i];"),
    # (every mutant stays inside its arrays: the pins load it into this process)
    "rope_interleaved_pairs": ("double a = x[i], b = x[i + half];\n    x[i] = a * c - b * s;\n    x[i + half] = a * s + b * c;",
                               "double a = x[2 * i], b = x[2 * i + 1];\n    x[2 * i] = a * c - b * s;\n    x[2 * i + 1] = a * s + b * c;"),
    "attn_residual_dropped": ("orc_matvec(&L->wo, int8, o, y);\n  for (int i = 0; i < E; ++i) h[i] = (float)((double)h[i] + y[i]);",
                              "orc_matvec(&L->wo, int8, o, y);\n  for (int i = 0; i < E; ++i) h[i] = (float)(y[i]);"),
    "attn_scale_one_over_hd": ("double scale = 1.0 / sqrt((double)hd);", "double scale = 1.0 / (double)hd;"),
    "norm_eps_outside_sqrt": ("sqrt(ss / n + eps)", "(sqrt(ss / n) + eps)"),
    "softmax_sums_raw_scores": ("s[t] = exp(s[t] - m);\n    l += s[t];", "l += s[t];\n    s[t] = exp(s[t] - m);"),
    "scores_against_v": ("acc += q[i] * bf16_value(K[(long)t * hd + i]);", "acc += q[i] * bf16_value(V[(long)t * hd + i]);"),
    "embed_next_row": ("w_at(&m->embed, d->weight_int8, tokens[b], i)",
                       "w_at(&m->embed, d->weight_int8, (tokens[b] + 1) % d->vocab, i)"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"snippet for {name} must occur exactly once"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(source.replace(old, new))
    so = str(tmp_path / f"liboracle_{name}.so")
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", so, str(src), "-lm"])
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib=so)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the mutant {name}"


def test_unmutated_passes_all(source, tmp_path):
    src = tmp_path / "oracle_same.c"
    src.write_text(source)
    so = str(tmp_path / "liboracle_same.so")
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", so, str(src), "-lm"])
    for pin in pins.ALL_PINS:
        pin(lib=so)
