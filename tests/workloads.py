"""Test helpers: bind the library on a synthetic workload and compare with the oracle."""
from __future__ import annotations

import numpy as np

import layer_pipeline_staged_gb300 as lps
import synth

TOL_BF16 = 2e-3  # max-abs error <= TOL * max|logit| per step and sequence (bf16 weights)
TOL_INT8 = 5e-3  # (int8 row-scale weights)


def tol(cfg) -> float:
    return TOL_INT8 if cfg.weight_dtype == "int8" else TOL_BF16


def desc(cfg, max_ctx: int | None = None, flags: int = 0, pending_depth: int = 0, layers: int | None = None) -> dict:
    return dict(n_layers=layers or cfg.n_layers, n_embd=cfg.n_embd, n_q_heads=cfg.q_heads, n_kv_heads=cfg.kv_heads,
                head_dim=cfg.head_dim, ffn=cfg.ffn, vocab=cfg.vocab,
                weight_dtype=1 if cfg.weight_dtype == "int8" else 0, kv_dtype=0,
                max_ctx=max_ctx or cfg.max_ctx, batch=cfg.batch, pending_depth=pending_depth,
                rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps, flags=flags)


def bind(cfg, w, fence=None, max_ctx: int | None = None, flags: int = 0, pending_depth: int = 0) -> lps.Model:
    n_layers = len(w["layers"])
    fence = tuple(fence or cfg.fence)
    plan = lps.stage_plan_create(n_layers, cuts=list(fence[1:-1]))
    assert plan.fence == fence
    return lps.model_bind(plan, desc(cfg, max_ctx, flags, pending_depth, layers=n_layers), w)


def rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """max|got - ref| / max|ref| per row (sequence)."""
    got = got.reshape(-1, got.shape[-1]).astype(np.float64)
    ref = ref.reshape(-1, ref.shape[-1]).astype(np.float64)
    return np.max(np.abs(got - ref), axis=1) / np.max(np.abs(ref), axis=1)


def assert_close(got, ref, cfg, what=""):
    e = rel_err(got, ref)
    assert np.all(e <= tol(cfg)), f"{what}: max-abs error {e.max():.3e} x max|logit| > {tol(cfg)}"
    return float(e.max())


def iter_random_kv(cfg, seed: int, layers: int, max_ctx: int, filled: int):
    """Synthetic cache rows [0, filled) for every (layer, sequence): uniform bf16
    in [-1, 1), yielded one (layer, sequence) at a time."""
    for l in range(layers):
        for b in range(cfg.batch):
            k = synth.uniform_bf16(seed, 2 * (l * cfg.batch + b), (cfg.kv_heads, max_ctx, cfg.head_dim))
            v = synth.uniform_bf16(seed, 2 * (l * cfg.batch + b) + 1, (cfg.kv_heads, max_ctx, cfg.head_dim))
            k[:, filled:] = 0
            v[:, filled:] = 0
            yield (l, b), (k, v)


def random_kv(cfg, seed: int, layers: int, max_ctx: int, filled: int):
    return dict(iter_random_kv(cfg, seed, layers, max_ctx, filled))
