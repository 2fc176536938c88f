"""Seeded synthetic workloads for the layer-staged decoder.

This package is the one thing the CPU oracle and the CUDA path share: it
defines the workload shapes and draws the weights and token ids, and it holds
none of the decode step's arithmetic (see ``synth.c`` for the generator's
definition). Both sides read what it returns.

Workload recipe (the decoder configurations of the layer-staged decode step):
weights ~ N(0, 0.02) drawn per tensor from a counter-based stream, RMSNorm gains
1, tokens uniform in [0, vocab). The zero-padded-head workload pads the base
model's drawn weights with zero q/k/v rows and zero o_proj columns at the global
end of each head axis (zero-padded dummy heads, "TP3 support via zero-padded
dummy heads", Geometry and Weight-padding design).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (gcc, no GPU needed)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-shared", "-fPIC", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, dbl, vp = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            L.synth_normal_bf16.argtypes = [u64, u64, dbl, vp, u64]
            L.synth_normal_f32.argtypes = [u64, u64, dbl, dbl, vp, u64]
            L.synth_normal_q8_rows.argtypes = [u64, u64, dbl, u64, u64, vp, vp]
            L.synth_tokens.argtypes = [u64, u64, ctypes.c_uint32, vp, u64]
            L.synth_uniform_bf16.argtypes = [u64, u64, dbl, vp, u64]
            L.synth_set_threads.argtypes = [ctypes.c_int]
            for f in ("synth_normal_bf16", "synth_normal_f32", "synth_normal_q8_rows", "synth_tokens",
                      "synth_uniform_bf16", "synth_set_threads"):
                getattr(L, f).restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


# ---------------------------------------------------------------------------
# draws
# ---------------------------------------------------------------------------

def normal_bf16(seed: int, stream: int, shape, stddev: float = 0.02) -> np.ndarray:
    """bf16 bit patterns (uint16) of round((float)(stddev * N)) for every element."""
    out = np.empty(shape, dtype=np.uint16)
    if out.size:
        lib().synth_normal_bf16(seed, stream, stddev, _ptr(out), out.size)
    return out


def normal_f32(seed: int, stream: int, shape, mean: float = 0.0, stddev: float = 0.02) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    if out.size:
        lib().synth_normal_f32(seed, stream, mean, stddev, _ptr(out), out.size)
    return out


def normal_q8_rows(seed: int, stream: int, rows: int, cols: int, stddev: float = 0.02):
    """Symmetric per-row int8 quantisation of the float draws: (q int8 [rows, cols], s f32 [rows])."""
    q = np.empty((rows, cols), dtype=np.int8)
    s = np.empty((rows,), dtype=np.float32)
    if rows and cols:
        lib().synth_normal_q8_rows(seed, stream, stddev, rows, cols, _ptr(q), _ptr(s))
    return q, s


def tokens(seed: int, stream: int, vocab: int, n: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.int32)
    if n:
        lib().synth_tokens(seed, stream, vocab, _ptr(out), n)
    return out


def uniform_bf16(seed: int, stream: int, shape, a: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    if out.size:
        lib().synth_uniform_bf16(seed, stream, a, _ptr(out), out.size)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    index: int            # seeds: weights 1000 + index, tokens 2000 + index
    n_layers: int
    n_embd: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    weight_dtype: str     # "bf16" or "int8" (int8 with one fp32 scale per output row)
    batch: int
    ctx: int              # context length filled before the measured decode steps
    steps: int            # teacher-forced decode steps after the context
    cuts: tuple           # stage cuts (the fence is [0, *cuts, n_layers])
    rope_theta: float = 10000.0
    rms_eps: float = 1e-5
    pad_q_heads: int = 0  # > 0: zero-padded-head workload widened to this many q heads
    pad_kv_heads: int = 0

    @property
    def seed_w(self) -> int:
        return 1000 + self.index

    @property
    def seed_t(self) -> int:
        return 2000 + self.index

    @property
    def q_heads(self) -> int:
        """q heads as bound (padded width for the zero-padded workload)."""
        return self.pad_q_heads or self.n_q_heads

    @property
    def kv_heads(self) -> int:
        return self.pad_kv_heads or self.n_kv_heads

    @property
    def max_ctx(self) -> int:
        return self.ctx + self.steps

    @property
    def fence(self) -> tuple:
        return (0, *self.cuts, self.n_layers)

    def replace(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)

    def base(self) -> "ModelConfig":
        """The unpadded model the zero-padded workload is derived from."""
        return self.replace(pad_q_heads=0, pad_kv_heads=0)

    # ---- algorithmic bytes of one decode step (all weights once, KV read over
    # [0, pos] for every layer and sequence, the KV row write, logits out) ----
    def weight_bytes(self) -> int:
        d, hd, L = self.n_embd, self.head_dim, self.n_layers
        nq, nkv = self.q_heads, self.kv_heads
        el = 1 if self.weight_dtype == "int8" else 2
        per_layer_rows = (nq + 2 * nkv) * hd + d + 2 * self.ffn + d  # qkv, o, gate+up, down (rows)
        per_layer = ((nq + 2 * nkv) * hd * d + d * nq * hd + 2 * self.ffn * d + d * self.ffn) * el
        per_layer += 2 * d * 4  # two RMSNorm gain vectors
        scales = per_layer_rows * 4 if el == 1 else 0
        head = self.vocab * d * el + (self.vocab * 4 if el == 1 else 0) + d * 4
        embed_rows = self.batch * (d * el + (4 if el == 1 else 0))
        return L * (per_layer + scales) + head + embed_rows

    def kv_bytes(self, pos: int) -> int:
        """KV bytes read (positions [0, pos]) plus the row written, all layers and sequences."""
        row = self.kv_heads * self.head_dim * 2  # bf16 K or V row of one layer
        return self.n_layers * self.batch * 2 * row * (pos + 1 + 1)

    def step_bytes(self, pos: int) -> int:
        return self.weight_bytes() + self.kv_bytes(pos) + self.batch * self.vocab * 4


CONFIGS = {
    "tiny": ModelConfig("tiny", 0, 4, 256, 4, 2, 64, 688, 4096, "bf16", 1, 64, 16, (2,)),
    "1b": ModelConfig("1b", 1, 16, 2048, 32, 8, 64, 8192, 32000, "bf16", 1, 1024, 128, (4, 8, 12)),
    "8b": ModelConfig("8b", 2, 32, 4096, 32, 8, 128, 14336, 128256, "bf16", 1, 8192, 256, (8, 16, 24)),
    "8b_q8": ModelConfig("8b_q8", 3, 32, 4096, 32, 8, 128, 14336, 128256, "int8", 1, 32768, 128, (16,)),
    "8b_q8_b8": ModelConfig("8b_q8_b8", 3, 32, 4096, 32, 8, 128, 14336, 128256, "int8", 8, 32768, 128, (16,)),
    "padded": ModelConfig("padded", 4, 24, 3072, 32, 8, 128, 8192, 65536, "bf16", 4, 4096, 64, (6, 15),
                          pad_q_heads=48, pad_kv_heads=12),
}

# stream ids of the per-tensor draws
S_EMBED, S_HEAD, S_OUT_NORM = 1, 2, 3
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def _layer_stream(layer: int, k: int) -> int:
    return 100 + 16 * layer + k


def _matrix(cfg: ModelConfig, seed: int, stream: int, rows: int, cols: int):
    if cfg.weight_dtype == "int8":
        return normal_q8_rows(seed, stream, rows, cols)
    return normal_bf16(seed, stream, (rows, cols))


def make_weights(cfg: ModelConfig, seed: int | None = None, random_gains: bool = False,
                 layers: int | None = None) -> dict:
    """Draw every tensor of the model (host numpy arrays).

    bf16 matrices are uint16 bit patterns [rows, cols]; int8 matrices are
    (q int8 [rows, cols], s f32 [rows]) pairs. Gains are fp32 ones unless
    ``random_gains`` (then 1 + N(0, 0.1), used to make a dropped gain visible).
    ``layers`` limits the layers drawn (the rest of the shape is unchanged).
    The zero-padded workload is drawn at its base shape and padded.
    """
    if cfg.pad_q_heads:
        return pad_heads(make_weights(cfg.base(), seed, random_gains, layers), cfg)
    seed = cfg.seed_w if seed is None else seed
    d, hd, nq, nkv, f, V = cfg.n_embd, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads, cfg.ffn, cfg.vocab

    def gain(stream):
        if random_gains:
            return normal_f32(seed, stream, (d,), mean=1.0, stddev=0.1)
        return np.ones((d,), dtype=np.float32)

    w = {"embed": _matrix(cfg, seed, S_EMBED, V, d), "lm_head": _matrix(cfg, seed, S_HEAD, V, d),
         "out_norm": gain(S_OUT_NORM), "layers": []}
    for l in range(cfg.n_layers if layers is None else layers):
        s = lambda k: _layer_stream(l, k)  # noqa: E731
        w["layers"].append({
            "attn_norm": gain(s(0)),
            "wq": _matrix(cfg, seed, s(1), nq * hd, d),
            "wk": _matrix(cfg, seed, s(2), nkv * hd, d),
            "wv": _matrix(cfg, seed, s(3), nkv * hd, d),
            "wo": _matrix(cfg, seed, s(4), d, nq * hd),
            "ffn_norm": gain(s(5)),
            "w_gate": _matrix(cfg, seed, s(6), f, d),
            "w_up": _matrix(cfg, seed, s(7), f, d),
            "w_down": _matrix(cfg, seed, s(8), d, f),
        })
    return w


def _pad_rows(m, rows: int):
    if isinstance(m, tuple):
        q, s = m
        return (np.concatenate([q, np.zeros((rows - q.shape[0], q.shape[1]), q.dtype)]),
                np.concatenate([s, np.zeros((rows - s.shape[0],), s.dtype)]))
    return np.concatenate([m, np.zeros((rows - m.shape[0], m.shape[1]), m.dtype)])


def _pad_cols(m, cols: int):
    if isinstance(m, tuple):
        q, s = m
        return (np.ascontiguousarray(np.pad(q, ((0, 0), (0, cols - q.shape[1])))), s)
    return np.ascontiguousarray(np.pad(m, ((0, 0), (0, cols - m.shape[1]))))


def pad_heads(w: dict, cfg: ModelConfig) -> dict:
    """Zero-padded dummy heads appended at the global end of each head axis:
    zero rows in W_q, W_k, W_v and zero input columns in W_o; the embedding,
    norms, MLP and head are untouched ("TP3 support via zero-padded dummy
    heads", Weight-padding design, per-suffix spec table)."""
    hd = cfg.head_dim
    out = {k: v for k, v in w.items() if k != "layers"}
    out["layers"] = []
    for lw in w["layers"]:
        p = dict(lw)
        p["wq"] = _pad_rows(lw["wq"], cfg.pad_q_heads * hd)
        p["wk"] = _pad_rows(lw["wk"], cfg.pad_kv_heads * hd)
        p["wv"] = _pad_rows(lw["wv"], cfg.pad_kv_heads * hd)
        p["wo"] = _pad_cols(lw["wo"], cfg.pad_q_heads * hd)
        out["layers"].append(p)
    return out


def make_tokens(cfg: ModelConfig, n: int, seed: int | None = None) -> np.ndarray:
    """Teacher-forced token ids [n, batch]: sequence b draws substream b."""
    seed = cfg.seed_t if seed is None else seed
    return np.stack([tokens(seed, b, cfg.vocab, n) for b in range(cfg.batch)], axis=1).astype(np.int32)
