"""ORACLE -- test infrastructure, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import, call, link or execute anything under ``oracle/``. The oracle shares
no code with the CUDA path; the only thing both read is the seeded workload
from ``synth``.

A ctypes wrapper over ``oracle.c``: a plain, slow CPU decoder for one eager
decode step of a layer-staged decoder trunk (fp64 arithmetic, f32 residual
stream, bf16 KV cache). Parity pins: ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_libs: dict = {}

CFLAGS = ["-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC"]


def build(src: str = SRC, out: str = SO, force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP over output rows)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "n_embd", "n_q_heads", "n_kv_heads", "head_dim",
                                            "ffn", "vocab", "weight_int8", "max_ctx", "batch")] + \
               [("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)]


class _Mat(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("s", ctypes.c_void_p), ("rows", ctypes.c_int), ("cols", ctypes.c_int)]


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` selects another build of it."""
    path = path or build()
    with _lock:
        if path in _libs:
            return _libs[path]
        L = ctypes.CDLL(path)
        vp, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.orc_create.restype = vp
        L.orc_create.argtypes = [ctypes.POINTER(_Desc), vp, i]
        L.orc_destroy.argtypes = [vp]
        L.orc_destroy.restype = None
        L.orc_set_layer.argtypes = [vp, i] + [vp] * 16
        L.orc_set_layer.restype = None
        L.orc_set_global.argtypes = [vp] * 6
        L.orc_set_global.restype = None
        L.orc_decode_step.argtypes = [vp, vp, vp, vp]
        L.orc_decode_step.restype = i
        L.orc_kv_export.argtypes = [vp, i, i, vp, vp]
        L.orc_kv_export.restype = i
        L.orc_kv_import.argtypes = [vp, i, i, vp, vp, i]
        L.orc_kv_import.restype = i
        L.orc_attn_out.argtypes = [vp, i, i, vp]
        L.orc_attn_out.restype = i
        L.orc_boundary.argtypes = [vp, i, vp]
        L.orc_boundary.restype = i
        L.orc_set_threads.argtypes = [i]
        L.orc_set_threads.restype = None
        L.orc_get_threads.restype = i
        L.orc_matvec.argtypes = [ctypes.POINTER(_Mat), i, vp, vp]
        L.orc_matvec.restype = None
        L.orc_rmsnorm.argtypes = [vp, vp, i, d, vp]
        L.orc_rmsnorm.restype = None
        L.orc_rope.argtypes = [vp, i, i, d]
        L.orc_rope.restype = None
        L.orc_attend_head.argtypes = [vp, vp, vp, i, i, vp]
        L.orc_attend_head.restype = None
        L.orc_bf16_round.argtypes = [d]
        L.orc_bf16_round.restype = ctypes.c_uint16
        _libs[path] = L
        return L


def _p(a) -> int | None:
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous, type(a)
    return a.ctypes.data


def _wp(m):
    """(weight pointer, scale pointer) of a bf16 array or an int8 (q, s) pair."""
    if isinstance(m, tuple):
        return _p(m[0]), _p(m[1])
    return _p(m), None


class Oracle:
    """The CPU decoder over host weights (borrowed, kept alive by this object)."""

    def __init__(self, cfg, weights: dict, fence=None, max_ctx: int | None = None, lib: str | None = None,
                 threads: int | None = None):
        self.L = load(lib)
        self.cfg = cfg
        self.w = weights
        self.fence = tuple(cfg.fence if fence is None else fence)
        n_layers = len(weights["layers"])
        d = _Desc(n_layers=n_layers, n_embd=cfg.n_embd, n_q_heads=cfg.q_heads, n_kv_heads=cfg.kv_heads,
                  head_dim=cfg.head_dim, ffn=cfg.ffn, vocab=cfg.vocab,
                  weight_int8=1 if cfg.weight_dtype == "int8" else 0,
                  max_ctx=max_ctx or cfg.max_ctx, batch=cfg.batch, rope_theta=cfg.rope_theta,
                  rms_eps=cfg.rms_eps)
        self.desc = d
        fence_arr = np.asarray(self.fence, dtype=np.int32)
        if threads:
            self.L.orc_set_threads(threads)
        self.m = self.L.orc_create(ctypes.byref(d), _p(fence_arr), len(self.fence) - 1)
        if not self.m:
            raise ValueError("oracle: invalid description or fence")
        for l, lw in enumerate(weights["layers"]):
            args = [_p(lw["attn_norm"]), *_wp(lw["wq"]), *_wp(lw["wk"]), *_wp(lw["wv"]), *_wp(lw["wo"]),
                    _p(lw["ffn_norm"]), *_wp(lw["w_gate"]), *_wp(lw["w_up"]), *_wp(lw["w_down"])]
            self.L.orc_set_layer(self.m, l, *args)
        self.L.orc_set_global(self.m, *_wp(weights["embed"]), _p(weights["out_norm"]), *_wp(weights["lm_head"]))

    def close(self):
        if getattr(self, "m", None):
            self.L.orc_destroy(self.m)
            self.m = None

    def __del__(self):
        self.close()

    def step(self, tokens, pos) -> np.ndarray:
        B = self.desc.batch
        t = np.ascontiguousarray(np.broadcast_to(np.asarray(tokens, dtype=np.int32), (B,)))
        p = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int32), (B,)))
        out = np.empty((B, self.desc.vocab), dtype=np.float32)
        rc = self.L.orc_decode_step(self.m, _p(t), _p(p), _p(out))
        if rc != 0:
            raise ValueError(f"oracle: decode step refused (rc={rc})")
        return out

    def kv_export(self, layer: int, b: int):
        shape = (self.desc.n_kv_heads, self.desc.max_ctx, self.desc.head_dim)
        k = np.empty(shape, np.uint16)
        v = np.empty(shape, np.uint16)
        if self.L.orc_kv_export(self.m, layer, b, _p(k), _p(v)) != 0:
            raise ValueError("oracle: bad kv_export index")
        return k, v

    def kv_import(self, layer: int, b: int, k: np.ndarray, v: np.ndarray, filled: int):
        k = np.ascontiguousarray(k, np.uint16)
        v = np.ascontiguousarray(v, np.uint16)
        assert k.size == v.size == self.desc.n_kv_heads * self.desc.max_ctx * self.desc.head_dim
        if self.L.orc_kv_import(self.m, layer, b, _p(k), _p(v), filled) != 0:
            raise ValueError("oracle: bad kv_import")

    def attn_out(self, layer: int, b: int) -> np.ndarray:
        out = np.empty((self.desc.n_q_heads, self.desc.head_dim), np.float64)
        if self.L.orc_attn_out(self.m, layer, b, _p(out)) != 0:
            raise ValueError("oracle: bad attn_out index")
        return out

    def boundary(self, s: int) -> np.ndarray:
        out = np.empty((self.desc.n_embd,), np.float32)
        if self.L.orc_boundary(self.m, s, _p(out)) != 0:
            raise ValueError("oracle: bad stage")
        return out


# ---- building blocks, exposed for the pins ----

def rmsnorm(h: np.ndarray, g: np.ndarray, eps: float, lib: str | None = None) -> np.ndarray:
    h = np.ascontiguousarray(h, np.float32)
    g = np.ascontiguousarray(g, np.float32)
    out = np.empty(h.shape, np.float64)
    load(lib).orc_rmsnorm(_p(h), _p(g), h.size, eps, _p(out))
    return out


def rope(x: np.ndarray, pos: int, theta: float = 10000.0, lib: str | None = None) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True)
    load(lib).orc_rope(_p(x), x.size, pos, theta)
    return x


def attend_head(q: np.ndarray, K: np.ndarray, V: np.ndarray, pos: int, lib: str | None = None) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.uint16)
    V = np.ascontiguousarray(V, np.uint16)
    out = np.empty(q.shape, np.float64)
    load(lib).orc_attend_head(_p(q), _p(K), _p(V), pos, q.size, _p(out))
    return out


def matvec(w, x: np.ndarray, lib: str | None = None) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    wp, sp = _wp(w)
    arr = w[0] if isinstance(w, tuple) else w
    m = _Mat(w=wp, s=sp, rows=arr.shape[0], cols=arr.shape[1])
    y = np.empty((arr.shape[0],), np.float64)
    load(lib).orc_matvec(ctypes.byref(m), 1 if isinstance(w, tuple) else 0, _p(x), _p(y))
    return y


def bf16_round(x: float, lib: str | None = None) -> int:
    return int(load(lib).orc_bf16_round(float(x)))
