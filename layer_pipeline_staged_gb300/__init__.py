"""Layer-staged eager decode step on one GB300: Python binding of ``liblps.so``.

The binding only marshals arguments; every step of the decode path runs in the
library's CUDA kernels. The same names as the C ABI (``include/lps.h``) are
exported: ``stage_plan_create``, ``model_bind``, ``decode_step``,
``decode_step_deferred``, ``pending_wait`` and the rest. PyTorch, when it is
importable and a GPU is present, supplies the device memory (its caching
allocator, through the ABI's alloc/free hooks) and the per-stage streams.

Weights are passed as host numpy arrays: bf16 matrices as uint16 bit patterns
[rows, cols]; int8 matrices as (q int8 [rows, cols], scale f32 [rows]) pairs;
gains as f32 vectors. Layout is row-major [out, in].
"""
from __future__ import annotations

import ctypes
import gc

import numpy as np

from . import _capi
from ._capi import (KERNELS, LPS_EBUSY, LPS_ECUDA, LPS_EINVAL, LPS_ENOMEM, LPS_ETIMEDOUT,  # noqa: F401
                    LPS_FLAG_KEEP_ATTN_OUT, LPS_FLAG_SERIAL_STEPS, LPS_FLAG_SINGLE_STREAM, LPS_FLAG_VERIFY, LPS_FLAG_PERSISTENT, LPS_FLAG_GRAPH,
                    LPS_NOALLOC_SCRATCH_BYTES,
                    LPS_OK)

__all__ = ["LpsError", "StagePlan", "Model", "Pending", "stage_plan_create", "stage_plan_from_counts",
           "stage_plan_solve", "model_stage_bytes", "model_bind", "decode_step", "decode_step_deferred",
           "pending_wait", "pending_free", "decode_step_device", "load"]


class LpsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def load():
    return _capi.load()


def _check(rc: int) -> int:
    if rc < 0:
        raise LpsError(rc, _capi.load().last_error_string().decode())
    return rc


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    if not (isinstance(a, np.ndarray) and a.flags.c_contiguous):
        raise ValueError("weights must be C-contiguous numpy arrays")
    return a.ctypes.data


def _matrix(m) -> _capi.Matrix:
    if isinstance(m, tuple):
        return _capi.Matrix(_ptr(m[0]), _ptr(m[1]))
    return _capi.Matrix(_ptr(m), None)


class StagePlan:
    """The stage fence of a trunk: from cuts, the even split, or per-stage layer counts."""

    def __init__(self, n_layers: int | None = None, cuts=None, n_stages: int | None = None, counts=None):
        L = load()
        h = ctypes.c_void_p()
        if counts is not None:
            c = np.ascontiguousarray(counts, np.int32)
            _check(L.stage_plan_from_counts(_ptr(c), len(c), ctypes.byref(h)))
        elif cuts is not None:
            c = np.ascontiguousarray(cuts, np.int32)
            _check(L.stage_plan_create(n_layers, _ptr(c) if len(c) else None, len(c), ctypes.byref(h)))
        else:
            _check(L.stage_plan_create(n_layers, None, (n_stages or 1) - 1, ctypes.byref(h)))
        self.h = h

    @property
    def n_stages(self) -> int:
        return _check(load().stage_plan_n_stages(self.h))

    @property
    def fence(self) -> tuple:
        out = np.zeros(self.n_stages + 1, np.int32)
        _check(load().stage_plan_fence(self.h, _ptr(out), len(out)))
        return tuple(int(x) for x in out)

    def stage_of(self, il: int) -> int:
        return _check(load().stage_of(self.h, il))

    def __del__(self):
        if getattr(self, "h", None):
            load().stage_plan_destroy(self.h)
            self.h = None


class _TorchMemory:
    """Device memory and streams from PyTorch, handed to the library's hooks."""

    def __init__(self, device: int, n_streams: int):
        import torch
        self.torch = torch
        self.device = device
        self.streams = [torch.cuda.Stream(device=device) for _ in range(n_streams)]
        self.stream_handles = (ctypes.c_void_p * n_streams)(*[s.cuda_stream for s in self.streams])

        def _alloc(_ctx, nbytes):
            try:
                return int(torch.cuda.caching_allocator_alloc(int(nbytes), device=device))
            except Exception as e:  # the library then reports LPS_ENOMEM
                self.last_alloc_error = repr(e)
                return None

        def _free(_ctx, ptr):
            try:
                if ptr:
                    torch.cuda.caching_allocator_delete(int(ptr))
            except Exception as e:
                self.last_alloc_error = repr(e)

        self.last_alloc_error = None

        self.alloc = _capi.ALLOC_FN(_alloc)
        self.free = _capi.FREE_FN(_free)


def weights_struct(weights: dict, n_layers: int) -> "_capi.ModelWeights":
    """The C ABI's lps_model_weights over the host arrays of ``weights`` (which
    must stay alive while the struct is used)."""
    layers = (_capi.LayerWeights * n_layers)()
    for l, lw in enumerate(weights["layers"]):
        layers[l] = _capi.LayerWeights(_ptr(lw["attn_norm"]), _matrix(lw["wq"]), _matrix(lw["wk"]),
                                       _matrix(lw["wv"]), _matrix(lw["wo"]), _ptr(lw["ffn_norm"]),
                                       _matrix(lw["w_gate"]), _matrix(lw["w_up"]), _matrix(lw["w_down"]))
    w = _capi.ModelWeights(_matrix(weights["embed"]), _ptr(weights["out_norm"]), _matrix(weights["lm_head"]),
                           layers)
    w._layers = layers  # keep the array alive with the struct
    return w


class Model:
    """A model bound to one GPU over a stage plan (see ``model_bind``)."""

    def __init__(self, plan: StagePlan, desc: dict, weights: dict, device: int = 0, use_torch: bool | None = None):
        L = load()
        self.plan = plan
        self.desc = _capi.ModelDesc(**desc)
        self.B, self.V = self.desc.batch, self.desc.vocab
        self._keep = weights  # host arrays must stay alive during bind only, but keep for clarity
        w = weights_struct(weights, self.desc.n_layers)
        if use_torch is None:
            try:
                import torch
                use_torch = torch.cuda.is_available()
            except Exception:
                use_torch = False
        rt = _capi.Runtime()
        rt.device = device
        self._mem = None
        if use_torch:
            self._mem = _TorchMemory(device, plan.n_stages + 1)
            rt.alloc = self._mem.alloc
            rt.free = self._mem.free
            rt.streams = ctypes.cast(self._mem.stream_handles, ctypes.POINTER(ctypes.c_void_p))
        h = ctypes.c_void_p()
        # no garbage collection (and so no other model's destroy) inside the allocator callbacks
        gc_was_on = gc.isenabled()
        gc.collect()
        gc.disable()
        try:
            rc = L.model_bind(plan.h, ctypes.byref(self.desc), ctypes.byref(w), ctypes.byref(rt), ctypes.byref(h))
        finally:
            if gc_was_on:
                gc.enable()
        if rc < 0 and self._mem is not None and self._mem.last_alloc_error:
            raise LpsError(rc, L.last_error_string().decode() + f" (allocator: {self._mem.last_alloc_error})")
        _check(rc)
        self.h = h
        self._keep = None

    def close(self):
        if getattr(self, "h", None):
            load().model_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()

    def _vec(self, x) -> np.ndarray:
        return np.ascontiguousarray(np.broadcast_to(np.asarray(x, dtype=np.int32), (self.B,)))

    def _pos(self, pos) -> np.ndarray:
        # verify rows (LPS_FLAG_VERIFY): a scalar is the first row's position
        if self.desc.flags & _capi.LPS_FLAG_VERIFY and np.ndim(pos) == 0:
            return np.ascontiguousarray(int(pos) + np.arange(self.B, dtype=np.int32))
        return self._vec(pos)

    def decode_step(self, tokens, pos, out: np.ndarray | None = None) -> np.ndarray:
        t, p = self._vec(tokens), self._pos(pos)
        out = np.empty((self.B, self.V), np.float32) if out is None else out
        _check(load().decode_step(self.h, _ptr(t), _ptr(p), _ptr(out)))
        return out

    def decode_step_deferred(self, tokens, pos) -> "Pending":
        t, p = self._vec(tokens), self._pos(pos)
        h = ctypes.c_void_p()
        _check(load().decode_step_deferred(self.h, _ptr(t), _ptr(p), ctypes.byref(h)))
        return Pending(self, h)

    def decode_step_device(self, tokens_dev_ptr: int, pos, logits_dev_ptr: int):
        p = self._pos(pos)
        _check(load().decode_step_device(self.h, ctypes.c_void_p(tokens_dev_ptr), _ptr(p),
                                         ctypes.c_void_p(logits_dev_ptr)))

    def prefill(self, tokens, pos0: int = 0, b: int = 0, chunk: int = 0, logits: bool = True):
        """model_prefill: the prompt tokens of sequence b at positions pos0.. in
        chunks through the stages; returns the last token's logits [vocab] (or None)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
        out = np.empty(self.V, np.float32) if logits else None
        _check(load().model_prefill(self.h, int(b), _ptr(t), int(t.size), int(pos0), int(chunk),
                                    _ptr(out) if logits else None))
        return out

    def synchronize(self):
        _check(load().model_synchronize(self.h))

    def stream(self, s: int) -> int:
        out = ctypes.c_void_p()
        _check(load().model_stream(self.h, s, ctypes.byref(out)))
        return out.value or 0

    def stats(self) -> dict:
        st = _capi.Stats()
        _check(load().model_stats(self.h, ctypes.byref(st)))
        d = {k: getattr(st, k) for k, _ in _capi.Stats._fields_ if k != "fence"}
        d["fence"] = tuple(st.fence[: st.n_stages + 1])
        return d

    def kv_export(self, layer: int, b: int):
        d = self.desc
        buf = np.empty((2, d.n_kv_heads, d.max_ctx, d.head_dim), np.uint16)
        _check(load().model_kv_export(self.h, layer, b, _ptr(buf), buf.nbytes))
        return buf[0], buf[1]

    def kv_import(self, layer: int, b: int, k: np.ndarray, v: np.ndarray, filled: int):
        buf = np.ascontiguousarray(np.stack([k, v]), np.uint16)
        _check(load().model_kv_import(self.h, layer, b, _ptr(buf), buf.nbytes, filled))

    def attn_out(self, layer: int, b: int) -> np.ndarray:
        out = np.empty((self.desc.n_q_heads, self.desc.head_dim), np.float32)
        _check(load().model_attn_out(self.h, layer, b, _ptr(out)))
        return out

    def trace_enable(self, capacity: int = 1 << 16):
        """Record every launch of the following steps (kind, stage, layer, step, device start/end ns)."""
        _check(load().model_trace_enable(self.h, capacity))

    def trace_read(self) -> tuple:
        """(records, dropped): the recorded launches in launch order as a list of dicts; restarts the recording."""
        cap = 1 << 20
        buf = (_capi.TraceRecord * cap)()
        n = ctypes.c_int()
        dropped = ctypes.c_uint64()
        _check(load().model_trace_read(self.h, buf, cap, ctypes.byref(n), ctypes.byref(dropped)))
        names = {v: k for k, v in KERNELS.items()}
        recs = [dict(kind=names.get(r.kind, r.kind), stage=r.stage, layer=r.layer, step=r.step, start_ns=r.start_ns,
                     end_ns=r.end_ns) for r in buf[: n.value]]
        return recs, dropped.value

    def trace_disable(self):
        _check(load().model_trace_disable(self.h))

    def set_wait_limit(self, cycles: int):
        """Test hook: the SM cycles a device-side wait may take before the kernel reports an error (0: default)."""
        _check(load().model_set_wait_limit(self.h, int(cycles)))

    def set_serial_steps(self, serial: bool):
        _check(load().model_set_serial_steps(self.h, int(serial)))

    def time_kernel(self, kind: str, enable: bool = True):
        _check(load().model_time_kernel(self.h, KERNELS[kind], int(enable)))

    def kernel_time(self, kind: str):
        ms = ctypes.c_double()
        n = ctypes.c_uint64()
        _check(load().model_kernel_time(self.h, KERNELS[kind], ctypes.byref(ms), ctypes.byref(n)))
        return ms.value, n.value


class Pending:
    """Logits of a deferred step, still on the device (``decode_step_deferred``)."""

    def __init__(self, model: Model, h):
        self.model = model
        self.h = h

    def wait(self, timeout_ms: int = -1, out: np.ndarray | None = None) -> np.ndarray:
        out = np.empty((self.model.B, self.model.V), np.float32) if out is None else out
        _check(load().pending_wait(self.h, _ptr(out), timeout_ms))
        return out

    def free(self):
        if getattr(self, "h", None):
            load().pending_free(self.h)
            self.h = None

    def __del__(self):
        self.free()


# ---- the C ABI's names ----

def stage_plan_create(n_layers: int, cuts=None, n_stages: int | None = None) -> StagePlan:
    return StagePlan(n_layers, cuts=cuts, n_stages=n_stages)


def stage_plan_from_counts(counts) -> StagePlan:
    return StagePlan(counts=counts)


def stage_plan_solve(layer_bytes, layer_unit_bytes, stage_free, stage_fixed=None, max_units: int = 1 << 40):
    """Memory-balancing cuts (the C ABI's stage_plan_solve): returns (cuts, units), units = -1
    when nothing fits (the cuts are then the even split)."""
    lb = np.ascontiguousarray(layer_bytes, np.uint64)
    lu = np.ascontiguousarray(layer_unit_bytes, np.uint64)
    sf = np.ascontiguousarray(stage_free, np.uint64)
    if len(lu) != len(lb):
        raise ValueError("layer_bytes and layer_unit_bytes differ in length")
    sx = None if stage_fixed is None else np.ascontiguousarray(stage_fixed, np.uint64)
    if sx is not None and len(sx) != len(sf):
        raise ValueError("stage_fixed and stage_free differ in length")
    cuts = np.zeros(max(len(sf) - 1, 1), np.int32)
    units = ctypes.c_int64()
    _check(load().stage_plan_solve(len(lb), len(sf), _ptr(lb), _ptr(lu), _ptr(sf), _ptr(sx), int(max_units),
                                   _ptr(cuts), ctypes.byref(units)))
    return [int(c) for c in cuts[:len(sf) - 1]], int(units.value)


def model_stage_bytes(desc: dict) -> dict:
    """The byte model of a bound model (the C ABI's model_stage_bytes): per-layer weight and
    per-position KV bytes, and the embedding / head / per-stage workspace constants."""
    d = _capi.ModelDesc(**desc)
    lb = np.zeros(d.n_layers, np.uint64)
    lu = np.zeros(d.n_layers, np.uint64)
    first, last, every = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    _check(load().model_stage_bytes(ctypes.byref(d), _ptr(lb), _ptr(lu), ctypes.byref(first), ctypes.byref(last),
                                    ctypes.byref(every)))
    return {"layer_bytes": lb, "layer_unit_bytes": lu, "first_stage_bytes": int(first.value),
            "last_stage_bytes": int(last.value), "every_stage_bytes": int(every.value)}


def model_bind(plan: StagePlan, desc: dict, weights: dict, device: int = 0, use_torch: bool | None = None) -> Model:
    return Model(plan, desc, weights, device=device, use_torch=use_torch)


def decode_step(model: Model, tokens, pos, out=None) -> np.ndarray:
    return model.decode_step(tokens, pos, out)


def decode_step_deferred(model: Model, tokens, pos) -> Pending:
    return model.decode_step_deferred(tokens, pos)


def pending_wait(p: Pending, timeout_ms: int = -1, out=None) -> np.ndarray:
    return p.wait(timeout_ms, out)


def pending_free(p: Pending):
    p.free()


def model_prefill(model: Model, b: int, tokens, pos0: int = 0, chunk: int = 0, logits: bool = True):
    return model.prefill(tokens, pos0=pos0, b=b, chunk=chunk, logits=logits)


def decode_step_device(model: Model, tokens_dev_ptr: int, pos, logits_dev_ptr: int):
    model.decode_step_device(tokens_dev_ptr, pos, logits_dev_ptr)
