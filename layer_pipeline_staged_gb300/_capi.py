"""ctypes declarations mirroring ``include/lps.h`` (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblps.so")

LPS_OK = 0
LPS_EINVAL = -1
LPS_ENOMEM = -2
LPS_ECUDA = -3
LPS_ETIMEDOUT = -4
LPS_EBUSY = -5

LPS_WEIGHT_BF16 = 0
LPS_WEIGHT_INT8_ROWSCALE = 1
LPS_KV_BF16 = 0
LPS_NOALLOC_SCRATCH_BYTES = 8 << 20
LPS_FLAG_SINGLE_STREAM = 1
LPS_FLAG_KEEP_ATTN_OUT = 2
LPS_FLAG_SERIAL_STEPS = 4
LPS_FLAG_VERIFY = 8
LPS_FLAG_PERSISTENT = 16
LPS_FLAG_GRAPH = 32

KERNELS = {"qkv": 0, "attn": 1, "oproj": 2, "gateup": 3, "down": 4, "head": 5, "embed": 6, "stage": 7, "merge": 8,
           "pf_split": 9, "pf_gemm": 10, "pf_attn": 11, "pf_merge": 12}

# every entry point the header declares
EXPORTS = (
    "stage_plan_create", "stage_plan_from_counts", "stage_plan_destroy", "stage_plan_n_stages",
    "stage_plan_fence", "stage_of", "model_bind", "model_destroy", "decode_step", "decode_step_deferred",
    "pending_wait", "pending_free", "decode_step_device", "model_synchronize", "model_stream",
    "last_error_string", "model_stats", "model_kv_export", "model_kv_import", "model_attn_out",
    "model_time_kernel", "model_kernel_time", "model_set_serial_steps", "attention_decode_noalloc", "attention_decode_noalloc_error",
    "attention_decode_noalloc_scratch_bytes", "model_trace_enable", "model_trace_read", "model_trace_disable",
    "stage_plan_solve", "model_stage_bytes", "model_set_wait_limit", "attention_decode_noalloc_status",
    "model_prefill",
)


class ModelDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("n_embd", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("weight_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
                ("max_ctx", ctypes.c_int), ("batch", ctypes.c_int), ("pending_depth", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


class Matrix(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("attn_norm", ctypes.c_void_p), ("wq", Matrix), ("wk", Matrix), ("wv", Matrix), ("wo", Matrix),
                ("ffn_norm", ctypes.c_void_p), ("w_gate", Matrix), ("w_up", Matrix), ("w_down", Matrix)]


class ModelWeights(ctypes.Structure):
    _fields_ = [("embed", Matrix), ("out_norm", ctypes.c_void_p), ("lm_head", Matrix),
                ("layers", ctypes.POINTER(LayerWeights))]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p)


class Runtime(ctypes.Structure):
    _fields_ = [("device", ctypes.c_int), ("alloc", ALLOC_FN), ("free", FREE_FN), ("alloc_ctx", ctypes.c_void_p),
                ("streams", ctypes.POINTER(ctypes.c_void_p))]


class TraceRecord(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("stage", ctypes.c_int32), ("layer", ctypes.c_int32),
                ("step", ctypes.c_int32), ("start_ns", ctypes.c_uint64), ("end_ns", ctypes.c_uint64)]


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("deferred_steps", ctypes.c_uint64), ("stage_walks", ctypes.c_uint64),
                ("boundary_crossings", ctypes.c_uint64), ("pending_drains", ctypes.c_uint64),
                ("kernel_launches", ctypes.c_uint64), ("n_stages", ctypes.c_int), ("fence", ctypes.c_int * 17),
                ("persistent", ctypes.c_int)]


_lib = None


def load(path: str = LIB_PATH):
    """Load the C-ABI library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -m layer_pipeline_staged_gb300.build)")
    L = ctypes.CDLL(path)
    vp, i, pp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "stage_plan_create": (i, [i, vp, i, pp]),
        "stage_plan_from_counts": (i, [vp, i, pp]),
        "stage_plan_destroy": (None, [vp]),
        "stage_plan_n_stages": (i, [vp]),
        "stage_plan_fence": (i, [vp, vp, i]),
        "stage_of": (i, [vp, i]),
        "model_bind": (i, [vp, ctypes.POINTER(ModelDesc), ctypes.POINTER(ModelWeights), ctypes.POINTER(Runtime), pp]),
        "model_destroy": (None, [vp]),
        "decode_step": (i, [vp, vp, vp, vp]),
        "decode_step_deferred": (i, [vp, vp, vp, pp]),
        "pending_wait": (i, [vp, vp, i]),
        "pending_free": (None, [vp]),
        "decode_step_device": (i, [vp, vp, vp, vp]),
        "model_prefill": (i, [vp, i, vp, i, i, i, vp]),
        "model_synchronize": (i, [vp]),
        "model_stream": (i, [vp, i, pp]),
        "last_error_string": (ctypes.c_char_p, []),
        "model_stats": (i, [vp, ctypes.POINTER(Stats)]),
        "model_kv_export": (i, [vp, i, i, vp, ctypes.c_size_t]),
        "model_kv_import": (i, [vp, i, i, vp, ctypes.c_size_t, i]),
        "model_attn_out": (i, [vp, i, i, vp]),
        "model_time_kernel": (i, [vp, i, i]),
        "model_set_serial_steps": (i, [vp, i]),
        "model_set_wait_limit": (i, [vp, ctypes.c_longlong]),
        "model_kernel_time": (i, [vp, i, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64)]),
        "model_trace_enable": (i, [vp, i]),
        "model_trace_read": (i, [vp, ctypes.POINTER(TraceRecord), i, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_uint64)]),
        "model_trace_disable": (i, [vp]),
        "attention_decode_noalloc": (i, [vp, vp, vp, vp, i, i, i, i, i, vp, vp]),
        "attention_decode_noalloc_error": (ctypes.c_char_p, []),
        "attention_decode_noalloc_status": (i, [vp]),
        "attention_decode_noalloc_scratch_bytes": (ctypes.c_longlong, [i, i, i, i, i]),
        "stage_plan_solve": (i, [i, i, vp, vp, vp, vp, ctypes.c_int64, vp, ctypes.POINTER(ctypes.c_int64)]),
        "model_stage_bytes": (i, [ctypes.POINTER(ModelDesc), vp, vp, ctypes.POINTER(ctypes.c_uint64),
                                  ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L
