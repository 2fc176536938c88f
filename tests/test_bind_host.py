"""The C ABI's argument checks on the CPU: model_bind refuses a bad descriptor,
missing weight pointers and incomplete runtime hooks before it touches the
device, and every entry point refuses a NULL handle. No device is needed (on
a machine with one, the valid descriptor binds instead of failing)."""
import ctypes

import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
from layer_pipeline_staged_gb300 import _capi
from layer_pipeline_staged_gb300 import build as lps_build
import synth
from workloads import desc

TINY = synth.CONFIGS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def built():
    lps_build.build()


@pytest.fixture(scope="module")
def tiny_w():
    return synth.make_weights(TINY)


@pytest.fixture(scope="module")
def tiny_q8_w():
    return synth.make_weights(TINY.replace(name="tiny_q8", weight_dtype="int8"))


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def _bind_raw(d: dict, w, rt=None):
    """model_bind through the C ABI with host weights; returns (rc, error text)."""
    L = lps.load()
    plan = lps.stage_plan_create(TINY.n_layers, cuts=[2])
    ws = w if isinstance(w, _capi.ModelWeights) else lps.weights_struct(w, len(w["layers"]))
    h = ctypes.c_void_p()
    rt = rt or _capi.Runtime()
    rc = L.model_bind(plan.h, ctypes.byref(_capi.ModelDesc(**d)), ctypes.byref(ws), ctypes.byref(rt), ctypes.byref(h))
    err = L.last_error_string().decode()
    if rc == lps.LPS_OK:
        L.model_destroy(h)
    return rc, err


BAD = [
    (dict(n_layers=3), "n_layers"),
    (dict(weight_dtype=2), "weight_dtype"),
    (dict(kv_dtype=1), "kv_dtype"),
    (dict(n_embd=0), "positive"),
    (dict(ffn=-4), "positive"),
    (dict(vocab=0), "positive"),
    (dict(max_ctx=0), "positive"),
    (dict(n_kv_heads=0), "positive"),
    (dict(batch=0), "batch"),
    (dict(batch=9), "batch"),
    (dict(n_q_heads=3), "multiple of n_kv_heads"),
    (dict(head_dim=96), "head_dim"),
    (dict(head_dim=256), "head_dim"),
    (dict(n_q_heads=32, n_kv_heads=2), "head_dim"),  # group 16
    (dict(n_q_heads=6, n_kv_heads=2), "head_dim"),   # group 3
    (dict(n_embd=258), "multiple of 4"),
    (dict(rms_eps=0.0), "rms_eps"),
    (dict(rms_eps=float("nan")), "rms_eps"),
    (dict(rope_theta=-1.0), "rope_theta"),
    (dict(batch=2, max_ctx=1 << 30), "2^31"),
    (dict(flags=lps.LPS_FLAG_GRAPH | lps.LPS_FLAG_PERSISTENT), "LPS_FLAG_GRAPH"),
]


@pytest.mark.parametrize("change,what", BAD, ids=[f"{next(iter(c))}={list(c.values())[0]}" for c, _ in BAD])
def test_bind_refuses_bad_descriptor_before_the_device(tiny_w, change, what):
    d = desc(TINY)
    d.update(change)
    rc, err = _bind_raw(d, tiny_w)
    assert rc == lps.LPS_EINVAL, err
    assert err.startswith("model_bind: ") and what in err, err


@pytest.mark.parametrize("hole", ["layers", "out_norm", "embed", "lm_head", "wq", "w_down", "attn_norm", "ffn_norm"])
def test_bind_refuses_missing_weights(tiny_w, hole):
    ws = lps.weights_struct(tiny_w, TINY.n_layers)
    if hole == "layers":
        ws.layers = ctypes.POINTER(_capi.LayerWeights)()
    elif hole == "out_norm":
        ws.out_norm = None
    elif hole in ("embed", "lm_head"):
        getattr(ws, hole).w = None
    elif hole in ("attn_norm", "ffn_norm"):
        setattr(ws.layers[3], hole, None)
    else:
        getattr(ws.layers[1], hole).w = None
    rc, err = _bind_raw(desc(TINY), ws)
    assert rc == lps.LPS_EINVAL, err
    want = {"layers": "missing weights", "out_norm": "missing weights", "embed": "missing weights",
            "lm_head": "missing weights", "wq": "layer 1", "w_down": "layer 1", "attn_norm": "layer 3",
            "ffn_norm": "layer 3"}[hole]
    assert want in err, err


@pytest.mark.parametrize("hole", ["wk", "w_up", "embed", "lm_head"])
def test_bind_refuses_int8_without_row_scales(tiny_q8_w, hole):
    cfg = TINY.replace(name="tiny_q8", weight_dtype="int8")
    ws = lps.weights_struct(tiny_q8_w, cfg.n_layers)
    if hole in ("embed", "lm_head"):
        getattr(ws, hole).scale = None
        want = "row scales"
    else:
        getattr(ws.layers[2], hole).scale = None
        want = "layer 2"
    rc, err = _bind_raw(desc(cfg), ws)
    assert rc == lps.LPS_EINVAL and want in err, err


def test_bind_refuses_alloc_hook_without_free(tiny_w):
    keep = _capi.ALLOC_FN(lambda ctx, n: None)
    rt = _capi.Runtime()
    rt.alloc = keep
    rc, err = _bind_raw(desc(TINY), tiny_w, rt=rt)
    assert rc == lps.LPS_EINVAL and "rt->free" in err, err


def test_bind_null_arguments(tiny_w):
    L = lps.load()
    plan = lps.stage_plan_create(TINY.n_layers, cuts=[2])
    d = _capi.ModelDesc(**desc(TINY))
    ws = lps.weights_struct(tiny_w, TINY.n_layers)
    h = ctypes.c_void_p()
    assert L.model_bind(plan.h, ctypes.byref(d), ctypes.byref(ws), None, None) == lps.LPS_EINVAL
    assert L.model_bind(None, ctypes.byref(d), ctypes.byref(ws), None, ctypes.byref(h)) == lps.LPS_EINVAL
    assert L.model_bind(plan.h, None, ctypes.byref(ws), None, ctypes.byref(h)) == lps.LPS_EINVAL
    assert L.model_bind(plan.h, ctypes.byref(d), None, None, ctypes.byref(h)) == lps.LPS_EINVAL
    assert not h.value


def test_valid_descriptor_reaches_the_device_query(tiny_w):
    """Past the argument checks the bind asks the device; with none, it fails
    closed with LPS_ECUDA and hands back no model."""
    if _has_gpu():
        pytest.skip("a device is present: the bind would succeed")
    rc, err = _bind_raw(desc(TINY), tiny_w)
    assert rc == lps.LPS_ECUDA and "cannot query device" in err, err


def test_entry_points_refuse_null_handles():
    L = lps.load()
    buf = np.zeros(64, np.int32)
    p = buf.ctypes.data
    out = ctypes.c_void_p()
    n = ctypes.c_int()
    tot, cnt = ctypes.c_double(), ctypes.c_uint64()
    stats = _capi.Stats()
    calls = {
        "decode_step": lambda: L.decode_step(None, p, p, p),
        "decode_step_deferred": lambda: L.decode_step_deferred(None, p, p, ctypes.byref(out)),
        "decode_step_device": lambda: L.decode_step_device(None, p, p, p),
        "pending_wait": lambda: L.pending_wait(None, p, 0),
        "model_prefill": lambda: L.model_prefill(None, 0, p, 4, 0, 0, p),
        "model_synchronize": lambda: L.model_synchronize(None),
        "model_stream": lambda: L.model_stream(None, 0, ctypes.byref(out)),
        "model_stats": lambda: L.model_stats(None, ctypes.byref(stats)),
        "model_kv_export": lambda: L.model_kv_export(None, 0, 0, p, 64),
        "model_kv_import": lambda: L.model_kv_import(None, 0, 0, p, 64, 1),
        "model_attn_out": lambda: L.model_attn_out(None, 0, 0, p),
        "model_set_wait_limit": lambda: L.model_set_wait_limit(None, 1000),
        "model_set_serial_steps": lambda: L.model_set_serial_steps(None, 1),
        "model_trace_enable": lambda: L.model_trace_enable(None, 16),
        "model_trace_read": lambda: L.model_trace_read(None, None, 0, ctypes.byref(n), None),
        "model_trace_disable": lambda: L.model_trace_disable(None),
        "model_time_kernel": lambda: L.model_time_kernel(None, 0, 1),
        "model_kernel_time": lambda: L.model_kernel_time(None, 0, ctypes.byref(tot), ctypes.byref(cnt)),
    }
    for name, call in calls.items():
        assert call() == lps.LPS_EINVAL, name
        assert L.last_error_string().decode().startswith(name + ":"), (name, L.last_error_string())
    # the destructors take NULL as a no-op
    L.model_destroy(None)
    L.pending_free(None)
    L.stage_plan_destroy(None)
