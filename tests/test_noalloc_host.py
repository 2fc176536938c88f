"""The allocation-free attention entry point's argument checks on the CPU:
every refusal is decided from the arguments alone, before the device is
asked for anything. The buffer addresses passed here are never dereferenced
(each call is refused first), so the test runs only where there is no device:
on a GPU machine the same refusals are covered with real buffers by the
device tests of this entry point."""
import ctypes

import pytest

import layer_pipeline_staged_gb300 as lps
from layer_pipeline_staged_gb300 import _capi
from layer_pipeline_staged_gb300 import build as lps_build


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


pytestmark = pytest.mark.skipif(_has_gpu(), reason="addresses here are placeholders: CPU-only test")

# placeholder device addresses, 16-byte aligned (never read: every call below is refused)
Q, K, V, OUT = 0x10000, 0x20000, 0x30000, 0x40000


@pytest.fixture(scope="module", autouse=True)
def built():
    lps_build.build()


def _call(q=Q, k=K, v=V, out=OUT, batch=1, nq=32, nkv=8, hd=128, max_ctx=64, pos=(5,)):
    L = _capi.load()
    pos_arr = (ctypes.c_int32 * max(len(pos), 1))(*pos)
    rc = L.attention_decode_noalloc(q, k, v, out, batch, nq, nkv, hd, max_ctx, pos_arr, None)
    return rc, L.attention_decode_noalloc_error().decode()


CASES = [
    (dict(q=None), "required"),
    (dict(k=None), "required"),
    (dict(out=None), "required"),
    (dict(batch=0), "batch"),
    (dict(batch=9, pos=(5,) * 9), "batch"),
    (dict(nkv=0), "head_dim"),
    (dict(nq=12, nkv=8), "head_dim"),            # not a multiple
    (dict(nq=48, nkv=8), "head_dim"),            # group 6
    (dict(nq=32, nkv=2), "head_dim"),            # group 16
    (dict(hd=96), "head_dim"),
    (dict(max_ctx=0, pos=(0,)), "max_ctx"),
    (dict(pos=(-1,)), "pos"),
    (dict(pos=(64,)), "pos"),                    # pos == max_ctx
    (dict(batch=2, pos=(3, 70)), "pos"),         # the second sequence
    (dict(k=K + 8), "16-byte"),
    (dict(v=V + 2), "16-byte"),
    (dict(batch=8, nq=64, nkv=8, max_ctx=1 << 25, pos=(1,) * 8), "2^31"),
]


@pytest.mark.parametrize("kw,what", CASES, ids=[f"{k}={v}" for kw, _ in CASES for k, v in [next(iter(kw.items()))]])
def test_noalloc_refuses_before_the_device(kw, what):
    rc, err = _call(**kw)
    assert rc == lps.LPS_EINVAL, err
    assert what in err, err


def test_scratch_query_refuses_bad_shapes():
    L = _capi.load()
    for args in [(0, 32, 8, 128, 10), (9, 32, 8, 128, 10), (1, 32, 0, 128, 10), (1, 12, 8, 128, 10),
                 (1, 32, 8, 96, 10), (1, 32, 8, 128, -1)]:
        assert L.attention_decode_noalloc_scratch_bytes(*args) == -1, args


def test_valid_call_stops_at_the_device():
    """Past the argument checks the call asks for the current device; with
    none it fails closed (LPS_ECUDA) and launches nothing."""
    rc, err = _call()
    assert rc == lps.LPS_ECUDA, err
