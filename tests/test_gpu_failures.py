"""Failure detection without a GPU fault: every failure here is made on the host
or by a device-side wait that is allowed to run out.

- ``pending_wait`` with a zero timeout on a step that cannot have finished
  (its stream is held behind a bounded spin) returns LPS_ETIMEDOUT and leaves
  the handle valid; a later wait returns the step's logits, bit-identical to the
  same step run eagerly (memra_engine::pp, PendingLogits: waiting is separate
  from enqueueing, and a pending step is read back intact);
- an allocator hook that fails on its k-th call, for every k of a bind, makes
  ``model_bind`` return LPS_ENOMEM and give back every allocation it made
  ("fail closed": memra_engine::pp, refuse_unsplit_if_remote);
- a device-side wait limit of one cycle makes the kernels give up: the next
  readback returns LPS_ECUDA naming the kernel that reported first, the model
  refuses further steps, and a freshly bound model on the same GPU still
  matches the oracle (the kernels drained their own copies before ending).
"""
import ctypes

import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from layer_pipeline_staged_gb300 import _capi
from workloads import assert_close, bind, desc

pytestmark = pytest.mark.gpu

TINY = synth.CONFIGS["tiny"]
# rings that wrap several times per CTA (gate/up: 54 row pairs per CTA), so a
# producer waits for slot releases; batch 1 (GEMV) and batch 2 (tensor-core GEMM)
WAITCFG = synth.ModelConfig("waitlimit", 92, 2, 2048, 16, 4, 128, 8192, 8192, "bf16", 1, 0, 0, (1,))


def test_pending_wait_times_out_then_completes():
    import torch

    w = synth.make_weights(TINY)
    toks = synth.make_tokens(TINY, 4)
    m = bind(TINY, w, max_ctx=8)
    for t in range(3):
        m.decode_step(toks[t], t)
    # hold stage 0's stream behind a bounded spin (about 0.2 s), so the step
    # enqueued next cannot have finished when it is first waited
    with torch.cuda.stream(torch.cuda.ExternalStream(m.stream(0))):
        torch.cuda._sleep(400_000_000)
    p = m.decode_step_deferred(toks[3], 3)
    with pytest.raises(lps.LpsError) as ei:
        p.wait(timeout_ms=0)
    assert ei.value.code == lps.LPS_ETIMEDOUT
    got = p.wait()              # the handle is still valid
    again = p.wait(timeout_ms=0)  # and may be waited again once drained
    p.free()
    assert np.array_equal(got, again)
    eager = m.decode_step(toks[3], 3)  # the same step (rewinding one position)
    assert np.array_equal(got, eager)
    assert m.stats()["pending_drains"] == 1


class _CountingAlloc:
    """Allocator hooks over PyTorch's caching allocator that fail on call k."""

    def __init__(self, fail_at: int | None):
        import torch

        self.torch = torch
        self.fail_at = fail_at
        self.calls = 0
        self.live = set()

        def _alloc(_ctx, nbytes):
            self.calls += 1
            if self.fail_at is not None and self.calls == self.fail_at:
                return None
            p = int(torch.cuda.caching_allocator_alloc(int(nbytes), device=0))
            self.live.add(p)
            return p

        def _free(_ctx, ptr):
            self.live.discard(int(ptr))
            torch.cuda.caching_allocator_delete(int(ptr))

        self.alloc = _capi.ALLOC_FN(_alloc)
        self.free = _capi.FREE_FN(_free)

    def runtime(self):
        rt = _capi.Runtime()
        rt.device = 0
        rt.alloc = self.alloc
        rt.free = self.free
        rt.streams = None
        return rt


def _bind_raw(cfg, w, hooks, fence):
    L = _capi.load()
    plan = lps.stage_plan_create(cfg.n_layers, cuts=list(fence[1:-1]))
    d = _capi.ModelDesc(**desc(cfg, max_ctx=16))
    ws = lps.weights_struct(w, cfg.n_layers)
    rt = hooks.runtime()
    h = ctypes.c_void_p()
    rc = L.model_bind(plan.h, ctypes.byref(d), ctypes.byref(ws), ctypes.byref(rt), ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("cfg", [TINY, TINY.replace(name="tiny_b2", batch=2)], ids=lambda c: c.name)
def test_bind_fails_closed_on_every_allocation(cfg):
    w = synth.make_weights(cfg)
    fence = (0, 1, 3, 4)  # three stages: every per-stage allocation appears
    ok = _CountingAlloc(None)
    rc, h = _bind_raw(cfg, w, ok, fence)
    assert rc == 0, _capi.load().last_error_string().decode()
    total = ok.calls
    assert total > 20 and len(ok.live) > 0
    _capi.load().model_destroy(h)
    assert not ok.live, "model_destroy left allocations behind"
    for k in range(1, total + 1):
        hooks = _CountingAlloc(k)
        rc, h = _bind_raw(cfg, w, hooks, fence)
        assert rc == lps.LPS_ENOMEM, (k, rc, _capi.load().last_error_string().decode())
        assert not h.value, k
        assert hooks.calls == k, "bind went on allocating after a failure"
        assert not hooks.live, f"failure at allocation {k} leaked {len(hooks.live)} allocations"
        assert "model_bind" in _capi.load().last_error_string().decode()


@pytest.mark.parametrize("batch,flags,kernel", [(1, lps.LPS_FLAG_PERSISTENT, "persistent stage kernel"), (1, 0, ""),
                                                (2, 0, "batch > 1")],
                         ids=["persistent", "chained", "tensor-core"])
def test_device_wait_limit_reports_the_kernel(batch, flags, kernel):
    cfg = WAITCFG.replace(batch=batch)
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, 3)
    m = bind(cfg, w, max_ctx=8, flags=flags)
    first = m.decode_step(toks[0], 0)
    m.set_wait_limit(1)
    with pytest.raises(lps.LpsError) as ei:
        m.decode_step(toks[1], 1)
    assert ei.value.code == lps.LPS_ECUDA
    msg = str(ei.value)
    assert "device-side error in" in msg and "timed out" in msg and kernel in msg, msg
    # the model fails closed from now on
    with pytest.raises(lps.LpsError) as ei:
        m.decode_step(toks[1], 1)
    assert ei.value.code == lps.LPS_ECUDA and "failed state" in str(ei.value)
    m.close()
    # the GPU is still usable: a new model computes the same first step and
    # matches the oracle on the next
    m2 = bind(cfg, w, max_ctx=8, flags=flags)
    assert np.array_equal(m2.decode_step(toks[0], 0), first)
    orc = oracle.Oracle(cfg, w, max_ctx=8)
    orc.step(toks[0], 0)
    assert_close(m2.decode_step(toks[1], 1), orc.step(toks[1], 1), cfg, "after a failed model")
    with pytest.raises(lps.LpsError):
        m2.set_wait_limit(-1)


def test_prefill_device_wait_limit_reports_the_kernel():
    """The prefill kernels' bounded waits (tcgen05 GEMM ring and accumulators,
    chunk-attention ring) run out under a 1-cycle limit: the call returns
    LPS_ECUDA naming a prefill kernel, every issued copy and MMA has landed
    before the CTAs ended, and the GPU stays usable for a new model."""
    cfg = WAITCFG
    w = synth.make_weights(cfg)
    toks = synth.make_tokens(cfg, 48)
    m = bind(cfg, w, max_ctx=64)
    first = m.prefill(toks, chunk=16)
    m.set_wait_limit(1)
    with pytest.raises(lps.LpsError) as ei:
        m.prefill(toks, chunk=16)
    assert ei.value.code == lps.LPS_ECUDA
    msg = str(ei.value)
    assert "device-side error in prefill" in msg and "timed out" in msg, msg
    with pytest.raises(lps.LpsError) as ei:
        m.prefill(toks, chunk=16)
    assert ei.value.code == lps.LPS_ECUDA and "failed state" in str(ei.value)
    m.close()
    m2 = bind(cfg, w, max_ctx=64)
    assert np.array_equal(m2.prefill(toks, chunk=16), first)
    orc = oracle.Oracle(cfg, w, max_ctx=64)
    for t in range(len(toks)):
        ref = orc.step(toks[t], t)
    assert_close(first, ref, cfg, "prefill before the failure")
    m2.close()
