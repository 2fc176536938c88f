"""attention_decode_noalloc against the oracle's attention, head by head.

The entry point exists for callers that may not allocate device memory once
they run (a latency-bound serving loop, a program with a fixed memory pool):
its scratch is a static device array inside the library. These tests call it
through the C ABI on seeded q and caches, with a different position for every
sequence (so the sequences have different chunk counts in one launch), at head
dim 64 with one q head per kv head and at head dim 128 with eight; every
(sequence, q head) output must match the oracle's attention of that head
within the tolerance the other GPU tests use, and two calls in a row must give
the same bits. The status query must then report no device-side failure. The
file is collected last and needs nothing from the other test files' state.
"""
import ctypes

import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import oracle
import synth
from layer_pipeline_staged_gb300 import _capi
from workloads import TOL_BF16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hd,group,nkv", [(64, 1, 6), (128, 8, 2)])
def test_noalloc_attention_matches_oracle(hd, group, nkv):
    import torch

    B, nq = 3, nkv * group
    pos = np.array([2999, 701, 0], np.int32)  # several chunks, a few, and a single row
    max_ctx = 3001
    seed = 95
    # caches: uniform bf16 in [-1, 1); q: N(0, 3) so the scores spread over a few units
    k = synth.uniform_bf16(seed, 0, (B, nkv, max_ctx, hd))
    v = synth.uniform_bf16(seed, 1, (B, nkv, max_ctx, hd))
    q = synth.normal_f32(seed, 2, (B, nq * hd), stddev=3.0)
    ref = np.empty((B, nq, hd), np.float64)
    for b in range(B):
        for h in range(nq):
            g = h // group
            ref[b, h] = oracle.attend_head(q[b, h * hd:(h + 1) * hd].astype(np.float64), k[b, g], v[b, g], int(pos[b]))

    k_dev = torch.tensor(k.view(np.int16), device="cuda")
    v_dev = torch.tensor(v.view(np.int16), device="cuda")
    q_dev = torch.tensor(q, device="cuda")
    out_dev = torch.full((B, nq * hd), float("nan"), device="cuda")
    cpos = (ctypes.c_int32 * B)(*pos.tolist())
    L = _capi.load()
    stream = torch.cuda.current_stream().cuda_stream

    results = []
    for call in range(2):
        rc = L.attention_decode_noalloc(q_dev.data_ptr(), k_dev.data_ptr(), v_dev.data_ptr(), out_dev.data_ptr(), B,
                                        nq, nkv, hd, max_ctx, cpos, stream)
        assert rc == 0, L.attention_decode_noalloc_error().decode()
        assert L.attention_decode_noalloc_status(stream) == 0, L.attention_decode_noalloc_error().decode()
        got = out_dev.cpu().numpy().reshape(B, nq, hd).astype(np.float64)
        assert np.all(np.isfinite(got))
        err = np.max(np.abs(got - ref), axis=2) / np.max(np.abs(ref), axis=2)
        assert np.all(err <= TOL_BF16), f"call {call}: error {err.max():.3e} x max|output| (head {np.argmax(err)})"
        assert np.array_equal(got[2], np.broadcast_to(synth.bf16_to_f32(v[2, np.arange(nq) // group, 0]), (nq, hd)))
        results.append(got)
        out_dev.fill_(float("nan"))
    assert np.array_equal(results[0], results[1])  # the shared scratch starts clean on every call


def test_noalloc_refuses_oversized_calls():
    """A call whose partials do not fit the static scratch is refused before
    any launch. The buffers are real and sized for the call, and the library's
    own requirement for these shapes is checked to exceed the scratch first, so
    the call is never made with shapes the entry point would accept."""
    import torch

    B, nq, nkv, hd, max_ctx, P = 8, 8192, 1024, 128, 2, 1
    L = _capi.load()
    need = L.attention_decode_noalloc_scratch_bytes(B, nq, nkv, hd, P)
    assert need > lps.LPS_NOALLOC_SCRATCH_BYTES, f"shapes need only {need} bytes: not an oversized call"
    q = torch.zeros(B, nq * hd, device="cuda")
    out = torch.zeros(B, nq * hd, device="cuda")
    k = torch.zeros(B * nkv * max_ctx * hd, dtype=torch.int16, device="cuda")
    v = torch.zeros(B * nkv * max_ctx * hd, dtype=torch.int16, device="cuda")
    pos = (ctypes.c_int32 * B)(*([P] * B))
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.attention_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, nq, nkv, hd, max_ctx,
                                    pos, stream)
    assert rc == lps.LPS_EINVAL
    assert "scratch" in L.attention_decode_noalloc_error().decode()
    # cache rows past 32-bit coordinates are refused before anything is read
    rc = L.attention_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), 8, 64, 8, hd,
                                    1 << 25, pos, stream)
    assert rc == lps.LPS_EINVAL
    assert "2^31" in L.attention_decode_noalloc_error().decode()
    assert L.attention_decode_noalloc_status(stream) == 0
    torch.cuda.synchronize()
