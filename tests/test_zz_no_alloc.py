"""attention_decode_noalloc against the regular decode step's attention.

The entry point exists for callers that may not allocate device memory once
they run (a latency-bound serving loop, a program with a fixed memory pool):
its scratch is a static device array inside the library. This test checks,
through the C ABI, that two calls in a row give the same attention output as
the decode step of a bound model (read with model_attn_out), within the
tolerance the other GPU tests use. It sits in a file of its own, collected
last, and needs nothing from the other test files' state.
"""
import ctypes

import numpy as np
import pytest

import layer_pipeline_staged_gb300 as lps
import synth
from layer_pipeline_staged_gb300 import _capi
from workloads import TOL_BF16, bind, random_kv, rel_err

pytestmark = pytest.mark.gpu

CFG = synth.ModelConfig("noalloc", 93, 2, 512, 32, 8, 128, 512, 1000, "bf16", 2, 0, 0, (1,))


def _q_layer0(w, tok, pos):
    """q of layer 0 for one token at `pos`: RMSNorm of the embedding row, W_q,
    then RoPE (rotate-half pairs, angle pos * 10000^(-2i/hd))."""
    h = synth.bf16_to_f32(w["embed"][tok]).astype(np.float64)
    xn = h / np.sqrt(np.mean(h * h) + CFG.rms_eps) * w["layers"][0]["attn_norm"].astype(np.float64)
    q = (synth.bf16_to_f32(w["layers"][0]["wq"]).astype(np.float64) @ xn).reshape(CFG.q_heads, CFG.head_dim)
    half = CFG.head_dim // 2
    ang = pos * CFG.rope_theta ** (-2.0 * np.arange(half) / CFG.head_dim)
    a, b = q[:, :half].copy(), q[:, half:].copy()
    q[:, :half] = a * np.cos(ang) - b * np.sin(ang)
    q[:, half:] = a * np.sin(ang) + b * np.cos(ang)
    return q.reshape(-1).astype(np.float32)


def test_noalloc_attention_matches_decode_step():
    import torch

    P = 3000  # cached rows before the step: several chunks per (sequence, kv head)
    max_ctx = P + 1
    w = synth.make_weights(CFG)
    m = bind(CFG, w, max_ctx=max_ctx, flags=lps.LPS_FLAG_KEEP_ATTN_OUT)
    for (l, b), (k, v) in random_kv(CFG, 31, CFG.n_layers, max_ctx, P).items():
        m.kv_import(l, b, k, v, P)
    toks = synth.make_tokens(CFG, 1, seed=91)[0]
    m.decode_step(toks, P)
    ref = np.stack([m.attn_out(0, b).reshape(-1) for b in range(CFG.batch)])

    # inputs of the regular step's layer-0 attention: its cache (row P included) and q
    kv = [m.kv_export(0, b) for b in range(CFG.batch)]
    k_dev = torch.tensor(np.stack([x[0] for x in kv]).view(np.int16), device="cuda")
    v_dev = torch.tensor(np.stack([x[1] for x in kv]).view(np.int16), device="cuda")
    q_dev = torch.tensor(np.stack([_q_layer0(w, toks[b], P) for b in range(CFG.batch)]), device="cuda")
    out_dev = torch.full((CFG.batch, CFG.q_heads * CFG.head_dim), float("nan"), device="cuda")
    pos = (ctypes.c_int32 * CFG.batch)(*([P] * CFG.batch))
    L = _capi.load()
    stream = torch.cuda.current_stream().cuda_stream

    results = []
    for call in range(2):
        rc = L.attention_decode_noalloc(q_dev.data_ptr(), k_dev.data_ptr(), v_dev.data_ptr(), out_dev.data_ptr(),
                                        CFG.batch, CFG.q_heads, CFG.kv_heads, CFG.head_dim, max_ctx, pos, stream)
        assert rc == 0, L.attention_decode_noalloc_error().decode()
        torch.cuda.synchronize()
        got = out_dev.cpu().numpy()
        assert np.all(np.isfinite(got))
        err = rel_err(got, ref)
        assert np.all(err <= TOL_BF16), f"call {call}: error {err.max():.3e} x max|output|"
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
    rc = L.attention_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, nq, nkv, hd, max_ctx,
                                    pos, torch.cuda.current_stream().cuda_stream)
    assert rc == lps.LPS_EINVAL
    assert "scratch" in L.attention_decode_noalloc_error().decode()
    torch.cuda.synchronize()
