"""bench.py's roofline arithmetic on the host: the algorithmic bytes of one
launch of each timed kernel family, counted here from the tensors the launch
must touch, and the rule that a committed ncu traffic figure is used only
while the kernel's sources are the ones it was captured from."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_gateup_bytes_8b_bf16():
    # gate and up: two [14336 x 4096] bf16 matrices read once; the f32 hidden
    # row and RMSNorm gain in (4096 floats each); the SwiGLU row out (14336 floats)
    cfg = synth.CONFIGS["8b"]
    assert bench.kernel_bytes(cfg, "gateup", 8192) == 2 * 14336 * 4096 * 2 + 4096 * 4 + 4096 * 4 + 14336 * 4
    assert bench.kernel_bytes(cfg, "gateup", 8192) == 234_971_136


def test_gateup_bytes_int8_batch8():
    # int8: one byte per weight plus one f32 scale per packed row; 8 hidden rows in, 8 SwiGLU rows out
    cfg = synth.CONFIGS["8b_q8_b8"]
    w = 2 * 14336 * 4096 + 2 * 14336 * 4
    assert bench.kernel_bytes(cfg, "gateup", 0) == w + 8 * 4096 * 4 + 4096 * 4 + 8 * 14336 * 4


@pytest.mark.parametrize("name,pos", [("8b", 8192), ("8b_q8", 32767), ("padded", 4096), ("tiny", 0)])
def test_attention_bytes(name, pos):
    # K and V rows [0, pos] of every (sequence, kv head), bf16, plus q in and o out in f32
    cfg = synth.CONFIGS[name]
    kv = cfg.batch * cfg.kv_heads * (pos + 1) * cfg.head_dim * 2 * 2
    qo = 2 * cfg.batch * cfg.q_heads * cfg.head_dim * 4
    assert bench.kernel_bytes(cfg, "attn", pos) == kv + qo
    if name == "8b":
        assert kv == 33_558_528  # the 33.6 MB per launch at position 8192


def test_attention_bytes_grow_one_row_per_position():
    cfg = synth.CONFIGS["8b"]
    step = bench.kernel_bytes(cfg, "attn", 101) - bench.kernel_bytes(cfg, "attn", 100)
    assert step == cfg.kv_heads * cfg.head_dim * 2 * 2


def test_unknown_kernel_family_refused():
    with pytest.raises(ValueError):
        bench.kernel_bytes(synth.CONFIGS["8b"], "lm_head", 0)


def _fake_tree(tmp_path, body: bytes, recorded: str):
    csrc = tmp_path / "layer_pipeline_staged_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(body)
    (tmp_path / "profiles").mkdir()
    ent = {"kernel": "gateup", "config": "8b", "sources": ["k.cu"], "sources_sha256_16": recorded,
           "dram_bytes_per_launch": 123456}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"entries": {"gateup:8b": ent}}))


def test_traffic_used_while_sources_match(tmp_path, monkeypatch):
    body = b"__global__ void k() {}\n"
    _fake_tree(tmp_path, body, hashlib.sha256(body).hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("gateup", "8b") == 123456
    assert bench.kernel_traffic("gateup", "1b") is None  # no entry for that workload


def test_traffic_dropped_once_sources_change(tmp_path, monkeypatch):
    _fake_tree(tmp_path, b"__global__ void k() { /* changed */ }\n",
               hashlib.sha256(b"__global__ void k() {}\n").hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("gateup", "8b") is None


def test_traffic_missing_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("gateup", "8b") is None
