"""Benchmark of the layer-staged eager decode step on GB300.

One step = one decode step of the whole trunk (embed, every layer's
RMSNorm+QKV+RoPE+KV append, split-K attention, o-proj+residual,
RMSNorm+gate/up+SwiGLU, down+residual, the boundary hand-overs, the final
norm + LM head) for the batch, teacher forced.

Default workload: the 8B-shape decoder (32 layers, n_embd 4096, 32 q / 8 kv
heads, head_dim 128, ffn 14336, vocab 128256), bf16 weights and KV cache,
batch 1, 4 stages (cuts 8, 16, 24), context 8192, 256 decode steps, deferred
logits readback. Weights are seeded N(0, 0.02) (synthetic: no checkpoint);
the context's cache rows are written by the chunked prefill of a seeded prompt
(model_prefill, timed and reported as "prefill"; batch > 1 workloads fill them
synthetically, as their values do not change the step time); the weights (15 GB) are far larger than L2, so every step streams
them from HBM.

Prints one JSON line. ``--impl reference`` times the CPU oracle on the same
workload instead (host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s and achieved HBM GB/s (% of 8 TB/s) per step, 1×GB300"
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="8b")
    ap.add_argument("--ctx", type=int, default=None, help="context length before the timed steps")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fill", default="auto", choices=["auto", "prefill", "synthetic", "decode"],
                    help="how the context rows before the timed steps are written: model_prefill (chunked "
                         "prefill through the stages, timed and reported), synthetic rows, or decode steps; "
                         "auto = prefill where the model takes it (batch 1), else synthetic")
    ap.add_argument("--serial", action="store_true", help="no overlap between consecutive steps' stages")
    ap.add_argument("--stages", type=int, default=0,
                    help="even split into this many stages instead of the workload's own cuts (0 = the workload's)")
    ap.add_argument("--verify", type=int, default=0,
                    help="speculative-verify rows: each step verifies this many consecutive positions of one "
                         "sequence (LPS_FLAG_VERIFY, batch = rows); 0 = ordinary decode")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: keep the first N layers (a smaller case for ncu); not a bench number")
    ap.add_argument("--persistent", action="store_true",
                    help="batch 1: the persistent stage kernel (one launch per stage and step) instead of "
                         "the default chained per-projection kernels")
    ap.add_argument("--graph", action="store_true",
                    help="every step replays as one CUDA graph (LPS_FLAG_GRAPH)")
    ap.add_argument("--repeats", type=int, default=None,
                    help="extra timed passes of the same K steps for a median (default: about 2 s worth)")
    return ap.parse_args()


def workload_name(cfg, ctx, steps, readback="deferred"):
    return (f"{cfg.name}-shape decoder: {cfg.n_layers} layers, n_embd {cfg.n_embd}, {cfg.q_heads} q / "
            f"{cfg.kv_heads} kv heads, head_dim {cfg.head_dim}, ffn {cfg.ffn}, vocab {cfg.vocab}, "
            f"{cfg.weight_dtype} weights, bf16 KV, batch {cfg.batch}, context {ctx}, {steps} decode steps, "
            f"{len(cfg.fence) - 1} stages (cuts {','.join(map(str, cfg.cuts))}), {readback} readback")


def resolve_fill(fill: str, batch: int, verify_rows: int) -> str:
    """How the context rows before the timed steps are written (auto: the chunked prefill
    where the model takes it, i.e. batch 1 without verify rows, else synthetic rows)."""
    if fill == "auto":
        return "prefill" if (batch == 1 and not verify_rows) else "synthetic"
    return fill


def arm_config(cfg, ctx: int, steps: int, n_stages: int, n_replicas: int, fill: str, overlap: bool) -> dict:
    """The line's `config`, the same for the GPU arm and the reference arm."""
    return {"workload": workload_name(cfg, ctx, steps),
            "l2": "inputs larger than L2 (every step streams all weights from HBM)",
            "cache_fill": fill, "steps_overlap": overlap,
            "parallelism": f"{n_stages} stages on one device"
            + (f", {n_replicas} independent replicas" if n_replicas > 1 else "")}


def dtype_of(cfg):
    return "int8" if cfg.weight_dtype == "int8" else "bf16"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


KERNEL_NAMES = {
    "gateup": ("RMSNorm + gate/up GEMV + SwiGLU" + " per layer"),
    "attn": "split-K GQA decode attention per layer",
    "stage": "persistent stage kernel (every layer of a stage, one launch per stage and step)",
}


def kernel_bytes(cfg, kind: str, pos: int) -> int:
    """Algorithmic HBM bytes of one launch of a kernel family at decode position pos."""
    el = 1 if cfg.weight_dtype == "int8" else 2
    B, E = cfg.batch, cfg.n_embd
    if kind == "gateup":
        b = 2 * cfg.ffn * E * el + (2 * cfg.ffn * 4 if el == 1 else 0)  # weights (and row scales)
        return b + B * E * 4 + E * 4 + B * cfg.ffn * 4  # h and gain in, SwiGLU activations out
    if kind == "attn":
        qw = cfg.q_heads * cfg.head_dim
        kv = B * cfg.kv_heads * cfg.head_dim * 2 * 2 * (pos + 1)  # K and V rows [0, pos], bf16
        return kv + 2 * B * qw * 4  # q in, attention output out
    raise ValueError(kind)


def max_over_ranks(values, dist=None, device: str = "cuda") -> list:
    """Each value's maximum over all ranks (a multi-rank job takes as long as its slowest
    rank); the values themselves with one rank."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rate(world: int, rows: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: the rows every rank processed in the slowest rank's time."""
    return world * rows * steps / seconds


def kernel_traffic(kind: str, cfg_name: str):
    """DRAM bytes per launch of a kernel family on a workload, from the committed ncu
    summary, if the kernel's sources still match the ones it was captured with."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        ent = json.load(open(path))["entries"].get(f"{kind}:{cfg_name}")
    except Exception:
        return None
    if not ent:
        return None
    h = hashlib.sha256()
    for f in ent["sources"]:
        h.update(open(os.path.join(ROOT, "layer_pipeline_staged_gb300", "csrc", f), "rb").read())
    if h.hexdigest()[:16] != ent.get("sources_sha256_16"):
        return None
    return ent.get("dram_bytes_per_launch")


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            time.sleep(0.25)
            self.p.terminate()
            try:
                self.out = self.p.communicate(timeout=5)[0]
            except Exception:
                self.p.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append(parts)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_baseline(cfg, w, ctx: int, budget_s: float):
    """The oracle as it stands, on this host's cores, at the workload's context
    (cache filled synthetically: contents do not change the time)."""
    import oracle
    import synth
    orc = oracle.Oracle(cfg, w, max_ctx=ctx + 64)
    zeros = np.zeros((cfg.kv_heads, ctx + 64, cfg.head_dim), np.uint16)
    for l in range(cfg.n_layers):
        for b in range(cfg.batch):
            orc.kv_import(l, b, zeros, zeros, ctx)
    toks = synth.make_tokens(cfg, 64, seed=cfg.seed_t + 17)
    n, t0 = 0, time.perf_counter()
    while n < 64:
        orc.step(toks[n], ctx + n)
        n += 1
        if time.perf_counter() - t0 >= budget_s and n >= 2:
            break
    dt = time.perf_counter() - t0
    threads = orc.L.orc_get_threads()
    orc.close()
    return {"value": cfg.batch * n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} decode steps at positions {ctx}..{ctx + n - 1} (batch {cfg.batch}) of the same workload, "
                      f"cache filled synthetically; {dt:.1f} s of CPU work"}


def run_reference(args, cfg, ctx):
    """The reference arm: the CPU oracle on the same workload, bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    t_gen = time.perf_counter()
    w = synth.make_weights(cfg)
    gen_s = time.perf_counter() - t_gen
    import oracle
    orc = oracle.Oracle(cfg, w, max_ctx=ctx + args.steps + args.warmup + 2)
    zeros = np.zeros((cfg.kv_heads, ctx + args.steps + args.warmup + 2, cfg.head_dim), np.uint16)
    for l in range(cfg.n_layers):
        for b in range(cfg.batch):
            orc.kv_import(l, b, zeros, zeros, ctx - args.warmup)
    toks = synth.make_tokens(cfg, args.steps + args.warmup, seed=cfg.seed_t + 17)
    for i in range(min(args.warmup, 1)):
        orc.step(toks[i], ctx - args.warmup + i)
    # bounded sample: at most ~60 s of oracle steps, each one full step of the workload
    n, t0 = 0, time.perf_counter()
    pos0 = ctx - args.warmup + min(args.warmup, 1)
    while n < args.steps:
        orc.step(toks[min(args.warmup, 1) + n], pos0 + n)
        n += 1
        if time.perf_counter() - t0 > 60.0 and n >= 2:
            break
    dt = time.perf_counter() - t0
    v = cfg.batch * n / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(cfg), "data": "synthetic",
            "config": arm_config(cfg, ctx, args.steps, len(cfg.fence) - 1, args.gpus,
                                 resolve_fill(args.fill, cfg.batch, args.verify), not args.serial),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": orc.L.orc_get_threads(), "kind": "oracle",
                             "sample": f"{n} of {args.steps} decode steps at positions {pos0}..{pos0 + n - 1}; "
                                       f"the oracle's cache rows before them are zeros (their values do not "
                                       f"change a step's time; weights drawn in {gen_s:.0f} s, untimed)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    import synth
    cfg = synth.CONFIGS[args.config]
    if args.layers:
        n = min(len(cfg.fence) - 1, args.layers)
        cfg = cfg.replace(n_layers=args.layers, cuts=tuple(s * args.layers // n for s in range(1, n)))
    if args.stages:
        n = args.stages
        cfg = cfg.replace(name=f"{cfg.name}_s{n}", cuts=tuple(s * cfg.n_layers // n for s in range(1, n)))
    ctx = args.ctx if args.ctx is not None else cfg.ctx
    M = args.verify  # verify rows per step (one sequence), 0 = ordinary decode
    if M:
        if args.impl == "reference" or os.environ.get("WORLD_SIZE", "1") != "1":
            raise SystemExit("--verify runs the GPU arm on one GPU only")
        cfg = cfg.replace(name=f"{cfg.name}_verify{M}", batch=M)
    if args.impl == "reference":
        run_reference(args, cfg, ctx)
        return

    import torch
    import layer_pipeline_staged_gb300 as lps
    from layer_pipeline_staged_gb300 import build as lps_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
    torch.cuda.set_device(local)
    lps_build.build()

    K, W = args.steps, args.warmup
    adv = M or 1  # positions a step advances
    max_ctx = ctx + K * adv
    w = synth.make_weights(cfg)
    desc = dict(n_layers=cfg.n_layers, n_embd=cfg.n_embd, n_q_heads=cfg.q_heads, n_kv_heads=cfg.kv_heads,
                head_dim=cfg.head_dim, ffn=cfg.ffn, vocab=cfg.vocab,
                weight_dtype=1 if cfg.weight_dtype == "int8" else 0, kv_dtype=0, max_ctx=max_ctx,
                batch=cfg.batch, pending_depth=4, rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps,
                flags=(lps.LPS_FLAG_SERIAL_STEPS if args.serial else 0) | (lps.LPS_FLAG_VERIFY if M else 0)
                | (lps.LPS_FLAG_PERSISTENT if args.persistent else 0) | (lps.LPS_FLAG_GRAPH if args.graph else 0))
    plan = lps.stage_plan_create(cfg.n_layers, cuts=list(cfg.cuts))
    model = lps.model_bind(plan, desc, w, device=local)
    B, V = cfg.batch, cfg.vocab
    toks = synth.make_tokens(cfg, W + K)
    start = ctx - W * adv
    seqs = 1 if M else B  # sequences with a cache of their own
    # context rows [0, start): the chunked prefill of a seeded prompt, synthetic
    # cache contents, or teacher-forced decode steps
    fill = resolve_fill(args.fill, B, M)
    prefill_info = None
    if fill == "prefill" and start > 0:
        ptoks = synth.make_tokens(cfg, start, seed=cfg.seed_t + 9)
        model.prefill(ptoks[:min(start, 128)], logits=False)  # allocates the prefill buffers (untimed)
        pf_s = []
        for _ in range(2):
            t0 = time.perf_counter()
            model.prefill(ptoks, logits=True)
            pf_s.append(time.perf_counter() - t0)
        pf = min(pf_s)
        layer_params = (cfg.n_embd * (cfg.q_heads + 2 * cfg.kv_heads) * cfg.head_dim
                        + cfg.q_heads * cfg.head_dim * cfg.n_embd + 3 * cfg.n_embd * cfg.ffn)
        flops = 2.0 * start * layer_params * cfg.n_layers
        prefill_info = {"tokens": start, "chunk": 128, "seconds": pf, "tokens_per_s": start / pf,
                        "projection_tflops": flops / pf / 1e12,
                        "how": "model_prefill of the seeded prompt (positions 0..ctx-1, chunks of 128 through "
                               "the stages), host wall time of the synchronous call, best of 2; "
                               "projection_tflops counts 2 x tokens x projection weights (attention excluded)"}
    elif fill == "synthetic" and start > 0:
        for l in range(cfg.n_layers):
            for b in range(seqs):
                k = synth.uniform_bf16(cfg.seed_t + 5, 2 * (l * B + b), (cfg.kv_heads, max_ctx, cfg.head_dim))
                v = synth.uniform_bf16(cfg.seed_t + 5, 2 * (l * B + b) + 1, (cfg.kv_heads, max_ctx, cfg.head_dim))
                model.kv_import(l, b, k, v, start)
    elif start > 0:
        ftoks = synth.make_tokens(cfg, start, seed=cfg.seed_t + 9)
        tdev = torch.tensor(ftoks, dtype=torch.int32, device="cuda")
        scratch = torch.empty((B, V), dtype=torch.float32, device="cuda")
        for t in range(0, start, adv):
            model.decode_step_device(tdev[t].data_ptr(), t, scratch.data_ptr())
        model.synchronize()

    persistent = bool(model.stats()["persistent"])
    tok_dev = torch.tensor(toks, dtype=torch.int32, device="cuda")
    logits_dev = torch.empty((B, V), dtype=torch.float32, device="cuda")
    s_first = torch.cuda.ExternalStream(model.stream(0))
    s_last = torch.cuda.ExternalStream(model.stream(plan.n_stages - 1))

    def device_pass(first_pos):
        for i in range(K):
            model.decode_step_device(tok_dev[W + i].data_ptr(), first_pos + i * adv, logits_dev.data_ptr())

    # warm-up steps at positions start .. ctx-1
    for i in range(W):
        model.decode_step_device(tok_dev[i].data_ptr(), start + i * adv, logits_dev.data_ptr())
    model.synchronize()

    def barrier():
        if dist:
            dist.barrier()

    # ---- timed region: inputs resident in HBM, K steps at positions ctx .. ctx+K-1
    launches0 = model.stats()["kernel_launches"]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        torch.cuda.synchronize()
        model.synchronize()
        ev0.record(s_first)
        device_pass(ctx)
        ev1.record(s_last)
        ev1.synchronize()
        torch.cuda.synchronize()
        barrier()
        elapsed_ms = ev0.elapsed_time(ev1)
        launches = model.stats()["kernel_launches"] - launches0

        # ---- e2e: the public API with host buffers (tokens in, logits out), deferred pipelined
        depth = 4
        host_logits = np.empty((B, V), np.float32)
        barrier()
        model.synchronize()
        t0 = time.perf_counter()
        pend = []
        for i in range(K):
            pend.append(model.decode_step_deferred(toks[W + i], ctx + i * adv))
            if len(pend) == depth:
                p = pend.pop(0)
                p.wait(out=host_logits)
                p.free()
        for p in pend:
            p.wait(out=host_logits)
            p.free()
        e2e_s = time.perf_counter() - t0
        barrier()

        # ---- repeats: the same K device-resident steps again (positions ctx .. ctx+K-1
        # rewritten with the same rows), each pass timed alone, for a median per-step time
        reps = args.repeats if args.repeats is not None else max(3, min(30, int(2000.0 / max(elapsed_ms, 1e-3))))
        rep_ms = []
        for _ in range(reps):
            model.synchronize()
            ev0.record(s_first)
            device_pass(ctx)
            ev1.record(s_last)
            ev1.synchronize()
            rep_ms.append(ev0.elapsed_time(ev1) / K)

        # ---- the dominant kernel timed live with CUDA events around each launch on its
        # stream (same steps again). Persistent path: the stage kernel, whose launches
        # together carry every byte of the step. Chained path: the kernel family with the
        # most bytes, stages serialized so that no other stage's kernels run beside it
        # (verify rows: one causal chunk-attention launch, with its merge, per layer).
        if persistent:
            dom = "stage"
            model.time_kernel(dom, True)
            device_pass(ctx)
            dom_ms, dom_n = model.kernel_time(dom)
            model.time_kernel(dom, False)
            pass_bytes = sum(cfg.step_bytes(ctx + i) for i in range(K))
            per_launch = {dom: pass_bytes / max(dom_n, 1)}
            per_step = {dom: pass_bytes / K}
        else:
            pos_mid = ctx + (K // 2) * adv
            per_launch = {k: kernel_bytes(cfg, k, pos_mid) for k in ("gateup", "attn")}
            if M:
                # verify rows: one causal chunk-attention launch reads the sequence's
                # rows [0, pos + M) once for all M rows
                qw = cfg.q_heads * cfg.head_dim
                per_launch["attn"] = kernel_bytes(cfg.replace(batch=1), "attn", pos_mid + M - 1) + 2 * (M - 1) * qw * 4
            per_step = {k: per_launch[k] * cfg.n_layers for k in per_launch}
            dom = max(per_step, key=per_step.get)
            if plan.n_stages > 1:
                model.set_serial_steps(True)
            model.time_kernel(dom, True)
            device_pass(ctx)
            dom_ms, dom_n = model.kernel_time(dom)
            model.time_kernel(dom, False)
            if plan.n_stages > 1:
                model.set_serial_steps(args.serial)

    elapsed_ms, e2e_s = max_over_ranks([elapsed_ms, e2e_s], dist)
    n = world
    tok_s = job_rate(n, B, K, elapsed_ms / 1e3)
    if M:
        # weights once per step; the one chunk-attention launch per layer reads the
        # sequence's rows [0, pos + M) once for all M rows; M rows written, M logits
        one = cfg.replace(batch=1)
        row = cfg.n_layers * 2 * cfg.kv_heads * cfg.head_dim * 2
        step_bytes = [one.step_bytes(ctx + i * M + M - 1) + (M - 1) * (row + cfg.vocab * 4) for i in range(K)]
    else:
        step_bytes = [cfg.step_bytes(ctx + i) for i in range(K)]
    hbm_gbs = sum(step_bytes) / (elapsed_ms / 1e3) / 1e9
    peaks, peak_src = measured_peaks()
    dom_bytes = per_launch[dom]
    dom_avg_s = dom_ms / 1e3 / max(dom_n, 1)
    # (graph steps run no per-kernel timers: no live launch time then)
    achieved = dom_bytes / dom_avg_s / 1e9 if dom_n else None
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, w, ctx, args.cpu_seconds)
    clocks = clk.summary()
    line = {
        "metric": METRIC if not M else f"speculative-verify tokens/s ({M} consecutive positions of one sequence "
                                          "per step) and achieved HBM GB/s, 1xGB300",
        "value": tok_s, "unit": "tokens/s", "n_gpus": n, "steps": K, "warmup": W,
        "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(cfg), "data": "synthetic",
        "config": arm_config(cfg, ctx, K, plan.n_stages, n, fill, not args.serial),
        "hbm_gbs": hbm_gbs, "hbm_frac_of_8tbs": hbm_gbs / NOMINAL_HBM_GBS,
        "hbm_frac_of_measured": hbm_gbs / peaks["hbm_gbs"],
        "bytes_per_step": sum(step_bytes) / K,
        "value_arm": "decode_step_device: token ids and logits resident in HBM, K steps enqueued back to back "
                     "(no host copies; the deferred host readback is timed in e2e)",
        "path": ("persistent stage kernel" if persistent else "chained per-projection kernels")
                + (", one CUDA graph per step" if args.graph else ""),
        "repeats": {"passes": len(rep_ms), "steps_per_pass": K, "ms_per_step_median": statistics.median(rep_ms),
                    "ms_per_step_min": min(rep_ms), "ms_per_step_max": max(rep_ms),
                    "tokens_per_s_median": job_rate(world, B, 1, statistics.median(rep_ms) / 1e3)},
        "roofline": {"kernel": KERNEL_NAMES[dom] + f" ({100 * per_step[dom] / (sum(step_bytes) / K):.0f}% "
                               "of step bytes; launches timed live" + ("" if persistent else
                                                                         ", stages serialized") + ")",
                     "bound": "hbm",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"] if achieved else None,
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_us": dom_avg_s * 1e6,
                     "launches_timed": dom_n, "traffic": kernel_traffic(dom, cfg.name)},
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(n, B, K, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": B * 8,
                "d2h_bytes_per_step": B * V * 4,
                "how": "decode_step_deferred + pending_wait with host token ids and host logits, 4 steps in flight"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if prefill_info:
        line["prefill"] = prefill_info
    if rank == 0:
        print(json.dumps(line), flush=True)
    model.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
