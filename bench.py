#!/usr/bin/env python
"""Throughput of the Llama ubatch forward on one GB300 (or N independent replicas).

Workload (default): the 8B-shape Llama with Q4_0 linear layers and Q8_0 embedding / head
(vocab 128256, d 4096, 32 layers, 32/8 heads, head_dim 128, FFN 14336, RoPE theta 5e5, n_ctx
8192), seeded synthetic weights and a uniform-random 2048-token prompt. One step = clear the
cache, prefill the prompt in ubatches of 512 tokens, then 256 greedy decode steps on the device.

Reported: decode tokens/s (value), prefill tokens/s, the roofline of the dominant kernel (the
weight-streaming GEMV, against measured HBM bandwidth) and of the prefill matmuls (against the
measured bf16 tensor peak), the end-to-end rate through the C ABI with host buffers, and the
CPU oracle timed on a bounded sample on this host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lcx|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the persistent
# decode step over its algorithmic bytes, from one ncu capture of the current kernel on the 8B
# shape cut to 4 layers (1057.9 MB read + 18.1 MB written against 1057.4 MB of stored weights and
# attended K/V): the step's traffic grows with the layers and cells it processes, so the full
# launch's traffic is this ratio times its algorithmic bytes.
STEP_NCU_TRAFFIC_RATIO = (1057.873e6 + 18.055e6) / 1057.4e6


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return j["hbm_gbs"], j["bf16_tflops"], j.get("bf16_tflops_sustained", j["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.th:
            self.th.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------- workload
def workload_args(a):
    import dataclasses

    import synth
    cfg = synth.CONFIGS[a.config]
    if a.layers:   # a shallower model of the same shape (the first layers of the same draws), for profiling
        cfg = dataclasses.replace(cfg, n_layer=a.layers)
    return cfg, a.prompt, a.decode_steps, a.n_ubatch


def workload_config(a, cfg, n_prompt, n_dec, n_ub, world):
    """The `config` of the JSON line, the same for both arms."""
    return {"workload": f"{cfg.name}: {n_prompt}-token prompt in ubatches of {n_ub}, then {n_dec} greedy "
                        f"decode steps", "n_ctx": a.n_ctx or cfg.n_ctx, "n_ubatch": n_ub,
            "l2": "inputs larger than L2 (4.5 GB of weights streamed per decode step)",
            "parallelism": f"replicas x{world}", **({"layers": cfg.n_layer} if a.layers else {})}


def linear_type(cfg):
    return {2: "Q4_0", 8: "Q8_0"}.get(cfg.t_linear, str(cfg.t_linear))


def max_over_ranks(values, device, world):
    """Element-wise maximum of the ranks' values (the slowest replica's times) when world > 1;
    the values themselves otherwise."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def decode_bytes_per_step(cfg, host, pos0, n_steps):
    """Algorithmic HBM bytes of the decode steps: all weights as stored (the embedding row only)
    plus the K/V of every attended cell."""
    w = host.output.nbytes + host.output_norm.nbytes
    for L in host.layers:
        w += sum(v.nbytes for v in L.values())
    emb_row = host.tok_embd.shape[1]
    kv_cell = cfg.n_layer * cfg.n_head_kv * cfg.head_dim * 2 * 2
    cells = sum(pos0 + i + 1 for i in range(n_steps))
    return n_steps * (w + emb_row) + kv_cell * cells


def prefill_flops(cfg, n_prompt):
    d, hd, H, KV, F, L, V = cfg.n_embd, cfg.head_dim, cfg.n_head, cfg.n_head_kv, cfg.n_ff, cfg.n_layer, cfg.n_vocab
    lin = (H * hd + 2 * KV * hd) * d + d * H * hd + 3 * F * d
    att = 4 * H * hd * sum(t + 1 for t in range(n_prompt)) * L
    return 2 * n_prompt * lin * L + att + 2 * V * d


def cpu_baseline(host, cfg, n_prompt=4, n_decode=2):
    """The oracle as it stands, on this host's cores, over a bounded sample."""
    import oracle
    n = oracle.set_threads()
    om = oracle.Model(host)
    octx = oracle.Context(om, cfg.n_ctx, 1, 512)
    prompt = np.asarray(host_prompt_cache.get("p"), dtype=np.int32)[:n_prompt]
    t0 = time.perf_counter()
    rc, _, am = octx.decode(prompt)
    t1 = time.perf_counter()
    tok = int(am[-1])
    for _ in range(n_decode):
        rc, _, am = octx.decode([tok])
        tok = int(am[0])
    t2 = time.perf_counter()
    return {"value": n_decode / (t2 - t1), "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{cfg.name} model, fp64 oracle: {n_prompt}-token prompt then {n_decode} decode steps "
                      f"(decode rate; prefill {n_prompt / (t1 - t0):.3f} tokens/s)",
            "prefill_tokens_per_s": n_prompt / (t1 - t0)}


host_prompt_cache = {}

SAMPLER_CHAIN = dict(top_k=40, top_p=0.95, min_p=0.05, temp=0.8)


PHASES = ("QKV", "attention", "O", "gate/up", "down")


def step_timeline(ctx, prompt, am_host, cfg, n_tok):
    """Per-phase timeline of the persistent decode step over n_tok greedy tokens after the
    prompt, from the in-kernel %globaltimer trace (lcx_set_profiling(ctx, 2)): per phase kind the
    mean span (first CTA in -> last CTA done), set-up (first CTA in -> last CTA done staging its
    input, or with its attention partial) and the gap to the next phase (next phase's first CTA in
    -> this phase's last CTA done; negative when they overlap), in microseconds."""
    import torch
    L = cfg.n_layer
    per = 5 * L + 2
    n_tok = max(1, min(n_tok, 8192 // per))
    ctx.kv_clear()
    assert ctx.decode(prompt, argmax_out=am_host) == 0
    gen = torch.zeros(n_tok, dtype=torch.int32, device="cuda")
    assert ctx.set_profiling(2) == 0
    assert ctx.decode_greedy(0, int(am_host[0]), n_tok, gen) == 0
    tr = ctx.trace().astype(np.float64)
    ctx.set_profiling(False)
    n = tr.shape[0] // per
    tr = tr[: n * per].reshape(n, per, 4)
    seq = tr[:, 1:1 + 5 * L]                                # [token][phase of the step][4]
    gap = np.concatenate([seq[:, 1:, 0] - seq[:, :-1, 3], tr[:, -1:, 0] - seq[:, -1:, 3]], axis=1)
    lay = seq.reshape(n, L, 5, 4)
    gl = gap.reshape(n, L, 5)
    out = {"tokens": n}
    for i, name in enumerate(PHASES):
        ph = lay[:, :, i]
        out[name] = {"span_us": round(float(np.mean(ph[..., 3] - ph[..., 0])) / 1e3, 2),
                     "setup_us": round(float(np.mean(ph[..., 2] - ph[..., 0])) / 1e3, 2),
                     "gap_after_us": round(float(np.mean(gl[:, :, i])) / 1e3, 2)}
    out["layer_us"] = round(float(np.mean(seq[:, -1, 3] - seq[:, 0, 0])) / L / 1e3, 2)
    out["embed_us"] = round(float(np.mean(tr[:, 0, 3] - tr[:, 0, 0])) / 1e3, 2)
    out["head_us"] = round(float(np.mean(tr[:, -1, 3] - tr[:, -1, 0])) / 1e3, 2)
    out["token_us"] = round(float(np.mean(tr[:, -1, 3] - tr[:, 0, 0])) / 1e3, 2)
    log("[bench] decode-step timeline (us, mean over %d tokens): %s" % (n, json.dumps(out)))
    return out


def time_sampler(n_vocab, stream, iters=50):
    """Device time of lcx_sample (the sampler chain) on logits rows of the model's vocabulary:
    one row (a batch-1 decode step) and 64 rows (one per sequence of the multi-sequence
    workload), CUDA events on the launching stream after warm-up. Not part of the greedy
    workload's timed region."""
    import torch

    import llama_ubatch_forward_gb300 as lcx
    import synth
    out = {"chain": "top_k 40, top_p 0.95, min_p 0.05, temp 0.8 (the draw: u uniform)", "n_vocab": n_vocab}
    for rows in (1, 64):
        x = synth.normal(0x5A11, 1, rows * n_vocab, 0.0, 2.0).reshape(rows, n_vocab).astype(np.float32)
        x[:, :: max(1, n_vocab // 7)] += 8.0           # a few strong candidates over the background
        dx = torch.from_numpy(x).to("cuda")
        du = torch.from_numpy((synth.uniform_int(0x5A11, 2, rows, 0, 1 << 24) / float(1 << 24)).astype(np.float32)).cuda()
        tok = torch.empty(rows, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(3):
                lcx.sample(dx, du, tokens_out=tok, stream=stream, **SAMPLER_CHAIN)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                rc, _ = lcx.sample(dx, du, tokens_out=tok, stream=stream, **SAMPLER_CHAIN)
            e1.record(stream)
        torch.cuda.synchronize()
        assert rc == 0, rc
        out[f"us_per_call_{rows}_rows"] = round(e0.elapsed_time(e1) * 1e3 / iters, 2)
    return out


def decode_bytes_seqs(cfg, host, ctx_lens):
    """Algorithmic HBM bytes of one decode ubatch whose tokens attend ctx_lens cells each: every
    weight as stored once (one embedding row per token) plus the K/V of every attended cell."""
    w = host.output.nbytes + host.output_norm.nbytes
    for L in host.layers:
        w += sum(v.nbytes for v in L.values())
    kv_cell = cfg.n_layer * cfg.n_head_kv * cfg.head_dim * 2 * 2
    return w + host.tok_embd.shape[1] * len(ctx_lens) + kv_cell * int(np.sum(ctx_lens))


def summarize_profile(pr):
    return {k: {"launches": v["launches"], "ms": round(v["ms"], 3),
                "GBps": round(v["bytes"] / v["ms"] / 1e6, 1) if v["ms"] else None,
                "TFLOPps": round(v["flops"] / v["ms"] / 1e9, 2) if v["ms"] else None}
            for k, v in pr.items() if v["launches"]}


def timed(stream, fn):
    """Device milliseconds of fn() between CUDA events on `stream` (synchronized on both sides)."""
    import torch
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def run_workloads(names, gm8, host8, stream, hbm, bf16):
    """Throughput of the other named workloads, each a warm-up run then one timed run; tokens/s and
    the fraction of the roofline that bounds each phase (decode: algorithmic bytes over the measured
    HBM bandwidth; prefill: algorithmic flops over the measured bf16 tensor peak)."""
    import torch

    import llama_ubatch_forward_gb300 as lcx
    import synth
    from llama_ubatch_forward_gb300.torch_io import upload
    out = {}

    def prefill_decode(key, cfg, host, gm, n_prompt, n_ub, n_ctx, n_dec):
        ctx = lcx.Context(gm, n_ctx, 1, n_ub, stream=stream)
        prompt = synth.prompt_tokens(cfg, n_prompt)
        gen = torch.zeros(n_dec, dtype=torch.int32, device="cuda")
        am = np.zeros(1, np.int32)
        res = {}
        for rep in range(2):   # warm-up, then timed
            ctx.kv_clear()
            pre = timed(stream, lambda: ctx.decode(prompt, argmax_out=am))
            dec = timed(stream, lambda: ctx.decode_greedy(0, int(am[0]), n_dec, gen))
            res = {"prefill_ms": pre, "decode_ms": dec}
        # per-kernel-class device time of the same run (events around every launch), after timing
        ctx.kv_clear()
        ctx.set_profiling(True)
        ctx.decode(prompt, argmax_out=am)
        prof_pre = ctx.profile()
        ctx.set_profiling(True)
        ctx.decode_greedy(0, int(am[0]), n_dec, gen)
        prof_dec = ctx.profile()
        ctx.set_profiling(False)
        del ctx
        dec_b = decode_bytes_per_step(cfg, host, n_prompt, n_dec) / n_dec
        pf = prefill_flops(cfg, n_prompt)
        dgbs = dec_b * n_dec / (res["decode_ms"] / 1e3) / 1e9
        ptf = pf / (res["prefill_ms"] / 1e3) / 1e12
        out[key] = {"workload": f"{cfg.name}: {n_prompt}-token prompt in ubatches of {n_ub}, then {n_dec} greedy "
                                f"decode steps", "warmup": 1, "steps": 1,
                    "decode": {"value": round(n_dec / (res["decode_ms"] / 1e3), 2), "unit": "tokens/s",
                               "bytes_per_step": round(dec_b), "achieved_gbs": round(dgbs, 1),
                               "frac": round(dgbs / hbm, 4), "bound": "hbm"},
                    "prefill": {"value": round(n_prompt / (res["prefill_ms"] / 1e3), 1), "unit": "tokens/s",
                                "flops": pf, "achieved_tflops": round(ptf, 2), "frac": round(ptf / bf16, 4),
                                "bound": "tensor"},
                    "kernel_profile": {"prefill": summarize_profile(prof_pre), "decode": summarize_profile(prof_dec)}}
        log(f"[bench] {key}: {json.dumps(out[key])}")

    if "1b" in names:
        cfg = synth.CONFIGS["1b"]
        host = synth.make_model(cfg)
        gm = upload(host)
        prefill_decode("1b", cfg, host, gm, 512, 512, cfg.n_ctx, 128)
        del gm, host
    if "long" in names:
        # the long-context workload runs on the 8B-shape model itself (its own prompt draw)
        cfg = synth.CONFIGS["long"]
        prefill_decode("long", cfg, host8, gm8, 32768, 2048, cfg.n_ctx, 128)
    if "multiseq" in names:
        cfg = synth.CONFIGS["multiseq"]
        n_seq, n_steps = 64, 128
        lens = synth.multiseq_prompt_lengths(cfg, n_seq)
        prompts = [synth.prompt_tokens(cfg, int(lens[s]), s) for s in range(n_seq)]
        ctx = lcx.Context(gm8, cfg.n_ctx, n_seq, 512, stream=stream)
        seqs = np.arange(n_seq, dtype=np.int32)
        flags = np.ones(n_seq, np.int8)
        am = np.zeros(n_seq, np.int32)
        res = {}
        for rep in range(2):   # warm-up, then timed
            ctx.kv_clear()
            first = np.zeros(n_seq, np.int32)

            def prefill():
                one = np.zeros(1, np.int32)
                for sq in range(n_seq):
                    assert ctx.decode(prompts[sq], seq_id=np.full(prompts[sq].size, sq, np.int32),
                                      argmax_out=one) == 0
                    first[sq] = one[0]

            def decode():
                toks = first.copy()
                for _ in range(n_steps):
                    assert ctx.decode(toks, seq_id=seqs, logits=flags, argmax_out=am) == 0
                    toks = am.copy()

            res = {"prefill_ms": timed(stream, prefill), "decode_ms": timed(stream, decode)}
        # per-kernel-class device time of 8 more decode steps (events around every launch)
        ctx.set_profiling(True)
        toks = am.copy()
        for _ in range(8):
            assert ctx.decode(toks, seq_id=seqs, logits=flags, argmax_out=am) == 0
            toks = am.copy()
        prof_dec = ctx.profile()
        ctx.set_profiling(False)
        del ctx
        n_pre = int(np.sum(lens))
        step_bytes = [decode_bytes_seqs(cfg, host8, lens + i + 1) for i in range(n_steps)]
        dgbs = sum(step_bytes) / (res["decode_ms"] / 1e3) / 1e9
        pf = sum(prefill_flops(cfg, int(n)) - 2 * cfg.n_vocab * cfg.n_embd for n in lens) + \
            n_seq * 2 * cfg.n_vocab * cfg.n_embd
        ptf = pf / (res["prefill_ms"] / 1e3) / 1e12
        out["multiseq"] = {
            "workload": f"multiseq: {n_seq} sequences, prompts of {int(lens.min())}-{int(lens.max())} tokens "
                        f"({n_pre} in total) prefilled in ubatches of 512, then {n_steps} steps of one "
                        f"{n_seq}-token ubatch (one token per sequence, every row flagged, host argmax per step)",
            "warmup": 1, "steps": 1,
            "decode": {"value": round(n_seq * n_steps / (res["decode_ms"] / 1e3), 1), "unit": "tokens/s",
                       "bytes_per_step": round(sum(step_bytes) / n_steps), "achieved_gbs": round(dgbs, 1),
                       "frac": round(dgbs / hbm, 4), "bound": "hbm"},
            "prefill": {"value": round(n_pre / (res["prefill_ms"] / 1e3), 1), "unit": "tokens/s", "flops": pf,
                        "achieved_tflops": round(ptf, 2), "frac": round(ptf / bf16, 4), "bound": "tensor"},
            "kernel_profile": {"decode_8_steps": summarize_profile(prof_dec)}}
        log(f"[bench] multiseq: {json.dumps(out['multiseq'])}")
    return out


def run_lcx(a, rank, world):
    import torch

    import llama_ubatch_forward_gb300 as lcx
    import synth
    from llama_ubatch_forward_gb300.torch_io import upload

    lcx.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg, n_prompt, n_dec, n_ub = workload_args(a)
    t0 = time.perf_counter()
    host = synth.make_model(cfg)
    prompt = synth.prompt_tokens(cfg, n_prompt)
    host_prompt_cache["p"] = prompt
    log(f"[bench] model {cfg.name}: {host.weight_bytes() / 1e9:.2f} GB stored, generated in {time.perf_counter() - t0:.1f}s")
    gm = upload(host)
    stream = torch.cuda.Stream()
    n_ctx = a.n_ctx or cfg.n_ctx
    ctx = lcx.Context(gm, n_ctx, 1, n_ub, stream=stream)
    gen = torch.zeros(n_dec, dtype=torch.int32, device=dev)
    am_host = np.zeros(1, dtype=np.int32)

    def step(ev=None):
        ctx.kv_clear()
        if ev:
            ev[0].record(stream)
        rc = ctx.decode(prompt, argmax_out=am_host)        # syncs for the first generated token
        assert rc == 0, rc
        if ev:
            ev[1].record(stream)
        rc = ctx.decode_greedy(0, int(am_host[0]), n_dec, gen)
        assert rc == 0, rc
        if ev:
            ev[2].record(stream)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for k in range(a.steps):
        step(evs[k])
    g1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = g0.elapsed_time(g1)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms, pre_sum, dec_sum = max_over_ranks([total_ms, sum(pre_ms), sum(dec_ms)], dev, world)
    decode_tps = world * a.steps * n_dec / (dec_sum / 1e3)
    prefill_tps = world * a.steps * n_prompt / (pre_sum / 1e3)

    # per-kernel-class durations: one more step with event brackets around every launch,
    # profiled separately for the prefill and the decode phase
    ctx.kv_clear()
    ctx.set_profiling(True)
    assert ctx.decode(prompt, argmax_out=am_host) == 0
    prof_pre = ctx.profile()
    ctx.set_profiling(True)
    assert ctx.decode_greedy(0, int(am_host[0]), n_dec, gen) == 0
    prof = ctx.profile()
    ctx.set_profiling(False)
    launches_per_step = None
    s0 = ctx.stats().n_kernels
    step()
    torch.cuda.synchronize()
    launches_per_step = ctx.stats().n_kernels - s0

    # end to end through the C ABI with host buffers: host token in, host argmax out, per step
    e2e_steps = max(1, min(a.steps, 2))
    torch.cuda.synchronize()
    t_e2e = 0.0
    for _ in range(e2e_steps):
        ctx.kv_clear()
        am = np.zeros(1, dtype=np.int32)
        assert ctx.decode(prompt, argmax_out=am) == 0
        tok = int(am[0])
        s = time.perf_counter()
        for _ in range(n_dec):
            assert ctx.decode(np.array([tok], np.int32), argmax_out=am) == 0
            tok = int(am[0])
        t_e2e += time.perf_counter() - s
    e2e_tps = world * e2e_steps * n_dec / t_e2e
    sampler = time_sampler(cfg.n_vocab, stream)
    timeline = None
    if a.timeline > 0:
        try:
            timeline = step_timeline(ctx, prompt, am_host, cfg, a.timeline)
        except Exception as ex:  # diagnostics only: never costs the bench line
            timeline = {"error": str(ex)}

    hbm, bf16, bf16_sus, src = peaks()
    workloads = None
    if a.workloads and not a.layers and cfg.name == "8b":
        names = [w for w in a.workloads.split(",") if w]
        try:
            workloads = run_workloads(names, gm, host, stream, hbm, bf16)
        except Exception as ex:  # reported, never costs the main line
            workloads = {"error": repr(ex)}
    g = prof["gemv"]
    # one launch per decode token: the persistent step kernel (weights, KV and head in one launch)
    step_kernel = g["launches"] == n_dec and prof["attention"]["launches"] == 0
    kv_pos_bytes = cfg.n_layer * cfg.n_head_kv * cfg.head_dim * 2 * 2   # K and V of one position, all layers
    if step_kernel:
        dom_kernel = "k_decode_step (persistent: every matmul, attention and the head of a token in one launch)"
        dom_traffic = None
        if cfg.name == "8b" and not a.layers:
            dom_traffic = round(STEP_NCU_TRAFFIC_RATIO * decode_bytes_per_step(cfg, host, n_prompt, n_dec) / n_dec)
    else:
        dom_kernel = "gemv (weight-streaming, all decode matmuls)"
        dom_traffic = None   # separate launches (LCX_DECODE_STEP=0): no current counters
    gemv_gbs = g["bytes"] / (g["ms"] / 1e3) / 1e9 if g["ms"] else 0.0
    gm_ = prof_pre["gemm"]
    gemm_tf = gm_["flops"] / (gm_["ms"] / 1e3) / 1e12 if gm_["ms"] else 0.0
    dec_bytes = decode_bytes_per_step(cfg, host, n_prompt, n_dec)
    dec_gbs = dec_bytes / (sum(dec_ms) / a.steps / 1e3) / 1e9
    pf = prefill_flops(cfg, n_prompt)
    pre_tf = pf / (sum(pre_ms) / a.steps / 1e3) / 1e12
    res = {
        "metric": f"decode tokens/s ({cfg.name}-shape Llama, {linear_type(cfg)} linears, batch 1, {n_dec} greedy steps after a "
                  f"{n_prompt}-token prefill)",
        "value": round(decode_tps, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": round(total_ms / a.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q4_0/q8_0 weights (as stored) x activations split per 32-block into int8 hi + lo "
                 "(about 14 bits; integer dot products, f32 accumulation) in decode; weights dequantized to "
                 "f16 x activations as f16 hi + lo pairs (about 22 bits) -> f32 on the tensor cores in prefill",
        "data": "synthetic (seeded N(0,0.02) weights, uniform token ids)",
        "config": workload_config(a, cfg, n_prompt, n_dec, n_ub, world),
        "prefill": {"value": round(prefill_tps, 1), "unit": "tokens/s",
                    "achieved_tflops": round(pre_tf, 2),
                    "roofline_frac": round(pre_tf / bf16, 4)},
        "decode_roofline": {"bytes_per_step": round(dec_bytes / n_dec), "achieved_gbs": round(dec_gbs, 1), "peak": hbm,
                            "frac": round(dec_gbs / hbm, 4), "peak_source": src},
        "roofline": {"bound": "hbm", "kernel": dom_kernel,
                     "achieved": round(gemv_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gemv_gbs / hbm, 4), "traffic": dom_traffic,
                     "peak_source": src, "launches_profiled": g["launches"],
                     "avg_launch_us": round(g["ms"] * 1e3 / max(1, g["launches"]), 2)},
        "roofline_prefill": {"bound": "tensor", "kernel": "gemm (prefill matmuls)", "achieved": round(gemm_tf, 2),
                             "peak": bf16, "unit": "TFLOP/s", "frac": round(gemm_tf / bf16, 4), "traffic": None,
                             "peak_source": src, "issued_tflops": round(2 * gemm_tf, 2),
                             "issued_frac": round(2 * gemm_tf / bf16, 4),
                             "note": "achieved counts 2 T N K algorithmic flops; every MMA multiplies the weights by "
                                     "the activations' f16 hi and lo parts, so twice that is issued and the "
                                     "design's ceiling is 0.5 of the peak in algorithmic flops"},
        "kernel_profile": {ph: {k: {"launches": v["launches"], "ms": round(v["ms"], 3),
                                    "GBps": round(v["bytes"] / v["ms"] / 1e6, 1) if v["ms"] else None,
                                    "TFLOPps": round(v["flops"] / v["ms"] / 1e9, 2) if v["ms"] else None}
                                for k, v in pr.items() if v["launches"]}
                           for ph, pr in (("prefill", prof_pre), ("decode", prof))},
        "e2e": {"value": round(e2e_tps, 2), "unit": "tokens/s",
                "h2d_bytes_per_step": n_prompt * 20 + n_dec * 20,
                "d2h_bytes_per_step": 4 * (1 + n_dec),
                "how": "lcx_decode per token with host token ids and host argmax (one sync per token)"},
        "gpu_launches": int(launches_per_step * a.steps),
        "sampler": sampler,
        **({"timeline": timeline} if timeline is not None else {}),
        **({"workloads": workloads} if workloads is not None else {}),
        "clocks": clk,
    }
    if rank == 0:
        try:
            if a.no_cpu_baseline:
                raise RuntimeError("skipped (--no-cpu-baseline)")
            res["cpu_baseline"] = cpu_baseline(host, cfg)
        except Exception as ex:  # the baseline is reported, not required
            res["cpu_baseline"] = {"error": str(ex)}
        print(json.dumps(res), flush=True)


def run_reference(a, rank, world):
    """The oracle as the reference arm: same workload shape and metric, bounded sample per step."""
    if rank != 0:
        return
    import oracle
    import synth
    cfg, n_prompt, n_dec, n_ub = workload_args(a)
    host = synth.make_model(cfg)
    prompt = synth.prompt_tokens(cfg, 4)
    n = oracle.set_threads()
    om = oracle.Model(host)
    per = 2  # decode steps per sample
    times = []
    for k in range(a.warmup + a.steps):
        octx = oracle.Context(om, cfg.n_ctx, 1, n_ub)
        rc, _, am = octx.decode(prompt)
        tok = int(am[-1])
        t0 = time.perf_counter()
        for _ in range(per):
            rc, _, am = octx.decode([tok])
            tok = int(am[0])
        if k >= a.warmup:
            times.append(time.perf_counter() - t0)
    v = a.steps * per / sum(times)
    sample = f"{cfg.name} model, fp64 oracle: 4-token prompt then {per} decode steps per step"
    print(json.dumps({
        "impl": "reference", "metric": f"decode tokens/s ({cfg.name}-shape Llama, {linear_type(cfg)} linears, batch 1, {n_dec} "
                                       f"greedy steps after a {n_prompt}-token prefill)",
        "value": round(v, 4), "unit": "tokens/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(1e3 * sum(times) / a.steps, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,0.02) weights, uniform token ids)",
        "config": {**workload_config(a, cfg, n_prompt, n_dec, n_ub, world),
                   "sample": f"each step times {per} decode steps after a 4-token prompt of the same model (the "
                             f"fp64 oracle cannot run the full workload in minutes)"},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lcx", choices=["lcx", "reference"])
    ap.add_argument("--config", default="8b")
    ap.add_argument("--prompt", type=int, default=2048)
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--n-ubatch", type=int, default=512)
    ap.add_argument("--n-ctx", type=int, default=0, help="override the context size (0: the config's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timeline", type=int, default=0,
                    help="diagnostics: per-phase timeline of the decode step over this many tokens (0: off)")
    ap.add_argument("--workloads", default="1b,long,multiseq",
                    help="other named workloads measured after the main one (comma list; empty: none)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: the first N layers of the model (0: all); the line is then not the workload's")
    a = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and a.impl == "lcx":
        import torch
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    if a.impl == "reference":
        run_reference(a, rank, world)
    else:
        run_lcx(a, rank, world)
    if world > 1 and a.impl == "lcx":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
