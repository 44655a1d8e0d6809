#!/usr/bin/env python3
"""Benchmark of the libqw decoder forward pass on GB300.

Default run (no --config): one JSON line whose headline is the 28-layer Qwen3-0.6B shape
with seeded random bf16 weights, batch 1, a 5-token uniform-random prompt, prefill + 64
greedy decode steps. One bench step is one such generation (KV reset + reserve, prefill, 64
decode steps replayed from CUDA graphs, each step feeding its pick back on the device).
``value`` counts the generated tokens (65 per step) per second of device time with inputs
resident in HBM; ``e2e`` is the same metric through ``qw_generate`` from pinned host
buffers (prompt copied in, picks copied out, every step). The same line carries one object
per other workload, each timed the same way (K timed steps after W warm-up steps), with its
own step-level roofline, ``e2e`` (host buffers, copies inside the timed region) and
``cpu_baseline`` (the fp64 oracle on a bounded sample):

  ``b64_decode``       batch 64, each sequence prefilled with 1024 tokens, then 128 greedy
                       decode steps (decode tokens/s; one bench step = the 128 steps);
  ``prefill_16x512``   batch 16 x 512-token prefill (prefill tokens/s);
  ``one_block``        one decoder block + tied head, batch 1, 5 + 16 steps (generated tok/s);
  ``long_context_b8``  batch 8, cached lengths uniform in [1024, 32768] injected by the
                       synthetic KV fill, 32 decode steps (decode tokens/s).

``--config N`` runs workload N alone as the headline (0: one block, 1: B=1, 2: B=64 decode,
3: 16 x 512 prefill, 4: long context).

Per-kernel times (``kernels``, and ``roofline`` of the headline) come from CUDA events around
every launch of one kernel kind in one extra step run with programmatic dependent launch off,
i.e. serialised; the timed steps overlap launches, so the step-level fractions
(``step_roofline`` / each workload's ``roofline``) are the ones consistent with ``value``.

Multi-GPU: replicas only (independent sequences per GPU, no collective on the data path).
``--gpus N`` without a launcher re-executes itself under ``torch.distributed.run`` with N
processes (one per GPU); ``value`` is the sum over ranks of the units processed divided by
the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on this host on a bounded sample of the same
workload (the only other program this bench runs); under N processes rank 0 alone runs it.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tok/s (B=1/64) & prefill tok/s, Qwen3-0.6B shape; % of HBM/TC roofline"

CONFIGS = {
    0: dict(workload="qwen3-0.6b-shape 1 block + tied head, B=1, 5-token prompt, prefill + 16 greedy decode steps",
            shape=synth.ONE_BLOCK, B=1, prompt=5, n_decode=16, unit="tok/s", kind="generate"),
    1: dict(workload="qwen3-0.6b-shape 28 layers, B=1, 5-token prompt, prefill + 64 greedy decode steps",
            shape=synth.QWEN3_0_6B, B=1, prompt=5, n_decode=64, unit="tok/s", kind="generate"),
    2: dict(workload="qwen3-0.6b-shape 28 layers, B=64, 1024-token prefill each, 128 greedy decode steps",
            shape=synth.QWEN3_0_6B, B=64, prompt=1024, n_decode=128, unit="tok/s", kind="decode"),
    3: dict(workload="qwen3-0.6b-shape 28 layers, prefill B=16 x 512 tokens",
            shape=synth.QWEN3_0_6B, B=16, prompt=512, n_decode=0, unit="tok/s", kind="prefill"),
    4: dict(workload="qwen3-0.6b-shape 28 layers, B=8, cached lengths U[1024, 32768] (paged, 16-token pages), "
                     "32 greedy decode steps",
            shape=synth.QWEN3_0_6B, B=8, prompt=None, n_decode=32, unit="tok/s", kind="decode_long"),
}


# DRAM bytes per launch of a kernel from one ncu capture (summaries under profiles/), reported
# as roofline.traffic only while the kernel's source file is byte-identical to the capture's.
NCU_TRAFFIC = {
    # batch-1 cluster path: one launch captured in a 28-layer decode step (cache of ~7 keys;
    # the K/V bytes of the bench's ~37-key caches add 0.15 MB per launch)
    (1, "rmsnorm+qkv+attention+o_proj (cluster kernel)"): (12744448, "decode_qwen3_decoder_gb300/csrc/k_dec1.cu",
                                                           "47f5ba5eece4a18f9646982d763c8af8ff0387b20584c6883ec4610537133ad2"),


    # 16 x 512 prefill, one gate/up launch (CTA pairs): read 29.39 MB + written 0.82 MB
    (3, "gate_up+silu_mul"): (29385984 + 822528, "decode_qwen3_decoder_gb300/csrc/k_gemm.cu",
                              "b9a1cb9f933fb98cbef3992ee013642777ea92516c576e65e423e1b31237671f"),
    # batched decode attention: one 32-sequence launch of the two-stream path over 1026-key
    # caches read 136.50 MB and wrote 2.77 MB, 1.033 x its algorithmic bytes; the bench times
    # one 64-sequence launch per layer (285.2 MB algorithmic), so 1.033 x 285.2 MB
    (2, "attention"): (294611600, "decode_qwen3_decoder_gb300/csrc/k_attn.cu",
                       "c7d1340c9aacb00eb320a872b80d25332c032f92af8f54b65538ea7a40888f8d"),
}


def ncu_traffic(config: int, kernel: str):
    ent = NCU_TRAFFIC.get((config, kernel))
    if ent is None:
        return None
    nbytes, src, sha = ent
    try:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), src), "rb") as fh:
            cur = hashlib.sha256(fh.read()).hexdigest()
    except OSError:
        return None
    return nbytes if cur == sha else None


def rank_token_seed(config: int, rank: int) -> int:
    """Seed of the token ids of one replica: each rank decodes its own synthetic prompts."""
    return 1000 + config + 17 * rank


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, ms_max: float) -> float:
    """Units per second over all ranks: every rank processed the same work in at most ms_max."""
    return units_per_rank_step * steps * world / (ms_max / 1e3)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def step_stats(events):
    """Median and 95th percentile (us) of the intervals between consecutive CUDA events
    recorded on one stream (one interval per step)."""
    d = sorted(events[i].elapsed_time(events[i + 1]) * 1e3 for i in range(len(events) - 1))
    p95 = d[min(len(d) - 1, int(math.ceil(0.95 * len(d))) - 1)]
    return {"median_us": round(statistics.median(d), 2), "p95_us": round(p95, 2), "n": len(d)}


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_bytes(kind: int, s, T: int, B: int, ctx: float = 0.0, clusters: bool = False) -> float:
    """Algorithmic bytes of one launch of a kernel kind (weights once + activations in/out;
    ctx: cached keys read by an attention launch). clusters: the batch-1 path of two cluster
    kernels per layer, whose attention launch (kind 3) also does q|k|v and whose MLP launch
    (kind 5) also does down_proj."""
    D, I, QD, KD, V = s.hidden, s.inter, s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim, s.vocab
    QKV = QD + 2 * KD
    if clusters and kind == 3:   # x + 8 down_proj slots in, q|k|v + o_proj weights, cached K/V, o_proj partials out
        return QKV * D * 2 + D * QD * 2 + ctx * KD * 2 * 2 + 2 * KD * 2 + (1 + 8) * D * 4 + s.n_kv_heads * D * 4
    if clusters and kind == 5:   # x + o_proj partials in, gate/up/down weights, down_proj partials added into 8 slots
        return 3 * I * D * 2 + (1 + s.n_kv_heads) * D * 4 + 8 * D * 4
    if kind == 1:   # q|k|v projection (+ fused input RMSNorm)
        return QKV * D * 2 + T * D * 4 + T * QKV * 4 + D * 2
    if kind == 3:   # attention fused with o_proj (one token): o_proj weights + the cached K/V once
        return D * QD * 2 + ctx * KD * 2 * 2 + s.n_kv_heads * T * D * 4
    if kind == 4:   # o_proj + residual
        return D * QD * 2 + T * QD * 2 + 2 * T * D * 4
    if kind == 5:   # gate/up + SiLU*mul (+ fused post-attention RMSNorm)
        return 2 * I * D * 2 + T * D * 4 + T * I * 2 + D * 2
    if kind == 6:   # down_proj + residual
        return D * I * 2 + T * I * 2 + 2 * T * D * 4
    if kind == 7:   # final norm + tied LM head + argmax
        return V * D * 2 + B * D * 4 + D * 2
    return float("nan")


def step_bytes(s, B: int, ctx: float) -> float:
    """Algorithmic bytes of one whole decode step: every weight once (fp16), the KV cache of
    each sequence once (ctx keys, fp16 K and V, all layers), the new K/V written, and the
    embedding rows, logits-free."""
    D, I, QD, KD, V, L = s.hidden, s.inter, s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim, s.vocab, s.n_layers
    weights = L * ((QD + 2 * KD) * D + D * QD + 2 * I * D + D * I) * 2 + V * D * 2
    kv = B * ctx * L * 2 * KD * 2
    return weights + kv + B * L * 2 * KD * 2 + B * D * 2


SERIAL_NOTE = ("CUDA events around each launch of the kind, in one extra step with programmatic dependent "
               "launch off (serialised); the timed steps overlap launches")

# the batch-1 path of two cluster kernels per layer
CLUSTER_KIND_NAMES = {3: "rmsnorm+qkv+attention+o_proj (cluster kernel)",
                      5: "rmsnorm+gate_up+swiglu+down_proj (cluster kernel)", 7: "lm_head+argmax"}
KIND_NAMES = {1: "qkv_proj(rmsnorm fused)", 2: "qknorm_rope_append", 3: "attention(+o_proj fused at B=1)",
              4: "o_proj+residual",
              5: "gate_up+silu_mul(rmsnorm fused)", 6: "down_proj+residual", 7: "lm_head+argmax"}
# names on the tensor-core path (more than 8 token rows)
TC_KIND_NAMES = {1: "qkv_proj+qk_norm+rope+kv_append", 3: "attention", 4: "o_proj+residual",
                 5: "gate_up+silu_mul", 6: "down_proj+residual", 7: "lm_head+argmax", 8: "rmsnorm"}


_WEIGHTS = {}


def model_weights(s) -> dict:
    """HF-named bf16 bit arrays of the seeded weights of shape `s`, drawn once per run. Every
    tensor has its own seed, so a shape with fewer layers is a subset of the 28-layer draw."""
    full = synth.QWEN3_0_6B
    if s != full and "full" in _WEIGHTS and dataclasses.replace(full, n_layers=s.n_layers) == s:
        keep = tuple(f"model.layers.{i}." for i in range(s.n_layers))
        return {k: v for k, v in _WEIGHTS["full"].items()
                if not k.startswith("model.layers.") or k.startswith(keep)}
    key = "full" if s == full else s
    if key not in _WEIGHTS:
        t0 = time.time()
        _WEIGHTS[key] = dict(synth.Weights(s, seed=0).named())
        log(f"weights of {s.n_layers} layer(s) drawn in {time.time() - t0:.1f}s")
    return _WEIGHTS[key]


def gpu_uuid_of(dev: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


def run_ours(args, cfg, rank, world):
    import torch
    import decode_qwen3_decoder_gb300 as pkg
    pkg.build()
    qw = pkg.qw
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    s = cfg["shape"]
    B, P, ND = cfg["B"], cfg["prompt"], cfg["n_decode"]
    max_ctx = P + ND + 16
    eng = qw.Engine(s, model_weights(s), max_tokens=max(B * P, 8), max_batch=max(B, 8), max_context=max_ctx,
                    kv_pages=B * ((max_ctx + 15) // 16) + 8, max_seqs=max(B, 8))
    st = eng.stream
    seqs = list(range(B))
    prompt = synth.make_tokens(s.vocab, B * P, rank_token_seed(cfg["id"], rank))
    d_prompt = torch.tensor(prompt, dtype=torch.int32, device="cuda")
    d_cur = torch.zeros(B, dtype=torch.int32, device="cuda")
    d_out = torch.zeros((ND + 1, B), dtype=torch.int32, device="cuda")
    launches = [0]

    def prefill():
        qw.qw_kv_reset(eng.kv, -1, st)
        for sq in seqs:
            qw.qw_kv_reserve(eng.kv, sq, P + ND, st)
        qw.qw_prefill(eng.model, eng.kv, seqs, [P] * B, d_prompt.data_ptr(), 0, d_out[0].data_ptr(), st)
        launches[0] += qw.qw_last_launch_count(eng.model)

    def decode_all():
        """The ND greedy steps, row i of d_out feeding row i + 1, as qw_decode_steps graphs."""
        done, n = 0, 0
        while done < ND:
            n = min(qw.QW_MAX_GRAPH_STEPS, ND - done)
            qw.qw_decode_steps(eng.model, eng.kv, seqs, n, d_out[done].data_ptr(), d_out[done + 1].data_ptr(), st)
            launches[0] += qw.qw_last_launch_count(eng.model)
            done += n
        return n

    def one_step():
        prefill()
        return decode_all()

    for _ in range(args.warmup):
        n_last = one_step()
    step_launches = qw.qw_last_launch_count(eng.model) // n_last  # per decode step
    st.synchronize()
    status = qw.qw_sync_status(eng.model, st)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up: {qw.qw_last_error()}")
    gpu_uuid = gpu_uuid_of(dev)
    barrier(world)
    launches[0] = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_uuid) as clk:
        torch.cuda.synchronize()
        e0.record(st)
        for _ in range(args.steps):
            one_step()
        e1.record(st)
        torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    ms_max = reduce_max(ms, world)
    gpu_launches = launches[0]
    tokens_per_step = B * (ND + 1)
    value = whole_job_rate(tokens_per_step, args.steps, world, ms_max)
    status = qw.qw_sync_status(eng.model, st)
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region: {qw.qw_last_error()}")

    # ---- decode-step latency alone (the timed region's graphs), for the record ----
    prefill()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(st)
    decode_all()
    eb.record(st)
    st.synchronize()
    decode_us = ea.elapsed_time(eb) * 1e3 / ND
    # spread of single steps: one graph per step (qw_decode_step), an event between steps
    prefill()
    with torch.cuda.stream(st):
        d_cur.copy_(d_out[0])
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(ND + 1)]
    evs[0].record(st)
    for i in range(ND):
        qw.qw_decode_step(eng.model, eng.kv, seqs, d_cur.data_ptr(), 0, d_cur.data_ptr(), st)
        evs[i + 1].record(st)
    st.synchronize()
    decode_stats = dict(step_stats(evs), graphs="one per step (qw_decode_step)",
                        mean_us=round(evs[0].elapsed_time(evs[ND]) * 1e3 / ND, 2))

    # ---- per-kernel timing with CUDA events around each launch of one kernel kind ----
    # (events bracket the launches inside the captured decode graphs; measured on the
    # same workload right after the timed region)
    hbm, bf16_burst, bf16_sust, peak_src = peaks()
    # one token per step: two cluster kernels per layer (step begin + 2 per layer + the LM
    # head, which also ends the step), else attention and o_proj as one kernel (kind 3)
    clusters = B == 1 and step_launches == 2 * s.n_layers + 2
    names = CLUSTER_KIND_NAMES if clusters else KIND_NAMES
    n_launch_per_step = ({3: s.n_layers, 5: s.n_layers, 7: 1} if clusters else
                         {1: s.n_layers, 3: s.n_layers, 5: s.n_layers, 6: s.n_layers, 7: 1} if B == 1 else
                         {1: s.n_layers, 4: s.n_layers, 5: s.n_layers, 6: s.n_layers, 7: 1})
    kinds = {}
    for kind, nl in n_launch_per_step.items():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nl)]
        for ev in evs:          # torch creates the CUDA event on its first record
            ev.record(st)
        handles = (qw.ctypes.c_void_p * (2 * nl))(*[ev.cuda_event for ev in evs])
        durs, ctxs = [], []
        qw.qw_kv_reset(eng.kv, -1, st)
        for sq in seqs:
            qw.qw_kv_reserve(eng.kv, sq, P + ND, st)
        qw.qw_prefill(eng.model, eng.kv, seqs, [P] * B, d_prompt.data_ptr(), 0, d_cur.data_ptr(), st)
        qw.qw_profile_set(eng.model, kind, handles, 2 * nl)
        for i in range(min(ND, 16)):
            qw.qw_decode_step(eng.model, eng.kv, seqs, d_cur.data_ptr(), 0, d_cur.data_ptr(), st)
            st.synchronize()
            if i >= 2:
                durs.extend(evs[2 * j].elapsed_time(evs[2 * j + 1]) for j in range(nl))
                ctxs.append(P + i + 1)
        qw.qw_profile_set(eng.model, 0, None, 0)
        st.synchronize()
        avg_us = statistics.mean(durs) * 1e3
        nbytes = kernel_bytes(kind, s, B, B, statistics.mean(ctxs), clusters)
        kinds[kind] = dict(name=names[kind], launches_per_step=nl, avg_us=avg_us,
                           total_us_per_step=avg_us * nl, bytes=nbytes)
    dom = max(kinds, key=lambda k: kinds[k]["total_us_per_step"])
    dk = kinds[dom]
    achieved = dk["bytes"] / (dk["avg_us"] * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dk["name"], "achieved": round(achieved, 1), "peak": hbm,
                "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": ncu_traffic(cfg["id"], dk["name"]), "algorithmic_bytes_per_launch": dk["bytes"],
                "avg_launch_us": round(dk["avg_us"], 3), "timing": SERIAL_NOTE}
    step_b = step_bytes(s, B, P + ND / 2)
    # ---- end to end through qw_generate with pinned host buffers ----
    h_prompt = torch.empty(B * P, dtype=torch.int32, pin_memory=True).numpy()
    h_prompt[:] = prompt
    h_out = torch.empty((B, ND + 1), dtype=torch.int32, pin_memory=True).numpy()
    e2e_steps = max(1, min(args.steps, 5))
    for i in range(e2e_steps + 1):
        if i == 1:
            t_e2e = time.perf_counter()
        qw.qw_kv_reset(eng.kv, -1, st)
        for sq in seqs:
            qw.qw_kv_reserve(eng.kv, sq, P + ND, st)
        qw.qw_generate(eng.model, eng.kv, seqs, [P] * B, h_prompt, ND, h_out, st)
    e2e_s = time.perf_counter() - t_e2e
    e2e_val = reduce_sum(tokens_per_step * e2e_steps / e2e_s, world)
    ref_ids = d_out.t().cpu().numpy()
    if not np.array_equal(h_out, ref_ids):
        log("warning: qw_generate picks differ from the device loop's picks")

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": cfg["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 weights x f32 activations, f32 accumulate, f16 KV cache",
        "data": "synthetic (seeded random-init bf16 weights N(0,0.02), uniform-random token ids)",
        "config": {"workload": cfg["workload"], "batch": B, "prompt_tokens": P, "decode_steps": ND,
                   "tokens_per_step": tokens_per_step, "parallelism": f"replicas x{world} (no collective)",
                   "l2": "weights (1.19 GB per decode step) exceed L2; no flush",
                   "decode_step_us": round(decode_us, 2),
                   "decode_step_stats": decode_stats,
                   "decode_step_bytes": step_b,
                   "decode_step_hbm_frac": round(step_b / (decode_us * 1e-6) / 1e9 / hbm, 4)},
        "roofline": roofline,
        "step_roofline": {"bound": "hbm", "achieved": round(step_b / (decode_us * 1e-6) / 1e9, 1), "peak": hbm,
                          "unit": "GB/s", "frac": round(step_b / (decode_us * 1e-6) / 1e9 / hbm, 4),
                          "bytes_per_step": step_b, "step_us": round(decode_us, 2),
                          "note": "whole decode step (weights + KV read once) over the event-timed graph replay"},
        "kernels": {names[k]: {"avg_us": round(v["avg_us"], 3), "per_step_us": round(v["total_us_per_step"], 2),
                                    "GB/s": round(v["bytes"] / (v["avg_us"] * 1e-6) / 1e9, 1)}
                    for k, v in kinds.items()},
        "kernels_timing": SERIAL_NOTE,
        "e2e": {"value": round(e2e_val, 2), "unit": cfg["unit"], "h2d_bytes_per_step": B * P * 4,
                "d2h_bytes_per_step": B * (ND + 1) * 4},
        "gpu_launches": gpu_launches,
        "clocks": clk.summary(),
    }
    if cfg["id"] == 1:
        out["sampling"] = time_sampling(qw, s.vocab, st)
    eng.close()
    if cfg["id"] == 1:
        out["quantized_decode"] = time_quantized_decode(qw, s, P, ND, hbm)
    return out


def time_quantized_decode(qw, s, P: int, ND: int, hbm: float):
    """B=1 decode steps (multi-step graph replays) with the layers' projections quantized to 8 and 4 bits
    (qw_quantize_weights; the tied LM head stays bf16), on the default workload's prompt
    length and step count: microseconds per step and the HBM fraction of the bytes a step
    reads (codes + scales, LM head, KV)."""
    import torch
    res = {}
    for bits in (8, 4):
        eng = qw.Engine(s, model_weights(s), max_tokens=8, max_batch=8, max_context=P + ND + 16,
                        kv_pages=(P + ND + 15) // 16 + 8, max_seqs=8)
        eng.quantize(bits)
        st = eng.stream
        d_prompt = torch.tensor(synth.make_tokens(s.vocab, P, 4242).astype(np.int32), device="cuda")
        d_out = torch.zeros((ND + 1, 1), dtype=torch.int32, device="cuda")

        def steps(n):   # n <= ND decode steps in qw_decode_steps graphs, as the bf16 line
            qw.qw_kv_reset(eng.kv, -1, st)
            qw.qw_kv_reserve(eng.kv, 0, P + ND, st)
            qw.qw_prefill(eng.model, eng.kv, [0], [P], d_prompt.data_ptr(), 0, d_out[0].data_ptr(), st)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            done = 0
            while done < n:
                k = min(qw.QW_MAX_GRAPH_STEPS, n - done)
                qw.qw_decode_steps(eng.model, eng.kv, [0], k, d_out[done].data_ptr(), d_out[done + 1].data_ptr(), st)
                done += k
            b.record(st)
            st.synchronize()
            return a.elapsed_time(b) * 1e3 / n

        steps(ND)  # warm-up: captures the graphs
        us = steps(ND)
        if qw.qw_sync_status(eng.model, st) != 0:
            raise RuntimeError(f"device status after quantized decode: {qw.qw_last_error()}")
        nbytes = qw.qw_quantize_bytes(eng.model, bits) + s.vocab * s.hidden * 2 + \
            (P + ND / 2) * s.n_layers * 2 * s.n_kv_heads * s.head_dim * 2
        res[f"{bits}bit"] = {"decode_step_us": round(us, 2), "tok_s": round(1e6 / us, 1),
                             "bytes_per_step": int(nbytes),
                             "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / hbm, 4)}
        eng.close()
    res["note"] = ("B=1 greedy decode, the layers' projections as grouped affine codes (groups of 64, "
                   "fp16 scale and bias); not the headline number, which uses the bf16 weights")
    return res


def time_sampling(qw, vocab: int, st, reps: int = 20):
    """qw_sample_top_p (temperature 0.7, top_p 0.9) on B rows of seeded N(0, 2) logits, for
    B = 1 and 64: microseconds per call (CUDA events on the launching stream, after 3 warm-up
    calls) and the rate at which the logits are read once (B * vocab * 4 bytes per call)."""
    import torch
    res = {}
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    for B in (1, 64):
        lg = torch.randn((B, vocab), device="cuda", generator=g) * 2.0
        u = torch.rand(B, device="cuda", generator=g)
        nx = torch.empty(B, dtype=torch.int32, device="cuda")
        call = lambda: qw.qw_sample_top_p(B, vocab, lg.data_ptr(), vocab, 0.7, 0.9, u.data_ptr(), nx.data_ptr(), st)
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        st.synchronize()
        e0.record(st)
        for _ in range(reps):
            call()
        e1.record(st)
        st.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        res[f"B{B}"] = {"us_per_call": round(us, 2), "logits_GB/s": round(B * vocab * 4 / (us * 1e-6) / 1e9, 1)}
    res["note"] = "temperature 0.7, top_p 0.9; one cluster of 8 CTAs per row, latency-bound"
    return res


def attn_bytes_layer(s, ctx_total: float) -> float:
    """KV bytes one attention launch reads: every cached key and value once (fp16)."""
    return ctx_total * s.n_kv_heads * s.head_dim * 2 * 2


def run_other(args, cfg, rank, world):
    """Batched decode (2), prefill (3) and long-context decode (4)."""
    import torch
    import decode_qwen3_decoder_gb300 as pkg
    pkg.build()
    qw = pkg.qw
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    s = cfg["shape"]
    B, ND = cfg["B"], cfg["n_decode"]
    kind = cfg["kind"]
    if kind == "decode_long":
        lens = synth.make_lengths(B, 1024, 32768, 2000)
    else:
        lens = np.full(B, cfg["prompt"], dtype=np.int64)
    max_ctx = int(lens.max()) + ND + 16
    chunk_seqs = 16 if kind != "decode_long" else B            # prefill 16 sequences per call
    max_tokens = max(int(lens[:chunk_seqs].sum()), B, 8) if kind != "decode_long" else max(B, 8)
    pages = int(sum((l + ND + 15) // 16 + 1 for l in lens)) + 8
    eng = qw.Engine(s, model_weights(s), max_tokens=max_tokens, max_batch=max(B, 8), max_context=max_ctx,
                    kv_pages=pages, max_seqs=max(B, 8))
    st = eng.stream
    seqs = list(range(B))
    rng_seed = rank_token_seed(cfg["id"], rank)
    d_cur = torch.zeros(B, dtype=torch.int32, device="cuda")
    hbm, bf16_burst, bf16_sust, peak_src = peaks()

    def fill_cache():
        qw.qw_kv_reset(eng.kv, -1, st)
        for sq in seqs:
            qw.qw_kv_reserve(eng.kv, sq, int(lens[sq]) + ND, st)
        if kind == "decode_long":
            for sq in seqs:
                qw.qw_kv_fill_synthetic(eng.kv, sq, int(lens[sq]), 77, st)
        else:
            toks = synth.make_tokens(s.vocab, int(lens.sum()), rng_seed)
            d_t = torch.tensor(toks, dtype=torch.int32, device="cuda")
            off = 0
            for a in range(0, B, chunk_seqs):
                grp = seqs[a:a + chunk_seqs]
                n = int(lens[a:a + chunk_seqs].sum())
                qw.qw_prefill(eng.model, eng.kv, grp, [int(lens[q]) for q in grp], d_t.data_ptr() + 4 * off, 0,
                              d_cur.data_ptr() + 4 * a, st)
                off += n
        st.synchronize()

    launches = [0]
    if kind == "prefill":
        toks = torch.tensor(synth.make_tokens(s.vocab, int(lens.sum()), rng_seed), dtype=torch.int32, device="cuda")

        def one_step():
            qw.qw_kv_reset(eng.kv, -1, st)
            for sq in seqs:
                qw.qw_kv_reserve(eng.kv, sq, int(lens[sq]), st)
            qw.qw_prefill(eng.model, eng.kv, seqs, [int(x) for x in lens], toks.data_ptr(), 0, d_cur.data_ptr(), st)
            launches[0] += qw.qw_last_launch_count(eng.model)
        units_per_step = int(lens.sum())
    else:
        fill_cache()

        def one_step():
            for sq in seqs:
                qw.qw_kv_truncate(eng.kv, sq, int(lens[sq]), st)
            for i in range(ND):
                qw.qw_decode_step(eng.model, eng.kv, seqs, d_cur.data_ptr(), 0, d_cur.data_ptr(), st)
                launches[0] += qw.qw_last_launch_count(eng.model)
        units_per_step = B * ND

    for _ in range(args.warmup):
        one_step()
    st.synchronize()
    if qw.qw_sync_status(eng.model, st) != 0:
        raise RuntimeError(f"device status after warm-up: {qw.qw_last_error()}")
    gpu_uuid = gpu_uuid_of(dev)
    barrier(world)
    launches[0] = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(gpu_uuid) as clk:
        torch.cuda.synchronize()
        e0.record(st)
        for i in range(args.steps):
            one_step()
            step_evs[i].record(st)
        e1.record(st)
        torch.cuda.synchronize()
    barrier(world)
    ms_max = reduce_max(e0.elapsed_time(e1), world)
    value = whole_job_rate(units_per_step, args.steps, world, ms_max)
    if qw.qw_sync_status(eng.model, st) != 0:
        raise RuntimeError(f"device status in the timed region: {qw.qw_last_error()}")
    if kind == "prefill":
        step_lat = step_stats([e0] + step_evs)
    else:
        # decode-step latency, one interval per step (the same graphs, right after the timed region)
        for sq in seqs:
            qw.qw_kv_truncate(eng.kv, sq, int(lens[sq]), st)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(ND + 1)]
        evs[0].record(st)
        for i in range(ND):
            qw.qw_decode_step(eng.model, eng.kv, seqs, d_cur.data_ptr(), 0, d_cur.data_ptr(), st)
            evs[i + 1].record(st)
        st.synchronize()
        step_lat = step_stats(evs)

    # per-kernel timing (events around each launch of a kind, one step after the timed region)
    L = s.n_layers
    kinds_n = {1: L, 3: L, 4: L, 5: L, 6: L, 7: 1}
    if (int(lens.sum()) if kind == "prefill" else B) > 8:
        kinds_n[8] = 2 * L + 1  # tensor-core path: RMSNorm runs as its own kernel
    kinds = {}
    for kd, nl in kinds_n.items():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nl)]
        for ev in evs:
            ev.record(st)
        handles = (qw.ctypes.c_void_p * (2 * nl))(*[ev.cuda_event for ev in evs])
        if kind != "prefill":
            for sq in seqs:
                qw.qw_kv_truncate(eng.kv, sq, int(lens[sq]), st)
        qw.qw_profile_set(eng.model, kd, handles, 2 * nl)
        if kind == "prefill":
            one_step()
        else:
            qw.qw_decode_step(eng.model, eng.kv, seqs, d_cur.data_ptr(), 0, d_cur.data_ptr(), st)
        st.synchronize()
        qw.qw_profile_set(eng.model, 0, None, 0)
        d = [evs[2 * j].elapsed_time(evs[2 * j + 1]) * 1e3 for j in range(nl)]
        names = TC_KIND_NAMES if 8 in kinds_n else KIND_NAMES
        kinds[kd] = dict(name=names.get(kd, str(kd)), avg_us=statistics.mean(d),
                         per_step_us=sum(d), launches=nl)
    T = int(lens.sum()) if kind == "prefill" else B
    D, I, QD, KD, V = s.hidden, s.inter, s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim, s.vocab
    step_ms = ms_max / args.steps
    if kind == "prefill":
        flops = {1: 2 * T * (QD + 2 * KD) * D, 4: 2 * T * D * QD, 5: 2 * T * 2 * I * D, 6: 2 * T * D * I,
                 7: 2 * B * V * D}
        for kd, f in flops.items():
            kinds[kd]["TFLOP/s"] = round(f / (kinds[kd]["avg_us"] * 1e-6) / 1e12, 1)
        gemm_kinds = [1, 4, 5, 6]
        dom = max(gemm_kinds, key=lambda k: kinds[k]["per_step_us"])
        ach = flops[dom] / (kinds[dom]["avg_us"] * 1e-6) / 1e12
        dominant = {"bound": "tensor", "kernel": kinds[dom]["name"] + " (tcgen05 GEMM)", "achieved": round(ach, 1),
                    "peak": bf16_sust, "peak_source": peak_src + " bf16 sustained (fp16 operands run at the bf16 rate)",
                    "unit": "TFLOP/s", "frac": round(ach / bf16_sust, 4),
                    "traffic": ncu_traffic(cfg["id"], kinds[dom]["name"]),
                    "algorithmic_flops_per_launch": flops[dom], "avg_launch_us": round(kinds[dom]["avg_us"], 2),
                    "timing": SERIAL_NOTE}
        attn_pairs = sum(int(l) * (int(l) + 1) // 2 for l in lens)
        total_flops = L * sum(flops[k] for k in gemm_kinds) + flops[7] + L * attn_pairs * 4 * s.head_dim * s.n_heads
        achieved = total_flops / (step_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_burst,
                    "peak_source": peak_src + " bf16 burst (fp16 operands run at the bf16 rate)", "unit": "TFLOP/s",
                    "frac": round(achieved / bf16_burst, 4), "flop_per_step": total_flops,
                    "frac_of_sustained": round(achieved / bf16_sust, 4),
                    "note": "whole prefill step (projection GEMMs, causal attention, LM head) over the timed step"}
        extra = {"step_tflop": total_flops / 1e12, "prefill_step_stats": step_lat}
    else:
        ctx = float(np.mean(lens)) + ND / 2
        kv_bytes = attn_bytes_layer(s, float(np.sum(lens)) + B * ND / 2)
        byts = {1: (QD + 2 * KD) * D * 2, 3: kv_bytes, 4: D * QD * 2, 5: 2 * I * D * 2, 6: D * I * 2, 7: V * D * 2}
        for kd, b in byts.items():
            kinds[kd]["GB/s"] = round(b / (kinds[kd]["avg_us"] * 1e-6) / 1e9, 1)
        dom = max(byts, key=lambda k: kinds[k]["per_step_us"])
        ach = byts[dom] / (kinds[dom]["avg_us"] * 1e-6) / 1e9
        dominant = {"bound": "hbm", "kernel": kinds[dom]["name"], "achieved": round(ach, 1), "peak": hbm,
                    "peak_source": peak_src, "unit": "GB/s", "frac": round(ach / hbm, 4),
                    "traffic": ncu_traffic(cfg["id"], kinds[dom]["name"]),
                    "algorithmic_bytes_per_launch": byts[dom], "avg_launch_us": round(kinds[dom]["avg_us"], 2),
                    "timing": SERIAL_NOTE}
        step_b = step_bytes(s, B, ctx)
        step_us = step_ms / ND * 1e3
        achieved = step_b / (step_us * 1e-6) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "peak_source": peak_src,
                    "unit": "GB/s", "frac": round(achieved / hbm, 4), "bytes_per_step": step_b,
                    "note": "whole decode step (every weight and cached K/V byte once) over the timed steps"}
        extra = {"decode_step_us": round(step_us, 2), "decode_step_stats": step_lat, "decode_step_bytes": step_b,
                 "mean_cached_len": float(np.mean(lens))}

    # ---- end to end through the C ABI with host buffers (copies inside the timed region) ----
    e2e = e2e_other(qw, eng, kind, seqs, lens, ND, s, rng_seed, args.steps, world, units_per_step)
    out = {"metric": METRIC, "value": round(value, 2), "unit": cfg["unit"], "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f16 tensor-core operands (bf16 weights converted), f32 accumulate, f16 KV cache"
           if T > 8 else "bf16 weights x f32 activations, f32 accumulate, f16 KV cache",
           "data": "synthetic (seeded random-init bf16 weights N(0,0.02), uniform-random token ids)",
           "config": dict({"workload": cfg["workload"], "batch": B, "l2": "working set exceeds L2; no flush"}, **extra),
           "roofline": roofline, "dominant_kernel": dominant,
           "kernels": {v["name"]: {k: (round(x, 2) if isinstance(x, float) else x) for k, x in v.items() if k != "name"}
                       for v in kinds.values()},
           "kernels_timing": SERIAL_NOTE,
           "e2e": e2e, "gpu_launches": launches[0], "clocks": clk.summary()}
    eng.close()
    return out


def e2e_other(qw, eng, kind, seqs, lens, ND, s, seed, steps, world, units_per_step):
    """The workload's metric through the C ABI from pinned host buffers, host<->device copies
    inside the timed region. Decode: every decode step copies the B token ids in, runs
    qw_decode_step and reads the B picks back (the host feeds them to the next step), i.e. a
    host-driven serving loop. Prefill: every step copies the prompt ids in, runs qw_prefill
    and reads the B picks back."""
    import torch
    st = eng.stream
    B = len(seqs)
    n = max(1, min(steps, 5))
    if kind == "prefill":
        T = int(np.sum(lens))
        h_in = torch.from_numpy(synth.make_tokens(s.vocab, T, seed).astype(np.int32)).pin_memory()
        d_in = torch.empty(T, dtype=torch.int32, device="cuda")
        h_out = torch.empty(B, dtype=torch.int32).pin_memory()
        d_out = torch.empty(B, dtype=torch.int32, device="cuda")
        t0 = None
        for i in range(n + 1):
            if i == 1:
                t0 = time.perf_counter()
            qw.qw_kv_reset(eng.kv, -1, st)
            for sq in seqs:
                qw.qw_kv_reserve(eng.kv, sq, int(lens[sq]), st)
            with torch.cuda.stream(st):
                d_in.copy_(h_in, non_blocking=True)
            qw.qw_prefill(eng.model, eng.kv, seqs, [int(x) for x in lens], d_in.data_ptr(), 0, d_out.data_ptr(), st)
            with torch.cuda.stream(st):
                h_out.copy_(d_out, non_blocking=True)
            st.synchronize()
        dt = time.perf_counter() - t0
        h2d, d2h = T * 4, B * 4
    else:
        h_in = torch.zeros(B, dtype=torch.int32).pin_memory()
        h_out = torch.empty(B, dtype=torch.int32).pin_memory()
        d_in = torch.empty(B, dtype=torch.int32, device="cuda")
        d_out = torch.empty(B, dtype=torch.int32, device="cuda")
        t0 = None
        for i in range(n + 1):
            if i == 1:
                t0 = time.perf_counter()
            for sq in seqs:
                qw.qw_kv_truncate(eng.kv, sq, int(lens[sq]), st)
            h_in.zero_()
            for _ in range(ND):
                with torch.cuda.stream(st):
                    d_in.copy_(h_in, non_blocking=True)
                qw.qw_decode_step(eng.model, eng.kv, seqs, d_in.data_ptr(), 0, d_out.data_ptr(), st)
                with torch.cuda.stream(st):
                    h_out.copy_(d_out, non_blocking=True)
                st.synchronize()
                h_in.copy_(h_out)
        dt = time.perf_counter() - t0
        h2d, d2h = B * 4 * ND, B * 4 * ND
    if qw.qw_sync_status(eng.model, st) != 0:
        raise RuntimeError(f"device status after the e2e loop: {qw.qw_last_error()}")
    val = reduce_sum(units_per_step * n / dt, world)
    return {"value": round(val, 2), "unit": "tok/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n}


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------------------
class _NamedWeights:
    """Weight provider of the oracle over the HF-named bf16 arrays this bench already drew."""

    def __init__(self, s, named):
        self.shape, self.named_ = s, named

    @property
    def embed(self):
        return self.named_["model.embed_tokens.weight"]

    @property
    def final_norm(self):
        return self.named_["model.norm.weight"]

    def layer(self, i):
        pre = f"model.layers.{i}."
        return {k[len(pre):]: v for k, v in self.named_.items() if k.startswith(pre)}


_ORACLES = {}


def oracle_model(s):
    """The fp64 oracle of shape `s` with every layer widened up front (kept for the run)."""
    import oracle
    if s.n_layers not in _ORACLES:
        m = oracle.Model(_NamedWeights(s, model_weights(s)))
        for i in range(s.n_layers):
            m.layer(i)
        _ = m.embed32
        _ORACLES[s.n_layers] = m
    return _ORACLES[s.n_layers]


def oracle_sample(cfg, n_decode: int, seed: int):
    """Generated tokens per second of the fp64 oracle on prefill + n_decode greedy steps."""
    import oracle
    s = cfg["shape"]
    m = oracle_model(s)
    prompt = synth.make_tokens(s.vocab, cfg["prompt"], seed).tolist()
    t0 = time.perf_counter()
    oracle.generate(m, prompt, n_decode, keep_hidden=False)
    dt = time.perf_counter() - t0
    return (n_decode + 1) / dt, dt


def oracle_decode_sample(s, ctx: int, n_steps: int, seed: int):
    """Decode tokens per second of the fp64 oracle: one sequence over a cache of `ctx` tokens
    (injected by the counter-based KV fill, as the long-context workload does; the values do
    not change the work of a step), n_steps greedy decode steps."""
    import oracle
    m = oracle_model(s)
    pos = np.arange(ctx)
    prior = {l: (synth.kv_fill_values(77, l, 0, pos, s.n_kv_heads, s.head_dim).astype(np.float64),
                 synth.kv_fill_values(77, l, 1, pos, s.n_kv_heads, s.head_dim).astype(np.float64))
             for l in range(s.n_layers)}
    cache = oracle.SeqCache(s.n_layers, prior=lambda l: prior[l], prior_len=ctx)
    tok = int(synth.make_tokens(s.vocab, 1, seed)[0])
    t0 = time.perf_counter()
    for _ in range(n_steps):
        tok = oracle.argmax_lowest(oracle.forward(m, [tok], cache)["logits"])
    dt = time.perf_counter() - t0
    return n_steps / dt, dt


def oracle_prefill_sample(s, n_tokens: int, seed: int):
    """Prefill tokens per second of the fp64 oracle on one sequence of n_tokens."""
    import oracle
    m = oracle_model(s)
    toks = synth.make_tokens(s.vocab, n_tokens, seed).tolist()
    t0 = time.perf_counter()
    oracle.forward(m, toks, oracle.SeqCache(s.n_layers))
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(cfg):
    """The oracle as it stands on this host's cores, on a bounded sample of the workload."""
    kind, s = cfg["kind"], cfg["shape"]
    if kind == "generate":
        n = 96 if s.n_layers > 1 else 32
        v, dt = oracle_sample(cfg, n, 4242)
        sample = (f"fp64 NumPy oracle, {cfg['prompt']}-token prompt prefill + {n} greedy decode steps of the same "
                  f"model shape, batch 1 ({dt:.1f} s)")
    elif kind == "decode":
        n = 32
        v, dt = oracle_decode_sample(s, cfg["prompt"], n, 4242)
        sample = (f"fp64 NumPy oracle, 1 of the {cfg['B']} sequences decoding {n} greedy steps over a "
                  f"{cfg['prompt']}-token cache ({dt:.1f} s); sequences are independent, so its rate per token is "
                  f"the oracle's rate for the batch")
    elif kind == "prefill":
        n_seq, dt, tok = 3, 0.0, 0
        for i in range(n_seq):
            v, d = oracle_prefill_sample(s, cfg["prompt"], 4242 + i)
            dt, tok = dt + d, tok + cfg["prompt"]
        v = tok / dt
        sample = (f"fp64 NumPy oracle, prefill of {n_seq} of the {cfg['B']} sequences of {cfg['prompt']} tokens "
                  f"({dt:.1f} s); sequences are independent")
    else:
        lens = synth.make_lengths(cfg["B"], 1024, 32768, 2000)
        n = 16
        v, dt = oracle_decode_sample(s, int(lens.min()), n, 4242)
        sample = (f"fp64 NumPy oracle, the shortest of the {cfg['B']} sequences ({int(lens.min())} cached tokens) "
                  f"decoding {n} greedy steps ({dt:.1f} s); longer caches cost more per step")
    return {"value": round(v, 4), "unit": cfg["unit"], "cores": cores(), "kind": "oracle", "sample": sample}


def run_reference(args, cfg):
    samples = []
    n_dec = 4
    for i in range(args.warmup + args.steps):
        v, dt = oracle_sample(cfg, n_dec, 5000 + i)
        if i >= args.warmup:
            samples.append(dt)
    tokens = (n_dec + 1) * args.steps
    total = sum(samples)
    val = tokens / total
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": cfg["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random-init bf16 weights widened to fp64)",
            "config": {"workload": cfg["workload"], "sample": f"prefill {cfg['prompt']} + {n_dec} decode steps per step",
                       "processes": "rank 0 alone runs the oracle on the host cores"},
            "cpu_baseline": {"value": round(val, 4), "unit": cfg["unit"], "cores": cores(), "kind": "oracle",
                             "sample": f"prefill + {n_dec} greedy decode steps per bench step"},
            "e2e": {"value": round(val, 4), "unit": cfg["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# workloads of the default line besides the headline, under these keys
SUB_KEYS = {2: "b64_decode", 3: "prefill_16x512", 0: "one_block", 4: "long_context_b8"}
COMMON_KEYS = ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data")


def free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def replica_command(n: int, argv) -> list:
    """The command that runs this bench as n replica processes (one per GPU) on this node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__)] + list(argv)


def workload(args, cid: int, alone: bool) -> dict:
    cfg = dict(CONFIGS[cid])
    cfg["id"] = cid
    if alone and args.prompt_len > 0 and cid in (2, 3):
        cfg["prompt"] = args.prompt_len
        cfg["workload"] += f" [reduced: {args.prompt_len} tokens per sequence]"
    if alone and args.decode_steps > 0 and cid in (2, 4):
        cfg["n_decode"] = args.decode_steps
        cfg["workload"] += f" [reduced: {args.decode_steps} decode steps]"
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=None, choices=[0, 1, 2, 3, 4],
                    help="run one workload alone (default: all five, the B=1 generation as headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prompt-len", type=int, default=0,
                    help="with --config 2/3: tokens per sequence instead of the configured length (smaller case "
                         "for profiling)")
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="with --config 2/4: decode steps per timed step instead of the configured count")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # replicas: one process per GPU, launched here when no launcher did it
        sys.exit(subprocess.call(replica_command(args.gpus, sys.argv[1:])))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, workload(args, 1 if args.config is None else args.config, True))),
                  flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    ids = [args.config] if args.config is not None else [1, 2, 3, 0, 4]
    results = []
    for cid in ids:
        cfg = workload(args, cid, args.config is not None)
        out = run_ours(args, cfg, rank, world) if cid in (0, 1) else run_other(args, cfg, rank, world)
        results.append((cid, cfg, out))
    if rank == 0:
        if not args.no_cpu_baseline:
            for cid, cfg, out in results:
                out["cpu_baseline"] = cpu_baseline(cfg)
        head = results[0][2]
        for cid, cfg, out in results[1:]:
            head[SUB_KEYS[cid]] = {k: v for k, v in out.items() if k not in COMMON_KEYS}
        print(json.dumps(head), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
