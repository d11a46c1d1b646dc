#!/usr/bin/env python
"""Throughput of the Qwen3-0.6B-shaped decoder step on one GB300 (or N replicas).

Headline workload (the serving configuration): bf16 weights, f16 paged KV
cache (16-token blocks), fp32 accumulation; 32 sequences preloaded with
uniform-random contexts of distinct lengths 1024..2048 by a real prefill, then
K greedy decode steps at batch 32 (each step feeds the previous step's argmax
ids).  `value` = decode tokens/s with every input resident in HBM; the same
run also reports batch-1 decode (context 2048) and a chunked prefill of
4 x 4096 tokens in 512-token chunks.  Weights are random-init N(0, 0.02).

Every timed step reads 1.19 GB of weights plus the KV cache (5.6+ GB at batch
32), far larger than the 129 MB L2, so no L2 flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch with torch.distributed.run: each rank runs an independent
replica on its own GPU (the step has no exchange), timing is max over ranks.
"""

from __future__ import annotations

import argparse
import ctypes as C
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s (batch 1/32) & prefill tokens/s at 0.6B shape; % HBM/TC roofline"
WORKLOAD = ("qwen3-0.6B-shape decoder (596,049,920 params), bf16 weights / f16 paged KV (block 16) / fp32 accum; "
            "greedy decode at batch 32, contexts 1024..2048 (distinct) preloaded by prefill")
KV_BYTES_PER_CTX_TOKEN_LAYER = 8 * 128 * 2 * 2  # K and V, 8 KV heads x 128, f16
WEIGHT_BYTES_BF16 = 1_192_099_840  # 596,049,920 params x 2 bytes (tied head read once per step)
WEIGHT_BYTES_F32 = 2_384_199_680   # the same in fp32
KV_BYTES_PER_CTX_TOKEN_F32 = 28 * 8 * 128 * 2 * 4  # K and V of every layer, fp32 (229,376 B)
NOMINAL_HBM_GBS = 8000.0           # the ~8 TB/s HBM3e figure the fractions are also given against
# fp32 FFMA peak from unit counts and clock: 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz
FP32_FFMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
PROF_STEPS = 4   # untimed steps whose dominant-class launches are timed with CUDA events
REPEATS = 5      # timed loops of K steps; the median loop is reported


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class Clocks:
    """Sample SM clocks and throttle reasons with nvidia-smi during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            time.sleep(0.3)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------

def build_model(shape, weights, max_positions, max_tokens, max_seqs, n_blocks):
    from decoder_qwen3_step_gb300 import dec
    from decoder_qwen3_step_gb300.runtime import Decoder

    return Decoder(shape, weights, mode=dec.DEC_BF16_F16KV, max_positions=max_positions, max_tokens=max_tokens,
                   max_seqs=max_seqs, n_blocks=n_blocks)


def profile_classes(m, classes, on):
    for c in classes:
        m.L.dec_profile_enable(m.handle, c, 1 if on else 0)


def read_profile(m, cls):
    ms, n = C.c_double(), C.c_int64()
    m.L.dec_profile_read(m.handle, cls, C.byref(ms), C.byref(n))
    return ms.value, n.value


def max_over_ranks(ms, device):
    """The slowest rank's elapsed time: every rank gets the maximum."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms, world):
    """Units processed by all ranks per second of the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def launches(m):
    n = C.c_int64()
    m.L.dec_launch_count(m.handle, C.byref(n))
    return n.value


def our_arm(args, rank, world):
    import torch

    from decoder_qwen3_step_gb300 import dec, inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    shape = inputs.SHAPES["qwen3_0p6b"]
    S = 32
    lens = inputs.serving_context_lengths(S)
    e2e_steps = max(8, args.steps // 4)
    b1_steps = max(32, args.steps)
    # positions every sequence may reach: warmup, 2 class-share steps, PROF_STEPS dominant-class steps,
    # 2 unprofiled steps (graph capture), REPEATS timed loops, e2e, batch-1 (last sequence only)
    extra = args.warmup + 2 + PROF_STEPS + 2 + REPEATS * args.steps + e2e_steps + 3 + b1_steps + 2 + 16
    max_positions = max(((max(lens) + extra + 15) // 16) * 16, 4096 + 64)
    weights = inputs.make_weights(shape)
    blocks_needed = sum((L + extra) // 16 + 1 for L in lens) + 4 * (4096 // 16 + 2) + 200
    m = build_model(shape, weights, max_positions, 8192, 64, blocks_needed)
    del weights
    stream = torch.cuda.current_stream()
    pk = peaks()

    # ---- preload: every sequence's context by a real prefill (rows: last token) ----
    ctx_ids = [inputs.make_ids(shape["vocab"], 2048, seed=100 + s)[:lens[s]] for s in range(S)]
    tables = [m.blocks_for(L + extra) for L in lens]
    group = 4
    first = []
    for g in range(0, S, group):
        _, am = m.prefill([(ctx_ids[s], 0, tables[s]) for s in range(g, g + group)], rows=dec.DEC_ROWS_LAST)
        first.append(am)
    next_ids = torch.cat(first).to(torch.int32)
    torch.cuda.synchronize()
    pos = list(lens)
    # the decode steps pass their block tables as int32 arrays (no per-step list conversion)
    tables = [np.asarray(t, dtype=np.int32) for t in tables]

    V = shape["vocab"]
    logits = torch.empty((S, V), dtype=torch.float32, device=dev)
    ids_buf = [torch.empty((S,), dtype=torch.int32, device=dev) for _ in range(2)]
    ids_buf[0].copy_(next_ids)

    def decode_step(i, batch_pos, seqs_idx, buf_in, buf_out):
        m.decode([([0], batch_pos[j], tables[s]) for j, s in enumerate(seqs_idx)], device_ids=buf_in,
                 out=(logits[:len(seqs_idx)], buf_out))

    # warmup
    for i in range(args.warmup):
        decode_step(i, pos, range(S), ids_buf[i & 1], ids_buf[(i + 1) & 1])
        pos = [p + 1 for p in pos]
    torch.cuda.synchronize()
    launches(m)
    # which kernel class dominates the step (short events pass, untimed)
    profile_classes(m, range(len(dec.KERNEL_CLASSES)), True)
    for i in range(2):
        decode_step(i, pos, range(S), ids_buf[(args.warmup + i) & 1], ids_buf[(args.warmup + i + 1) & 1])
        pos = [p + 1 for p in pos]
    shares = {name: read_profile(m, c)[0] for c, name in enumerate(dec.KERNEL_CLASSES)}
    profile_classes(m, range(len(dec.KERNEL_CLASSES)), False)
    dom_name = max(shares, key=shares.get)
    dom = dec.KERNEL_CLASSES.index(dom_name)
    launches(m)

    # the dominant class's time per launch: CUDA events around its launches in
    # PROF_STEPS untimed steps (their events are record nodes in a graph of their own)
    step_no = args.warmup + 2
    prof_ctx = 0
    profile_classes(m, [dom], True)
    for i in range(PROF_STEPS):
        prof_ctx += sum(p + 1 for p in pos)
        decode_step(i, pos, range(S), ids_buf[(step_no + i) & 1], ids_buf[(step_no + i + 1) & 1])
        pos = [p + 1 for p in pos]
    torch.cuda.synchronize()
    step_no += PROF_STEPS
    # (a new set of profiled classes runs eagerly once, is captured the next step, then replays)
    dom_ms, dom_n = read_profile(m, dom)
    profile_classes(m, [dom], False)
    # two unprofiled steps: the headline graph is captured (first eager, second captured)
    for i in range(2):
        decode_step(i, pos, range(S), ids_buf[(step_no + i) & 1], ids_buf[(step_no + i + 1) & 1])
        pos = [p + 1 for p in pos]
    step_no += 2
    launches(m)

    # ---- timed region: REPEATS loops of K decode steps at batch 32, no profiling nodes ----
    # every loop decodes the same K positions (contexts start at 1,024..2,048 plus the
    # steps above), rewriting the same cache slots, so each loop times the same workload
    pos0 = list(pos)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    loop_ms = []
    with Clocks(dev.index) as clk:
        for r in range(REPEATS):
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            pos = list(pos0)
            t_start.record(stream)
            for i in range(args.steps):
                decode_step(i, pos, range(S), ids_buf[(step_no + i) & 1], ids_buf[(step_no + i + 1) & 1])
                pos = [p + 1 for p in pos]
            t_end.record(stream)
            torch.cuda.synchronize()
            step_no += args.steps
            t = t_start.elapsed_time(t_end)
            if world > 1:
                t = max_over_ranks(t, dev)
            loop_ms.append(t)
    if world > 1:
        dist.barrier()
    ms = statistics.median(loop_ms)
    n_launch = launches(m)
    value = whole_job_rate(S * args.steps, ms, world)
    ctx_sum = prof_ctx
    # roofline of the dominant kernel class: algorithmic bytes per launch / event time per launch
    L = shape["n_layers"]
    per_launch_s = (dom_ms / max(dom_n, 1)) / 1e3
    launches_per_step = max(dom_n, 1) / PROF_STEPS
    if dom_name == "step":
        # the whole step in one kernel: every weight byte once, every cached K/V byte once,
        # the new K/V rows and the logits written
        alg_bytes = (WEIGHT_BYTES_BF16 + ctx_sum * KV_BYTES_PER_CTX_TOKEN_LAYER * L / PROF_STEPS
                     + S * KV_BYTES_PER_CTX_TOKEN_LAYER * L + S * shape["vocab"] * 4)
        unit_note = ("per step: 1,192,099,840 B of bf16 weights + 4,096 B of K+V per context token per layer "
                     "(28 layers) + the new K/V rows + fp32 logits [32, 151936]")
    elif dom_name == "attn":
        alg_bytes = ctx_sum * KV_BYTES_PER_CTX_TOKEN_LAYER / PROF_STEPS * L / launches_per_step  # per launch (one layer)
        unit_note = "4,096 B of K+V per context token per layer; units = sum of the 32 context lengths"
    else:
        alg_bytes = _class_weight_bytes(dom_name, shape) + 0.0
        unit_note = "weight bytes of this projection (bf16), read once per launch"
    achieved = alg_bytes / per_launch_s / 1e9
    # DRAM bytes (read + write) per launch over algorithmic bytes, from one ncu capture of the same
    # kernel on a smaller case (attention: 32 sequences x 1,025 keys, 142.92 MB for 134.35 MB; the
    # one-kernel step: batch 1 at context 2,048, 1.4349 GB for 1.4271 GB), scaled to this launch
    traffic_ratio = {"attn": 142.92 / 134.35, "step": 1.4349 / 1.4271}.get(dom_name)
    traffic = int(alg_bytes * traffic_ratio) if traffic_ratio else None
    roofline = {"bound": "hbm", "kernel": dom_name, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "peak_nominal": NOMINAL_HBM_GBS,
                "traffic": traffic,
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of a smaller case, "
                                  "scaled by algorithmic bytes" if traffic else None,
                "peak_source": pk["source"], "bytes_per_launch": int(alg_bytes), "per_unit": unit_note,
                "launch_us": round(per_launch_s * 1e6, 2), "launches": dom_n,
                "timing": f"CUDA events around the class's {dom_n} launches in {PROF_STEPS} untimed steps",
                "step_share": {k: round(v / max(sum(shares.values()), 1e-9), 4) for k, v in shares.items()}}

    # ---- e2e: host ids in, host ids out, every step ----
    host_ids = next_ids.cpu().numpy().astype(np.int32)
    pinned_out = torch.empty((S,), dtype=torch.int32, pin_memory=True)
    torch.cuda.synchronize()
    h2d = 0
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        seqs = [([int(host_ids[s])], pos[s], tables[s]) for s in range(S)]
        m.decode(seqs, out=(logits, ids_buf[0]))
        pinned_out.copy_(ids_buf[0], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        host_ids = pinned_out.numpy().copy()
        pos = [p + 1 for p in pos]
    e2e_s = time.perf_counter() - t0
    if world > 1:
        e2e_s = max_over_ranks(e2e_s * 1e3, dev) / 1e3
    MB = (max_positions + 15) // 16
    h2d = 4 * (3 * S + (S + 1) + S + S + S * MB)
    e2e = {"value": round(whole_job_rate(S * e2e_steps, e2e_s * 1e3, world), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": 4 * S, "steps": e2e_steps}

    # ---- batch-1 decode of the longest sequence from context 2,048 (its prefilled ids;
    # later positions are rewritten) ----
    s1 = S - 1
    b1_ids = [torch.empty((1,), dtype=torch.int32, device=dev) for _ in range(2)]
    b1_ids[0].copy_(ids_buf[0][s1:s1 + 1])
    lg1 = torch.empty((1, V), dtype=torch.float32, device=dev)
    p1 = lens[s1]
    for i in range(3):
        m.decode([([0], p1, tables[s1])], device_ids=b1_ids[i & 1], out=(lg1, b1_ids[(i + 1) & 1]))
        p1 += 1
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    b1_ctx = 0
    for i in range(b1_steps):
        b1_ctx += p1 + 1
        m.decode([([0], p1, tables[s1])], device_ids=b1_ids[(i + 3) & 1], out=(lg1, b1_ids[(i + 4) & 1]))
        p1 += 1
    e1.record(stream)
    torch.cuda.synchronize()
    b1_ms = e0.elapsed_time(e1) / b1_steps
    # kernel-class shares of a batch-1 step (two extra steps with events, untimed)
    profile_classes(m, range(len(dec.KERNEL_CLASSES)), True)
    for i in range(2):
        m.decode([([0], p1, tables[s1])], device_ids=b1_ids[i & 1], out=(lg1, b1_ids[(i + 1) & 1]))
        p1 += 1
    b1_cls = {name: read_profile(m, c) for c, name in enumerate(dec.KERNEL_CLASSES)}
    profile_classes(m, range(len(dec.KERNEL_CLASSES)), False)
    b1_tot = sum(v[0] for v in b1_cls.values()) or 1e-9
    b1_bytes = WEIGHT_BYTES_BF16 + (b1_ctx / b1_steps) * KV_BYTES_PER_CTX_TOKEN_LAYER * L
    decode_b1 = {"tokens_per_s": round(1e3 / b1_ms, 1), "ms_per_token": round(b1_ms, 4),
                 "hbm_frac": round(b1_bytes / (b1_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                 "hbm_frac_nominal": round(b1_bytes / (b1_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4),
                 "bytes_per_token": int(b1_bytes), "context": p1,
                 "kernel_us_per_step": {k: round(v[0] * 1e3 / 2, 1) for k, v in b1_cls.items() if v[1]},
                 "kernel_share": {k: round(v[0] / b1_tot, 4) for k, v in b1_cls.items() if v[1]}}

    # ---- chunked prefill: 4 x 4096 tokens, 512-token chunks interleaved across sequences ----
    pf_ids = [inputs.make_ids(V, 4096, seed=200 + s) for s in range(4)]
    pf_tab = [m.blocks_for(4096) for _ in range(4)]

    def prefill_pass():
        for k in range(8):
            m.prefill([(pf_ids[s][512 * k:512 * (k + 1)], 512 * k, pf_tab[s]) for s in range(4)],
                      rows=dec.DEC_ROWS_LAST, out=(logits[:4], ids_buf[1][:4]))

    prefill_pass()
    torch.cuda.synchronize()
    e0.record(stream)
    prefill_pass()
    e1.record(stream)
    torch.cuda.synchronize()
    pf_ms = e0.elapsed_time(e1)
    # one more pass with events around every kernel class: the products' tensor-core rate
    profile_classes(m, range(len(dec.KERNEL_CLASSES)), True)
    prefill_pass()
    pf_cls = {name: read_profile(m, c) for c, name in enumerate(dec.KERNEL_CLASSES)}
    profile_classes(m, range(len(dec.KERNEL_CLASSES)), False)
    d, H, Hkv, D, F = (shape[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "ff_hidden"))
    ntok = 16384
    nl = shape["n_layers"]
    flops = {"qkv": 2 * ntok * nl * (H + 2 * Hkv) * D * d, "oproj": 2 * ntok * nl * d * H * D,
             "gateup": 2 * ntok * nl * 2 * F * d, "down": 2 * ntok * nl * d * F}
    proj_ms = sum(pf_cls[k][0] for k in flops)
    proj_tf = sum(flops.values()) / (proj_ms / 1e3) / 1e12
    prefill = {"tokens_per_s": round(16384 / (pf_ms / 1e3), 1), "ms": round(pf_ms, 3),
               "kernel_ms": {k: round(v[0], 3) for k, v in pf_cls.items() if v[1]},
               "projection_tflops": round(proj_tf, 1),
               "projection_tc_frac": round(proj_tf / pk["bf16_tflops"], 4),
               "per_product_tc_frac": {k: round(flops[k] / (pf_cls[k][0] / 1e3) / 1e12 / pk["bf16_tflops"], 4)
                                       for k in flops},
               "tc_peak_tflops": pk["bf16_tflops"], "tc_peak_source": pk["source"]}

    status = m.device_status()
    m.close()
    fp32 = fp32_parity_runs(dev, pk)
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": S, "context_lengths": [min(lens), max(lens)],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1.19 GB weights + >5.6 GB KV read per step); no flush",
                   "launch": "each step replays a captured CUDA graph (no profiling nodes in the timed loops)",
                   "timing": f"median of {REPEATS} timed loops of {args.steps} steps each, every loop over the same positions",
                   "loop_ms": [round(t, 3) for t in loop_ms]},
        "roofline": roofline, "e2e": e2e, "gpu_launches": n_launch, "clocks": clk.summary(),
        "decode_b1": decode_b1, "prefill_4x4096": prefill, "fp32_parity_mode": fp32, "device_status": status,
    }


def _class_weight_bytes(name, shape):
    d, H, Hkv, D, F, V = (shape[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "ff_hidden", "vocab"))
    return 2 * {"qkv": (H + 2 * Hkv) * D * d, "oproj": d * H * D, "gateup": 2 * F * d, "down": d * F,
                "lmhead": V * d}.get(name, 0)


def fp32_parity_runs(dev, pk):
    """The parity mode at the Qwen3-0.6B shape (fp32 weights, KV and
    arithmetic): the 188-token prompt prefilled with logits at every position
    (P-C3: 228.2 GFLOP, FFMA), then 256 greedy decode tokens at batch 1,
    context 189 -> 444 (D-b1-fp32: 2,384,199,680 B of weights + 229,376 B of
    K/V per context token)."""
    import torch

    from decoder_qwen3_step_gb300 import dec, inputs
    from decoder_qwen3_step_gb300.runtime import Decoder

    shape = inputs.SHAPES["qwen3_0p6b"]
    V = shape["vocab"]
    m = Decoder(shape, inputs.make_weights(shape), mode=dec.DEC_FP32, max_positions=512, max_tokens=512, max_seqs=1,
                n_blocks=40)
    ids = inputs.make_ids(V, 188)
    table = m.blocks_for(188 + 257)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    logits = torch.empty((188, V), dtype=torch.float32, device=dev)
    am = torch.empty((188,), dtype=torch.int32, device=dev)
    warm = m.blocks_for(188)
    for _ in range(2):
        m.prefill([(ids, 0, warm)], out=(logits, am))
    torch.cuda.synchronize()
    e0.record(stream)
    m.prefill([(ids, 0, table)], out=(logits, am))
    e1.record(stream)
    torch.cuda.synchronize()
    pf_ms = e0.elapsed_time(e1)
    d, H, Hkv, D, F, L = (shape[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "ff_hidden", "n_layers"))
    proj = 2 * ((H + 2 * Hkv) * D * d + d * H * D + 2 * F * d + d * F) * L
    attn = 4 * H * D * L * sum(p + 1 for p in range(188))
    flops = 188 * proj + 188 * 2 * V * d + attn
    tok = torch.empty((1,), dtype=torch.int32, device=dev)
    nxt = torch.empty((1,), dtype=torch.int32, device=dev)
    tok.copy_(am[187:188])
    lg1 = torch.empty((1, V), dtype=torch.float32, device=dev)
    steps, ctx_sum = 256, 0
    for i in range(3):  # warm-up and graph capture; the timed loop rewrites these positions
        m.decode([([0], 188 + i, table)], device_ids=tok, out=(lg1, nxt))
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        ctx_sum += 188 + i + 1
        m.decode([([0], 188 + i, table)], device_ids=tok if i % 2 == 0 else nxt, out=(lg1, nxt if i % 2 == 0 else tok))
    e1.record(stream)
    torch.cuda.synchronize()
    d_ms = e0.elapsed_time(e1) / steps
    bytes_tok = WEIGHT_BYTES_F32 + ctx_sum / steps * KV_BYTES_PER_CTX_TOKEN_F32
    status = m.device_status()
    m.close()
    return {"prefill_188": {"ms": round(pf_ms, 3), "tokens_per_s": round(188 / (pf_ms / 1e3), 1),
                            "gflop": round(flops / 1e9, 1), "tflops": round(flops / (pf_ms / 1e3) / 1e12, 2),
                            "ffma_frac": round(flops / (pf_ms / 1e3) / 1e12 / FP32_FFMA_TFLOPS, 4),
                            "ffma_peak_tflops": round(FP32_FFMA_TFLOPS, 1),
                            "ffma_peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz"},
            "decode_b1": {"tokens_per_s": round(1e3 / d_ms, 1), "ms_per_token": round(d_ms, 4),
                          "context": [189, 188 + steps], "bytes_per_token": int(bytes_tok),
                          "hbm_frac": round(bytes_tok / (d_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                          "hbm_frac_nominal": round(bytes_tok / (d_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4)},
            "device_status": status}


# ------------------------------------------------------------------------------------------------
# the oracle on host cores: the CPU baseline and the reference arm
# ------------------------------------------------------------------------------------------------

def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


def _oracle_sample(n_sample, horizon):
    """The oracle at the headline shape and caches for n_sample of the 32
    sequences, at their context lengths, with room for `horizon` new tokens.

    The caches hold seeded random K/V (the cost of a decode step does not
    depend on the cached values), so no prefill is timed."""
    from decoder_qwen3_step_gb300 import inputs
    from oracle.model import DecoderConfig, Oracle

    shape = inputs.SHAPES["qwen3_0p6b"]
    lens = inputs.serving_context_lengths(32)
    pick = [lens[i] for i in np.linspace(0, 31, n_sample).astype(int)]
    cfg = DecoderConfig(**shape, max_positions=max(pick) + horizon + 1)
    orc = Oracle(cfg, inputs.make_weights(shape), mode="bf16")
    rng = np.random.default_rng(5)
    caches = []
    for L in pick:
        c = orc.new_cache(L + horizon + 1)
        for l in range(cfg.n_layers):
            c.k[l][:L] = rng.standard_normal((L, cfg.n_kv_heads, cfg.head_dim))
            c.v[l][:L] = rng.standard_normal((L, cfg.n_kv_heads, cfg.head_dim))
            c.written[l][:L] = True
        caches.append(c)
    return orc, cfg, caches, pick


def _oracle_step(orc, cfg, caches, pick, step):
    """One float64 decode step: one new token for each sampled sequence."""
    for c, L in zip(caches, pick):
        orc.forward(c, [step % cfg.vocab], L + step)


def _filled_cache(orc, cfg, n_ctx, room):
    """A cache holding n_ctx positions of constant K/V (the cost of the next
    tokens does not depend on the cached values)."""
    c = orc.new_cache(n_ctx + room)
    for l in range(cfg.n_layers):
        c.k[l][:n_ctx] = 0.01
        c.v[l][:n_ctx] = 0.01
        c.written[l][:n_ctx] = True
    return c


def cpu_baselines(budget_s=2.5):
    """The oracle on the host cores: the headline decode rate (one float64
    token for each of the shortest and longest of the 32 serving sequences)
    and, per configuration, prefill and decode tokens/s on bounded samples
    (each timed piece stops after about budget_s): the tiny and small
    decoders, the Qwen3-0.6B shape in the parity mode (fp32 weights) and in
    the serving mode (bf16-rounded weights)."""
    from decoder_qwen3_step_gb300 import inputs
    from oracle.model import DecoderConfig, Oracle

    def timed(fn, units_per_call, limit):
        n, t0 = 0, time.perf_counter()
        while n < limit:
            fn(n)
            n += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return n * units_per_call / dt, n, dt

    def run(orc, vocab, n_prompt, start, pre, dctx, caches):
        ids = inputs.make_ids(vocab, n_prompt, seed=3)

        def prefill(i):
            c = pre if pre is not None else orc.new_cache(n_prompt + 1)
            orc.forward(c, ids, start, rows="all" if start == 0 else "last")

        pf, n_pf, t_pf = timed(prefill, n_prompt, 3)

        def decode(i):
            for c, L in zip(caches, dctx):
                orc.forward(c, [i % vocab], L + i)

        dc, n_dc, t_dc = timed(decode, len(dctx), 64)
        sample = (f"prefill: {n_pf} x {n_prompt} tokens" + (f" after {start} cached" if start else "")
                  + f" ({t_pf:.1f} s); decode: {n_dc} step(s) at batch {len(dctx)}, contexts {dctx} ({t_dc:.1f} s)")
        return {"prefill_tokens_per_s": round(pf, 2), "decode_tokens_per_s": round(dc, 2), "sample": sample}

    out = {}
    for name, shp, n_prompt, dctx in (("C1 tiny fp32", "tiny", 16, [16]), ("C2 small fp32", "small", 128, [128] * 4)):
        shape = inputs.SHAPES[shp]
        orc = Oracle(DecoderConfig(**shape, max_positions=256), inputs.make_weights(shape), mode="fp32")
        out[name] = run(orc, shape["vocab"], n_prompt, 0, None, dctx,
                        [_filled_cache(orc, orc.cfg, L, 64) for L in dctx])
    shape = inputs.SHAPES["qwen3_0p6b"]
    V = shape["vocab"]
    w = inputs.make_weights(shape)
    orc = Oracle(DecoderConfig(**shape, max_positions=512), w, mode="fp32")
    out["C3 qwen3-0.6B fp32"] = run(orc, V, 188, 0, None, [188], [_filled_cache(orc, orc.cfg, 188, 64)])
    del orc
    orc = Oracle(DecoderConfig(**shape, max_positions=4096 + 128), w, mode="bf16")
    del w
    lens = inputs.serving_context_lengths(32)
    pick = [lens[0], lens[-1]]
    caches = [_filled_cache(orc, orc.cfg, L, 64) for L in pick]
    c4 = run(orc, V, 64, 0, None, pick, caches)
    c4["sample"] += "; the serving contexts' shortest and longest"
    out["C4 qwen3-0.6B serving"] = c4
    del caches
    pre = _filled_cache(orc, orc.cfg, 3968, 160)
    out["C5 qwen3-0.6B chunked prefill"] = run(orc, V, 64, 3968, pre, [4032], [pre])
    for v in out.values():
        v["sample"] += "; caches of constant K/V where a context precedes"
    head = {"kind": "oracle", "cores": blas_threads(), "value": c4["decode_tokens_per_s"], "unit": "tokens/s",
            "sample": "float64 decode tokens of 2 of the 32 serving sequences, " + c4["sample"].split("decode: ")[1],
            "configs": out}
    return head


# One float64 decode token of the 0.6B shape costs about 0.09 s on a 16-core host.
ORACLE_TOKEN_S = 0.09


def reference_arm(args, rank, world):
    """The oracle as the reference arm: W untimed and K timed steps, a step
    being one float64 decode token for each of a sample of the 32 sequences
    (4, fewer when K + W is large, so the run stays near a minute)."""
    if rank != 0:
        return None
    n_sample = int(min(4, max(1, 60.0 / ((args.steps + args.warmup) * ORACLE_TOKEN_S))))
    orc, cfg, caches, pick = _oracle_sample(n_sample, args.warmup + args.steps)
    for i in range(args.warmup):
        _oracle_step(orc, cfg, caches, pick, i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_step(orc, cfg, caches, pick, args.warmup + i)
    dt = time.perf_counter() - t0
    v = n_sample * args.steps / max(dt, 1e-9)
    info = {"kind": "oracle", "cores": blas_threads(), "value": round(v, 3),
            "sample": f"{args.steps} timed float64 decode step(s) after {args.warmup} untimed, each one token "
                      f"for {n_sample} of the 32 sequences (contexts {pick}), caches filled with seeded random "
                      f"K/V; {dt:.1f} s"}
    return {"metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "batch": 32, "sampled_sequences": n_sample,
                       "parallelism": "host cores"},
            "cpu_baseline": info,
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
    else:
        line = our_arm(args, rank, world)
        if rank == 0 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baselines()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
