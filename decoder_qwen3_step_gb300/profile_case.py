"""A bounded-size case of the serving decode (or prefill) step, for profilers.

Builds the Qwen3-0.6B-shaped decoder in the serving mode (bf16 weights, f16
KV), preloads `--batch` sequences of `--ctx` uniform-random tokens by
prefill (8,192 tokens per step), then runs `--steps` decode steps at that
batch, or `--steps` passes of a chunked prefill (`--case prefill`: `--batch`
sequences, 512-token chunks up to `--ctx`).  Sized to keep a profiler's
save/restore of device memory small (the default case holds about 5 GB).

`--case sample` times the device sampler alone on `--batch` rows of seeded
logits at the Qwen3 vocabulary (normal, sigma 2.5), with 64 prompt and 32
output ids per row and the parameters `--sampling` names, and prints the
mean time per call over `--steps` calls (CUDA events, after 3 warm-up calls).

    python -m decoder_qwen3_step_gb300.profile_case --case decode --batch 16 --ctx 2048 --steps 3
    python -m decoder_qwen3_step_gb300.profile_case --case sample --batch 32 --sampling topk_topp --steps 50
"""

from __future__ import annotations

import argparse
import sys

import torch

import numpy as np

from . import dec, inputs
from .runtime import Decoder, DeviceHistory, Sampler, sampling_params

SAMPLINGS = {
    "greedy": dict(temperature=0.0),
    "topk_topp": dict(temperature=0.7, top_k=40, top_p=0.9),
    "topp": dict(temperature=1.0, top_p=0.95),
    "all": dict(temperature=0.8),
    "minp": dict(temperature=1.2, min_p=0.05),
}


def sample_case(S, which, steps, use_range):
    """Mean microseconds per dec_sample call on S rows of the Qwen3 vocabulary."""
    V = inputs.SHAPES["qwen3_0p6b"]["vocab"]
    g = np.random.default_rng(0)
    s = Sampler(V, S)
    x = torch.from_numpy(g.normal(0, 2.5, (S, V)).astype(np.float32)).cuda()
    hist = DeviceHistory([(list(g.integers(0, V, 64)), list(g.integers(0, V, 32))) for _ in range(S)])
    gen = s.streams(range(S))
    ps = [sampling_params(**SAMPLINGS[which])] * S
    tok = torch.empty(S, dtype=torch.int32, device="cuda")
    lp = torch.empty(S, dtype=torch.float64, device="cuda")
    for _ in range(3):
        s.sample(x, ps, hist, gen, out=(tok, lp))
    torch.cuda.synchronize()
    if use_range:
        torch.cuda.cudart().cudaProfilerStart()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        s.sample(x, ps, hist, gen, out=(tok, lp))
    b.record()
    torch.cuda.synchronize()
    if use_range:
        torch.cuda.cudart().cudaProfilerStop()
    status = s.status()
    s.close()
    if status:
        print(f"sampler status {status}", file=sys.stderr)
        return 1
    print(f"sample batch {S} {which}: {a.elapsed_time(b) / steps * 1000:.1f} us/call")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["decode", "prefill", "sample"], default="decode")
    ap.add_argument("--sampling", choices=sorted(SAMPLINGS), default="topk_topp")
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--ctx", type=int, default=2048)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--graphs", type=int, default=1)
    ap.add_argument("--mode", choices=["bf16", "int4"], default="bf16", help="weight format of the serving mode")
    ap.add_argument("--time", action="store_true", help="print the mean ms per measured step (CUDA events)")
    ap.add_argument("--range", action="store_true",
                    help="open a profiler range around the measured loop only (ncu --profile-from-start off)")
    args = ap.parse_args(argv)
    if args.case == "sample":
        return sample_case(args.batch, args.sampling, args.steps, args.range)
    shape = inputs.SHAPES["qwen3_0p6b"]
    S, L = args.batch, args.ctx
    max_pos = ((L + args.steps + 16 + 15) // 16) * 16
    blocks = S * ((max_pos + 15) // 16) + 8
    mode = dec.DEC_INT4_F16KV if args.mode == "int4" else dec.DEC_BF16_F16KV
    m = Decoder(shape, inputs.make_weights(shape), mode=mode, max_positions=max_pos, max_tokens=8192,
                max_seqs=max(S, 1), n_blocks=blocks)
    m.set_graphs(bool(args.graphs))
    tables = [m.blocks_for(max_pos) for _ in range(S)]
    ids = [inputs.make_ids(shape["vocab"], L, seed=300 + s) for s in range(S)]
    V = shape["vocab"]
    if args.case == "decode":
        per = max(1, 8192 // L)
        for g in range(0, S, per):
            m.prefill([(ids[s], 0, tables[s]) for s in range(g, min(S, g + per))], rows=dec.DEC_ROWS_LAST)
        logits = torch.empty((S, V), dtype=torch.float32, device=m.device)
        buf = [torch.zeros((S,), dtype=torch.int32, device=m.device) for _ in range(2)]
        for i in range(3 if args.time else 0):  # warm-up steps (graph capture) at the timed positions' shape
            m.decode([([0], L, tables[s]) for s in range(S)], device_ids=buf[0], out=(logits, buf[1]))
        torch.cuda.synchronize()
        if args.range:
            torch.cuda.cudart().cudaProfilerStart()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for i in range(args.steps):
            m.decode([([0], L + i, tables[s]) for s in range(S)], device_ids=buf[i & 1], out=(logits, buf[(i + 1) & 1]))
        ev[1].record()
        if args.time:
            torch.cuda.synchronize()
            ms = ev[0].elapsed_time(ev[1]) / args.steps
            print(f"decode {args.mode} batch {S} context {L}: {ms:.3f} ms/step, {S / ms * 1000:.0f} tokens/s")
    else:
        logits = torch.empty((S, V), dtype=torch.float32, device=m.device)
        am = torch.empty((S,), dtype=torch.int32, device=m.device)
        torch.cuda.synchronize()
        if args.range:
            torch.cuda.cudart().cudaProfilerStart()
        for _ in range(args.steps):
            for k in range(0, L, 512):
                m.prefill([(ids[s][k:k + 512], k, tables[s]) for s in range(S)], rows=dec.DEC_ROWS_LAST,
                          out=(logits, am))
    torch.cuda.synchronize()
    if args.range:
        torch.cuda.cudart().cudaProfilerStop()
    status = m.device_status()
    m.close()
    if status:
        print(f"device status {status}", file=sys.stderr)
        return 1
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
