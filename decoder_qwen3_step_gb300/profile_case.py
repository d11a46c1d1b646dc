"""A bounded-size case of the serving decode (or prefill) step, for profilers.

Builds the Qwen3-0.6B-shaped decoder in the serving mode (bf16 weights, f16
KV), preloads `--batch` sequences of `--ctx` uniform-random tokens by
prefill (8,192 tokens per step), then runs `--steps` decode steps at that
batch, or `--steps` passes of a chunked prefill (`--case prefill`: `--batch`
sequences, 512-token chunks up to `--ctx`).  Sized to keep a profiler's
save/restore of device memory small (the default case holds about 5 GB).

    python -m decoder_qwen3_step_gb300.profile_case --case decode --batch 16 --ctx 2048 --steps 3
"""

from __future__ import annotations

import argparse
import sys

import torch

from . import dec, inputs
from .runtime import Decoder


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=["decode", "prefill"], default="decode")
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--ctx", type=int, default=2048)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--graphs", type=int, default=1)
    ap.add_argument("--range", action="store_true",
                    help="open a profiler range around the measured loop only (ncu --profile-from-start off)")
    args = ap.parse_args(argv)
    shape = inputs.SHAPES["qwen3_0p6b"]
    S, L = args.batch, args.ctx
    max_pos = ((L + args.steps + 16 + 15) // 16) * 16
    blocks = S * ((max_pos + 15) // 16) + 8
    m = Decoder(shape, inputs.make_weights(shape), mode=dec.DEC_BF16_F16KV, max_positions=max_pos, max_tokens=8192,
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
        torch.cuda.synchronize()
        if args.range:
            torch.cuda.cudart().cudaProfilerStart()
        for i in range(args.steps):
            m.decode([([0], L + i, tables[s]) for s in range(S)], device_ids=buf[i & 1], out=(logits, buf[(i + 1) & 1]))
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
