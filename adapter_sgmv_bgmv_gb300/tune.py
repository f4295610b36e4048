"""Offline shape -> launch-configuration search (VaLoRA blog, section 4.3.2: profile
every candidate tiling of each input shape offline, keep the best in a table that
the runtime looks up).

    python -m adapter_sgmv_bgmv_gb300.tune --shapes shapes.json --out tiles.tbl

Each shape is {"kind": "rows"|"tiles"|"merge", "n": rows, "d_in": .., "d_out": ..,
"rank": r, "adapters": distinct adapters, "run": rows per request (prefill)}.  The
inputs are random device tensors of that shape.

Two objectives:
  latency     the search runs in the library (`lora_tune_shape`): every candidate is
              timed call by call, each call started with L2 cold;
  throughput  (row-gather shapes, the default for them) every candidate is installed
              in the table and timed over back-to-back calls that rotate through
              copies of the adapters and inputs larger than L2, as a decode loop runs
              them: consecutive calls overlap (programmatic dependent launch), which
              the call-by-call timing cannot see.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import tempfile

import numpy as np
import torch

from . import (KIND_MERGE, KIND_ROWS_FUSED, KIND_TILE_FUSED, AdapterTable, Context,
               PreparedFused, lora_tune_shape)

# The shapes of the workloads this library is measured on.
DEFAULT_SHAPES = [
    {"kind": "rows", "n": 64, "d_in": 4096, "d_out": 4096, "rank": 16, "adapters": 64},
    {"kind": "rows", "n": 64, "d_in": 4096, "d_out": 4096, "rank": 16, "adapters": 1},
    {"kind": "rows", "n": 16, "d_in": 256, "d_out": 256, "rank": 8, "adapters": 4},
    {"kind": "rows", "n": 128, "d_in": 8192, "d_out": 8192, "rank": 16, "adapters": 72},
    {"kind": "rows", "n": 200, "d_in": 8192, "d_out": 8192, "rank": 16, "adapters": 100},
    {"kind": "tiles", "n": 5353, "d_in": 4096, "d_out": 4096, "rank": 64, "adapters": 8,
     "run": 670},
    {"kind": "tiles", "n": 16896, "d_in": 4096, "d_out": 11008, "rank": 64, "adapters": 4,
     "run": 1056},
    {"kind": "merge", "n": 1, "d_in": 4096, "d_out": 11008, "rank": 64, "adapters": 1},
]

KINDS = {"rows": KIND_ROWS_FUSED, "tiles": KIND_TILE_FUSED, "merge": KIND_MERGE}


def _bf16(shape, std, gen):
    return (torch.randn(shape, generator=gen, device="cuda") * std).to(torch.bfloat16)


def tune_shape(ctx: Context, spec: dict, iters: int = 20, seed: int = 0) -> float:
    gen = torch.Generator(device="cuda").manual_seed(seed)
    n, d_in, d_out, r = spec["n"], spec["d_in"], spec["d_out"], spec["rank"]
    na = spec["adapters"]
    a_pool = _bf16((na * r, d_in), 1 / math.sqrt(d_in), gen)
    b_pool = _bf16((na * r, d_out), 1 / math.sqrt(r), gen)
    pages = np.arange(na * r, dtype=np.int32).reshape(na, r)
    table = AdapterTable(ctx, a_pool, b_pool, np.full(na, r, np.int32),
                         np.full(na, 16.0 / r, np.float32), pages, pages)
    kind = KINDS[spec["kind"]]
    if kind == KIND_MERGE:
        W = _bf16((d_in, d_out), 1 / math.sqrt(d_in), gen)
        return lora_tune_shape(ctx, table, kind, np.zeros(1, np.int32), W, W, iters)
    if "run" in spec:
        ids = (np.arange(n) // spec["run"]) % na
    else:
        ids = np.arange(n) % na
    x = _bf16((n, d_in), 1.0, gen)
    y = _bf16((n, d_out), 1.0, gen)
    return lora_tune_shape(ctx, table, kind, ids.astype(np.int32), x, y, iters)


def _pow2(m: int) -> int:
    b = 1
    while b < m:
        b <<= 1
    return b


def tune_rows_throughput(ctx: Context, spec: dict, steps: int = 1500, seed: int = 0):
    """Best (cluster, rows per item, us per call) of a row-gather shape by throughput."""
    gen = torch.Generator(device="cuda").manual_seed(seed)
    n, d_in, d_out, r, na = spec["n"], spec["d_in"], spec["d_out"], spec["rank"], spec["adapters"]
    per_set = 2 * (na * r * (d_in + d_out) + n * (d_in + 2 * d_out))
    n_sets = max(2, math.ceil((256 << 20) / per_set))
    ids = (np.arange(n) % na).astype(np.int32)
    pages = np.arange(na * r, dtype=np.int32).reshape(na, r)
    calls = []
    for _ in range(n_sets):
        a_pool = _bf16((na * r, d_in), 1 / math.sqrt(d_in), gen)
        b_pool = _bf16((na * r, d_out), 1 / math.sqrt(r), gen)
        table = AdapterTable(ctx, a_pool, b_pool, np.full(na, r, np.int32),
                             np.full(na, 16.0 / r, np.float32), pages, pages)
        x = _bf16((n, d_in), 1.0, gen)
        y = _bf16((n, d_out), 1.0, gen)
        calls.append(PreparedFused(ctx, table, x, y))
    seg_max = n if na == 1 else math.ceil(n / na)
    key = f"0 {_pow2(n)} {_pow2(min(na, n))} {d_in} {d_out} {r}"
    best = None
    fd, path = tempfile.mkstemp(suffix=".tbl")
    os.close(fd)
    try:
        C = 1
        while C <= 16 and (C == 1 or min(d_in, d_out) // C >= 64):
            R = 1
            while R <= 16 and (R == 1 or R // 2 < seg_max):
                with open(path, "w") as fh:
                    fh.write(f"{key} {C} {R} 0 0\n")
                ctx.tiles_load(path)
                for i in range(20):
                    calls[i % n_sets](ids)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for i in range(steps):
                    calls[i % n_sets](ids)
                e1.record()
                torch.cuda.synchronize()
                us = 1000.0 * e0.elapsed_time(e1) / steps
                if best is None or us < best[2]:
                    best = (C, R, us)
                R *= 2
            C *= 2
        with open(path, "w") as fh:
            fh.write(f"{key} {best[0]} {best[1]} 0 0\n")
        ctx.tiles_load(path)
    finally:
        os.unlink(path)
    return best


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default=None, help="JSON list of shapes (default: built-in)")
    ap.add_argument("--out", required=True)
    ap.add_argument("--iters", type=int, default=31)
    ap.add_argument("--objective", choices=("throughput", "latency"), default="throughput",
                    help="row-gather shapes: back-to-back throughput (default) or cold latency")
    args = ap.parse_args()
    shapes = DEFAULT_SHAPES
    if args.shapes:
        with open(args.shapes) as fh:
            shapes = json.load(fh)
    ctx = Context(0, max_rows=1 << 15, max_rank=128)
    for spec in shapes:
        if spec["kind"] == "rows" and args.objective == "throughput":
            c, rr, us = tune_rows_throughput(ctx, spec)
            print(json.dumps({**spec, "objective": "throughput", "cluster": c, "rows": rr,
                              "us_per_call": round(us, 3)}), flush=True)
        else:
            us = tune_shape(ctx, spec, args.iters)
            print(json.dumps({**spec, "objective": "latency", "best_us": round(us, 3)}), flush=True)
    ctx.tiles_save(args.out)
    print(f"wrote {ctx.tiles_count()} entries to {args.out}")


if __name__ == "__main__":
    main()
