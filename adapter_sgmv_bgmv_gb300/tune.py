"""Offline shape -> launch-configuration search (VaLoRA blog, section 4.3.2: profile
every candidate tiling of each input shape offline, keep the best in a table that
the runtime looks up).  A thin caller of the library's `lora_tune`, which reads the
shape file, fills synthetic device buffers, runs the search and writes the table.

    python -m adapter_sgmv_bgmv_gb300.tune --out tiles.tbl [--shapes shapes.txt]

A shape file has one shape per line: ``kind n d_in d_out rank adapters [run
[objective]]`` (see include/lora.h).  Without --shapes the built-in list of the
workloads this library is measured on is used.  Two objectives:
  latency     every candidate is timed call by call, each call started with L2 cold;
  throughput  (row-gather shapes, the default for them here) every candidate is timed
              over back-to-back calls that rotate through copies of the adapters and
              inputs larger than L2, as a decode loop runs them: consecutive calls
              overlap (programmatic dependent launch), which the call-by-call timing
              cannot see.
The search runs with LORA_OPT_EARLY_PAGES and LORA_OPT_EARLY_INPUT on (the way a
decode loop of this library's calls runs, and the way bench.py measures); --no-early
tunes with both off.
"""
from __future__ import annotations

import argparse
import os
import tempfile

from . import OPT_EARLY_INPUT, OPT_EARLY_PAGES, Context

DEFAULT_SHAPES = """\
# kind   n      d_in  d_out  rank adapters run objective
rows     64     4096  4096   16   64       0   throughput
rows     64     4096  4096   16   1        0   throughput
rows     16     256   256    8    4        0   throughput
rows     128    8192  8192   16   72       0   throughput
rows     100    8192  8192   16   50       0   throughput
rows     64     8192  8192   16   40       0   throughput
rows     56     8192  8192   16   28       0   throughput
rows     32     8192  8192   16   24       0   throughput
rows     200    8192  8192   16   100      0   throughput
tiles    5353   4096  4096   64   8        670
tiles    16896  4096  11008  64   4        1056
merge    1      4096  11008  64   1
"""


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default=None, help="shape file (default: built-in list)")
    ap.add_argument("--out", required=True)
    ap.add_argument("--no-early", action="store_true",
                    help="tune with LORA_OPT_EARLY_PAGES and LORA_OPT_EARLY_INPUT off")
    args = ap.parse_args()
    ctx = Context(0, max_rows=1 << 15, max_rank=128)
    early = 0 if args.no_early else 1
    ctx.set_option(OPT_EARLY_PAGES, early)
    ctx.set_option(OPT_EARLY_INPUT, early)
    path = args.shapes
    tmp = None
    if path is None:
        fd, tmp = tempfile.mkstemp(suffix=".shapes")
        with os.fdopen(fd, "w") as fh:
            fh.write(DEFAULT_SHAPES)
        path = tmp
    try:
        ctx.tune(path, args.out)
    finally:
        if tmp:
            os.unlink(tmp)
    with open(args.out) as fh:
        print(fh.read(), end="")
    ctx.close()


if __name__ == "__main__":
    main()
