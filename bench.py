#!/usr/bin/env python3
"""Throughput of the heterogeneous multi-LoRA delta on one GB300 (or N replicas).

Default workload (the line's headline): the VaLoRA-style vision prefill, the
largest configuration -- Qwen-VL-7B MLP up-projection 4096 -> 11008, 16 requests x
(1024 visual + 32 text) tokens, 4 rank-64 adapters with Zipf(1.2) popularity; one
step = one lora_fused call over the 16,896 tokens.  Inputs rotate over enough
device copies that one pass over them is several times the 129 MB L2, so every
step reads cold HBM.

The same JSON line carries `per_config`: every other workload measured in the same
run (tiny decode, the Llama-7B decode pair, S-LoRA prefill, the VaLoRA merge +
unmerge, the LoRazor active-row decode with its microseconds-vs-active-rows curve),
each with device and host microseconds per call, tokens/s, the dominant kernel's
fraction of its roofline, the end-to-end rate and the oracle's rate on the host.

`--impl reference` times the CPU oracle instead, on a bounded sample of the same
workload.  `--all` prints one line per workload.  `--config NAME` makes NAME the
headline.
"""
from __future__ import annotations

import argparse
import ctypes
import ctypes.util
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = ("multi-LoRA delta tokens/s and µs/call; % of HBM (decode) / TC (prefill) "
          "roofline")
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DEFAULT_CONFIG = "valora_prefill"
CONFIGS = ("valora_prefill", "llama7b_decode", "tiny_decode", "slora_prefill", "valora_merge",
           "lorazor_decode", "valora_base_fused")
DEVICE_IDS_CONFIGS = ("llama7b_decode", "tiny_decode", "lorazor_decode")
# Steps of a per_config entry (a fixed count, independent of --steps, sized so that
# each timed region is a few tens to a few hundred milliseconds).
PER_CONFIG_STEPS = {"llama7b_decode": 10000, "tiny_decode": 20000, "lorazor_decode": 10000,
                    "slora_prefill": 2000, "valora_prefill": 500, "valora_merge": 1000,
                    "valora_base_fused": 200}
WORKLOAD_DESC = {
    "valora_prefill": ("Qwen-VL-7B MLP up-proj 4096->11008, 16 requests x (1024 visual + 32 "
                       "text) tokens = 16896, 4 rank-64 adapters (Zipf 1.2), contiguous storage"),
    "llama7b_decode": ("Llama-7B projection 4096x4096, 64 requests x 1 token, rank 16; per step "
                       "one call with 64 distinct adapters (heterogeneous) + one call with all "
                       "rows on one adapter (homogeneous)"),
    "tiny_decode": "d=256, 16 requests x 1 token, 4 rank-8 adapters, contiguous storage",
    "slora_prefill": ("S-LoRA prefill 4096x4096, 8 requests with log-normal lengths (5353 "
                      "tokens), ranks in {8,16,32,64}, 8 of 1000 adapters resident in shuffled "
                      "4096-wide pages"),
    "valora_merge": "merge then unmerge of a rank-64 adapter into W 4096x11008 bf16",
    "lorazor_decode": ("70B projection 8192x8192, 256 requests x 1 token, 512 resident rank-16 "
                       "adapters (Zipf 1.0) in shuffled 8192-wide pages; step t releases 128+t "
                       "rows (t = 0..99, cycled)"),
    "valora_base_fused": ("the VaLoRA prefill through the base projection with the adapter term "
                          "fused in: y = x W + s (x A) B, W 4096x11008 bf16, 16896 tokens, 4 "
                          "rank-64 adapters (Zipf 1.2); y written once"),
}
# Source files of each kernel family: a DRAM-traffic figure measured by ncu holds only
# while their contents are those it was measured on.
FAMILY_SOURCES = {
    "rows": ["rows.cu", "ptx.cuh"],
    "shrink": ["tile_tc.cu", "dense.cu", "tc.cuh"],
    "expand": ["stream_tc.cu", "tc.cuh"],
    "merge": ["stream_tc.cu", "tc.cuh"],
    "proj": ["proj_tc.cu", "tc.cuh"],
}
KERNEL_NAMES = {"rows": "k_rows_inline<fused>", "shrink": "k_shrink_tc (+ k_stage_rows)",
                "expand": "k_stream_tc(expand)", "merge": "k_stream_tc(merge)",
                "proj": "k_proj_tc (base GEMM + adapter term, + k_proj_prep)"}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def config_for(name: str, early_pages: bool = True, device_ids: bool = False,
               early_input: bool = True) -> dict:
    """The line's `config` (the same dict for both arms: a function of the workload)."""
    return {"workload": WORKLOAD_DESC[name], "name": name,
            "l2": "inputs rotate over device copies; one pass touches more than 3 x the "
                  "129 MB L2 (no flush needed)",
            "parallelism": "single GPU (replicas under torchrun)",
            "early_pages": bool(early_pages), "early_input": bool(early_input),
            "device_ids": bool(device_ids)}


# --------------------------------------------------------------------------- peaks

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        hbm = float(d.get("hbm_gbs") or d.get("hbm_GBps"))
        tc = float(d.get("bf16_tflops"))
        tcs = float(d.get("bf16_tflops_sustained", tc))
        return {"hbm_gbs": hbm, "bf16_tflops": tc, "bf16_tflops_sustained": tcs,
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def source_sha(family: str) -> str:
    h = hashlib.sha256()
    for f in FAMILY_SOURCES.get(family, []):
        with open(os.path.join(ROOT, "adapter_sgmv_bgmv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(name: str, family: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of this
    workload's kernel family from the ncu figures kept in the traffic file, or None
    when there is none or the kernel's sources changed since it was measured."""
    try:
        with open(TRAFFIC_FILE) as fh:
            for line in fh:
                f = line.split("#", 1)[0].split()
                if len(f) >= 4 and f[0] == name and f[1] == family:
                    return float(f[2]) if f[3] == source_sha(family) else None
    except OSError:
        pass
    return None


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock, its maximum, power and the clock-event (throttle) reasons of this
    GPU, read through NVML in this process every half millisecond while sampling is
    on, so that even a timed region of a few milliseconds has samples; falls back to
    nvidia-smi at 200 ms when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, index: int):
        self.rows = []                # (t, sm_mhz, max_mhz, reasons bitmask, power W)
        self.lib = self.dev = None
        self.on = threading.Event()
        self.stop_ev = threading.Event()
        self.proc = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            dev = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(index).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) != 0:
                cnt = ctypes.c_uint()
                if lib.nvmlDeviceGetCount_v2(ctypes.byref(cnt)) != 0 or cnt.value != 1 or \
                        lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(dev)) != 0:
                    raise OSError("no NVML handle for this GPU")
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.lib, self.dev = lib, dev
            self.max_mhz = self._clock(lib.nvmlDeviceGetMaxClockInfo)
        except Exception:
            self.lib = None
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _clock(self, fn):
        v = ctypes.c_uint()
        return v.value if fn(self.dev, 1, ctypes.byref(v)) == 0 else None   # 1: SM clock

    def _sample(self):
        sm = self._clock(self.lib.nvmlDeviceGetClockInfo)
        r = ctypes.c_ulonglong()
        reasons = r.value if self.reason_fn(self.dev, ctypes.byref(r)) == 0 else 0
        p = ctypes.c_uint()
        power = p.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(p)) == 0 else None
        self.rows.append((time.perf_counter(), sm, self.max_mhz, reasons, power))

    def _run(self):
        if self.lib is None:
            self._run_smi()
            return
        while not self.stop_ev.is_set():
            if self.on.wait(0.05):
                self._sample()
                time.sleep(0.0005)

    def _run_smi(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        bits = (0x8, 0x40, 0x20, 0x4)
        for line in self.proc.stdout:
            p = [x.strip() for x in line.split(",")]
            if len(p) < 7:
                continue
            try:
                mask = sum(b for b, v in zip(bits, p[3:7]) if v.lower().startswith("active"))
                self.rows.append((time.perf_counter(), float(p[0]), float(p[1]), mask,
                                  float(p[2]) if p[2].replace(".", "", 1).isdigit() else None))
            except ValueError:
                continue

    def start(self):
        """Begin sampling: one sample now (in this thread, so that even a region
        shorter than the thread's first turn has one), then every half millisecond."""
        if self.lib is not None:
            self._sample()
        self.on.set()

    def pause(self):
        """Stop sampling, with one last sample taken now, at the region's end."""
        self.on.clear()
        if self.lib is not None:
            self._sample()

    def close(self):
        self.stop_ev.set()
        self.on.set()
        if self.proc is not None:
            self.proc.terminate()
        self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        win = [r for r in self.rows if t0 <= r[0] <= t1]
        src = "nvml" if self.lib is not None else "nvidia-smi"
        if not win:
            # a region shorter than the sampling period: the samples nearest to it
            near = sorted(self.rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:4]
            if not near:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"],
                        "samples": 0, "source": src}
            out = self._stats(near)
            out.update(in_timed_window=False, source=src)
            return out
        out = self._stats(win)
        out.update(in_timed_window=True, source=src)
        return out

    def _stats(self, rows):
        sm = [r[1] for r in rows if r[1] is not None]
        mx = [r[2] for r in rows if r[2] is not None]
        pw = [r[4] for r in rows if r[4] is not None]
        reasons = sorted({name for r in rows for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# --------------------------------------------------------------------------- algorithmic bytes

def alg_bytes_delta(case, ids):
    """Algorithmic bytes of one fused call: x read, y read + write, the A and B pages
    of every distinct active adapter, and the plan (items + permutation)."""
    ids = np.asarray(ids)
    act = ids[ids >= 0]
    n_act = int(act.size)
    d_in, d_out = case["d_in"], case["d_out"]
    distinct = np.unique(act)
    ab = int(sum(2 * int(case["rank"][k]) * (d_in + d_out) for k in distinct))
    return 2 * n_act * d_in + 4 * n_act * d_out + ab + 4 * n_act + 16 * len(distinct)


def alg_bytes_split(case, ids, tiles: bool) -> dict:
    """alg_bytes_delta split by the kernel family that moves each part: on the tile
    path the shrink reads x and the A pages, the expand reads and writes y and reads
    the B pages; on the row-gather path one kernel does all of it."""
    ids = np.asarray(ids)
    act = ids[ids >= 0]
    n_act = int(act.size)
    d_in, d_out = case["d_in"], case["d_out"]
    distinct = np.unique(act)
    a_b = int(sum(2 * int(case["rank"][k]) * d_in for k in distinct))
    b_b = int(sum(2 * int(case["rank"][k]) * d_out for k in distinct))
    plan = 4 * n_act + 16 * len(distinct)
    if tiles:
        return {"shrink": 2 * n_act * d_in + a_b + plan, "expand": 4 * n_act * d_out + b_b}
    return {"rows": 2 * n_act * d_in + 4 * n_act * d_out + a_b + b_b + plan}


def flops_delta(case, ids):
    ids = np.asarray(ids)
    act = ids[ids >= 0]
    return int(sum(2 * int(case["rank"][k]) * (case["d_in"] + case["d_out"]) for k in act))


# --------------------------------------------------------------------------- workload on the device

class Bench:
    """Device-resident rotating copies of one workload and the per-step calls."""

    def __init__(self, name: str, L, torch, ctx, device_ids: bool = False):
        self.name, self.L, self.torch, self.ctx = name, L, torch, ctx
        if device_ids and name not in DEVICE_IDS_CONFIGS:
            raise ValueError(f"--device-ids applies to the decode workloads {DEVICE_IDS_CONFIGS}")
        # decode through lora_fused_device_ids: every set holds its steps' ids in
        # device memory (the end-to-end loop copies them in with the step's inputs)
        self.device_ids = device_ids
        if name == "llama7b_decode":
            het = workloads.make("llama7b_decode_het", seed=0)
            hom = workloads.make("llama7b_decode_hom", seed=0)
            self.cases = {"het": het, "hom": hom}
            self.steps_ids = [[("het", het["ids"]), ("hom", hom["ids"])]]
        elif name == "lorazor_decode":
            c = workloads.make("lorazor_decode", seed=0)
            self.cases = {"main": c}
            self.steps_ids = [[("main", workloads.lorazor_ids(c, t))] for t in range(100)]
        elif name in ("tiny_decode", "slora_prefill", "valora_prefill"):
            c = workloads.make(name, seed=0)
            self.cases = {"main": c}
            self.steps_ids = [[("main", c["ids"])]]
        elif name == "valora_base_fused":
            c = workloads.make("valora_prefill", seed=0)
            c["W"] = workloads.make_W(c["d_in"], c["d_out"], seed=0)
            self.cases = {"main": c}
            self.steps_ids = [[("main", c["ids"])]]
        elif name == "valora_merge":
            c = workloads.make("valora_merge", seed=0)
            self.cases = {"main": c}
            self.steps_ids = None
        else:
            raise KeyError(name)
        self.workload = WORKLOAD_DESC[name]
        self.is_merge = name == "valora_merge"
        self.is_proj = name == "valora_base_fused"
        self._upload()

    # ---- device data, rotated so that one pass over the sets exceeds L2
    def _unique_bytes_per_step(self):
        if self.is_merge:
            c = self.cases["main"]
            return 2 * c["d_in"] * c["d_out"]
        if self.is_proj:
            c = self.cases["main"]
            return 2 * c["n"] * (c["d_in"] + c["d_out"]) + 2 * c["d_in"] * c["d_out"]
        return sum(alg_bytes_delta(self.cases[key], ids) for key, ids in self.steps_ids[0])

    def _upload(self):
        torch, L = self.torch, self.L
        from tests.gpu_util import to_dev
        per = max(1, self._unique_bytes_per_step())
        # enough sets that a pass touches > 3 x L2, and at least two, so that the end
        # to end loop can copy one step's inputs in while the previous result is read
        # back (a set is refilled only after its result has left the device)
        self.n_sets = int(min(32, max(2, math.ceil(3 * L2_BYTES / per))))
        self.sets = []
        base = {}
        for key, c in self.cases.items():
            d = {"a_pool": to_dev(c["a_pool"])}
            d["b_pool"] = d["a_pool"] if c["b_pool"] is c["a_pool"] else to_dev(c["b_pool"])
            if self.is_merge:
                d["W"] = to_dev(c["W"])
            else:
                d["x"] = to_dev(c["x"])
                d["y"] = to_dev(c["y"])
                if self.is_proj:
                    d["W"] = to_dev(c["W"])
            base[key] = d
        # Per set, the step's activations sit in one block, every x first and every y
        # after it, so that the end-to-end loop copies a step in with one copy and
        # reads its result back with another.
        keys = list(self.cases)
        fields = [] if self.is_merge else [(k, "x") for k in keys] + [(k, "y") for k in keys]
        self.blk_elems = sum(base[k][f].numel() for k, f in fields)
        self.y_offset = sum(base[k]["x"].numel() for k in keys) if not self.is_merge else 0
        for s in range(self.n_sets):
            st = {}
            blk = torch.empty(max(1, self.blk_elems), dtype=torch.bfloat16, device="cuda")
            views, off = {}, 0
            for k, f in fields:
                t = base[k][f]
                views[(k, f)] = blk[off:off + t.numel()].view(t.shape)
                views[(k, f)].copy_(t)
                off += t.numel()
            for key, c in self.cases.items():
                b = base[key]
                if s == 0:
                    d = {"a_pool": b["a_pool"], "b_pool": b["b_pool"]}
                else:
                    d = {"a_pool": b["a_pool"].clone()}
                    d["b_pool"] = d["a_pool"] if b["b_pool"] is b["a_pool"] else b["b_pool"].clone()
                if self.is_merge:
                    d["W"] = b["W"] if s == 0 else b["W"].clone()
                else:
                    d["x"], d["y"] = views[(key, "x")], views[(key, "y")]
                    if self.is_proj:
                        d["W"] = b["W"] if s == 0 else b["W"].clone()
                d["table"] = L.AdapterTable(self.ctx, d["a_pool"], d["b_pool"], c["rank"],
                                            c["scale"], c["a_pages"], c["b_pages"])
                if not self.is_merge and not self.is_proj:
                    prep = L.PreparedFusedDeviceIds if self.device_ids else L.PreparedFused
                    d["call"] = prep(self.ctx, d["table"], d["x"], d["y"],
                                     torch.cuda.current_stream())
                st[key] = d
            if self.device_ids:
                for t, calls in enumerate(self.steps_ids):
                    for key, ids in calls:
                        st[("ids", t, key)] = torch.from_numpy(
                            np.ascontiguousarray(ids, np.int32)).cuda()
            st["_blk"] = blk
            self.sets.append(st)
        # every set's call holds the arguments of every step before the first one, so
        # that no argument conversion falls inside a timed region
        if not self.is_merge and not self.is_proj:
            for st in self.sets:
                for t, calls in enumerate(self.steps_ids):
                    for key, ids in calls:
                        st[key]["call"].bind(st[("ids", t, key)] if self.device_ids else ids)
        torch.cuda.synchronize()

    # ---- one step
    def step(self, i: int, stream):
        L = self.L
        st = self.sets[i % self.n_sets]
        if self.is_merge:
            d = st["main"]
            k = self.cases["main"]["merge_adapter"]
            L.lora_merge(self.ctx, d["table"], k, d["W"], stream)
            L.lora_unmerge(self.ctx, d["table"], k, d["W"], stream)
            return
        t = i % len(self.steps_ids)
        for key, ids in self.steps_ids[t]:
            self._call(st, t, key, ids, stream)

    def step_on(self, set_idx: int, t: int, stream):
        """The calls of step t (its ids) on device set set_idx."""
        st = self.sets[set_idx % self.n_sets]
        for key, ids in self.steps_ids[t]:
            self._call(st, t, key, ids, stream)

    def _call(self, st, t, key, ids, stream):
        if self.is_proj:
            d = st[key]
            self.L.lora_base_fused(self.ctx, d["table"], ids, d["x"], d["W"], d["y"], stream)
        elif self.device_ids:
            st[key]["call"](st[("ids", t, key)])
        else:
            st[key]["call"](ids)

    def one_call(self, i: int, key: str, stream):
        """One library call of step i's case `key` (merge: the merge alone)."""
        st = self.sets[i % self.n_sets]
        if self.is_merge:
            d = st["main"]
            self.L.lora_merge(self.ctx, d["table"], self.cases["main"]["merge_adapter"], d["W"],
                              stream)
            return
        t = i % len(self.steps_ids)
        for k, ids in self.steps_ids[t]:
            if k == key:
                self._call(st, t, k, ids, stream)

    def call_keys(self):
        return ["merge"] if self.is_merge else [k for k, _ in self.steps_ids[0]]

    def tokens_per_step(self, i: int) -> int:
        if self.is_merge:
            return 0
        return sum(int((np.asarray(ids) >= 0).sum()) for _, ids in self.steps_ids[i % len(self.steps_ids)])

    def calls_per_step(self) -> int:
        """Library calls per step (a tile-path call launches two or three kernels)."""
        return 2 if (self.is_merge or self.name == "llama7b_decode") else 1

    def alg_bytes_step(self, i: int) -> int:
        if self.is_merge:
            c = self.cases["main"]
            r = int(c["rank"][c["merge_adapter"]])
            return 2 * (4 * c["d_in"] * c["d_out"] + 2 * r * (c["d_in"] + c["d_out"]))
        return sum(alg_bytes_delta(self.cases[k], ids) for k, ids in self.steps_ids[i % len(self.steps_ids)])

    def learn_paths(self, stream):
        """Which kernels each call of a step runs (one untimed call per case)."""
        self.paths = {}
        if self.is_merge:
            return
        for key, ids in self.steps_ids[0]:
            self._call(self.sets[0], 0, key, ids, self.torch.cuda.current_stream())
            self.paths[key] = self.ctx.last_path()[0]
        self.torch.cuda.synchronize()

    def alg_bytes_family(self, i: int) -> dict:
        if self.is_merge:
            return {"merge": self.alg_bytes_step(i)}
        if self.is_proj:
            c = self.cases["main"]
            ids = np.asarray(self.steps_ids[0][0][1])
            sp = alg_bytes_split(c, ids, True)
            n, d_in, d_out = c["n"], c["d_in"], c["d_out"]
            b_pages = sp["expand"] - 4 * int((ids >= 0).sum()) * d_out
            return {"shrink": sp["shrink"],
                    "proj": 2 * n * d_in + 2 * d_in * d_out + 2 * n * d_out + b_pages}
        out = {}
        for k, ids in self.steps_ids[i % len(self.steps_ids)]:
            tiles = bool(self.paths.get(k, 1) & 2) and not (self.paths.get(k, 1) & 1)
            for f, v in alg_bytes_split(self.cases[k], ids, tiles).items():
                out[f] = out.get(f, 0) + v
        return out

    def flops_family(self, i: int) -> dict:
        """Algorithmic flops per kernel family (the adapter term once, though the
        tensor cores run it on both halves of s v)."""
        if self.is_proj:
            c = self.cases["main"]
            ids = np.asarray(self.steps_ids[0][0][1])
            act = ids[ids >= 0]
            r = np.asarray(c["rank"])[act].astype(np.int64)
            return {"shrink": int(2 * r.sum() * c["d_in"]),
                    "proj": int(2 * c["n"] * c["d_in"] * c["d_out"] + 2 * r.sum() * c["d_out"])}
        return {}

    def flops_step(self, i: int) -> int:
        if self.is_proj:
            return sum(self.flops_family(i).values())
        if self.is_merge:
            c = self.cases["main"]
            r = int(c["rank"][c["merge_adapter"]])
            return 2 * 2 * c["d_in"] * c["d_out"] * r
        return sum(flops_delta(self.cases[k], ids) for k, ids in self.steps_ids[i % len(self.steps_ids)])

    # ---- end to end through host buffers
    def e2e_setup(self):
        """Pinned host copies of a step's inputs (one block, laid out as on the
        device), per device set a pinned result buffer and three events, and two
        copy streams.  The loop issues its copies and event operations through the
        CUDA runtime with arguments built here, so a step costs the host little more
        than the library calls themselves."""
        torch = self.torch
        if self.is_merge:
            w = self.cases["main"]["W"]
            self.host_in = torch.from_numpy(w.view(np.int16).reshape(-1)).pin_memory()
            self.out_elems = w.size
        else:
            # the step's inputs: x, and y where the call updates it in place (the base
            # projection only writes y, so it copies x in alone)
            parts = [self.cases[k]["x"] for k in self.cases]
            if not self.is_proj:
                parts += [self.cases[k]["y"] for k in self.cases]
            self.host_in = torch.from_numpy(
                np.concatenate([p.view(np.int16).reshape(-1) for p in parts])).pin_memory()
            self.out_elems = self.blk_elems - self.y_offset
        self.host_out = [torch.empty(self.out_elems, dtype=torch.int16).pin_memory()
                         for _ in range(self.n_sets)]
        if self.device_ids:
            self.host_ids = {(t, key): torch.from_numpy(np.ascontiguousarray(ids, np.int32)).pin_memory()
                             for t, calls in enumerate(self.steps_ids) for key, ids in calls}
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        rt = _runtime()
        self.rt = rt
        V, S = ctypes.c_void_p, ctypes.c_size_t
        in_bytes, out_bytes = self.host_in.numel() * 2, self.out_elems * 2
        s_in, s_out = V(self.s_in.cuda_stream), V(self.s_out.cuda_stream)
        s_comp = V(torch.cuda.current_stream().cuda_stream)
        self.e2e_ops = []
        for k in range(self.n_sets):
            ev = []
            for _ in range(3):
                e = V()
                _rt_check(rt.cudaEventCreateWithFlags(ctypes.byref(e), 2))   # no timing
                ev.append(e)
            blk = self._dev_block(self.sets[k])
            dev_in, dev_out = V(blk.data_ptr()), V(blk.data_ptr() + 2 * self.y_offset)
            self.e2e_ops.append({
                "refill_wait": (s_in, ev[2], 0),
                "copy_in": (dev_in, V(self.host_in.data_ptr()), S(in_bytes), 1, s_in),
                "rec_in": (ev[0], s_in), "wait_in": (s_comp, ev[0], 0),
                "rec_c": (ev[1], s_comp), "wait_c": (s_out, ev[1], 0),
                "copy_out": (V(self.host_out[k].data_ptr()), dev_out, S(out_bytes), 2, s_out),
                "rec_out": (ev[2], s_out), "drain": (s_comp, ev[2], 0)})
        self.used = [False] * self.n_sets
        self.e2e_bytes = (in_bytes, out_bytes)

    def _dev_block(self, st):
        if self.is_merge:
            return st["main"]["W"]
        return st["_blk"]

    def e2e_step(self, i: int, stream):
        """One step end to end, pipelined with its neighbours: step i's inputs are
        copied in on one stream while step i-1 computes and step i-2's result is read
        back on another.  A device set is refilled only after its previous result
        has been read back."""
        k = i % self.n_sets
        st, op, rt = self.sets[k], self.e2e_ops[k], self.rt
        if self.used[k]:
            _rt_check(rt.cudaStreamWaitEvent(*op["refill_wait"]))
        self.used[k] = True
        _rt_check(rt.cudaMemcpyAsync(*op["copy_in"]))
        t = 0 if self.is_merge else i % len(self.steps_ids)
        if self.device_ids:
            for key, _ in self.steps_ids[t]:
                dev, host = st[("ids", t, key)], self.host_ids[(t, key)]
                _rt_check(rt.cudaMemcpyAsync(ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.data_ptr()),
                                             ctypes.c_size_t(4 * host.numel()), 1, op["copy_in"][4]))
        _rt_check(rt.cudaEventRecord(*op["rec_in"]))
        _rt_check(rt.cudaStreamWaitEvent(*op["wait_in"]))
        h2d = self.e2e_bytes[0]
        if self.is_merge:
            d = st["main"]
            a = self.cases["main"]["merge_adapter"]
            self.L.lora_merge(self.ctx, d["table"], a, d["W"], stream)
            self.L.lora_unmerge(self.ctx, d["table"], a, d["W"], stream)
        else:
            for key, ids in self.steps_ids[t]:
                self._call(st, t, key, ids, stream)
                h2d += 4 * len(ids)
        _rt_check(rt.cudaEventRecord(*op["rec_c"]))
        _rt_check(rt.cudaStreamWaitEvent(*op["wait_c"]))
        _rt_check(rt.cudaMemcpyAsync(*op["copy_out"]))
        _rt_check(rt.cudaEventRecord(*op["rec_out"]))
        return h2d, self.e2e_bytes[1]

    def e2e_drain(self, stream):
        """Make the compute stream wait for every read-back issued so far."""
        for k in range(self.n_sets):
            if self.used[k]:
                _rt_check(self.rt.cudaStreamWaitEvent(*self.e2e_ops[k]["drain"]))

    def release(self):
        self.sets = []
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


class _RuntimeFns:
    pass


_RT = None


def _runtime():
    """The CUDA runtime's copy / event / stream-wait entry points, each a foreign
    function without argument types (called with ready-made ctypes objects)."""
    global _RT
    if _RT is not None:
        return _RT
    cands = ["/usr/local/cuda/lib64/libcudart.so", ctypes.util.find_library("cudart")]
    cands += sorted(glob.glob(os.path.join(os.path.dirname(np.__file__), "..", "nvidia", "*", "lib",
                                           "libcudart.so*")))
    for path in cands:
        if path and os.path.exists(path):
            lib = ctypes.CDLL(path)
            break
    else:
        raise RuntimeError("no CUDA runtime library found for the end-to-end loop")
    rt = _RuntimeFns()
    for name in ("cudaMemcpyAsync", "cudaEventRecord", "cudaStreamWaitEvent",
                 "cudaEventCreateWithFlags"):
        fn = lib._FuncPtr((name, lib))
        fn.restype = ctypes.c_int
        setattr(rt, name, fn)
    _RT = rt
    return rt


def _rt_check(rc: int):
    if rc != 0:
        raise RuntimeError(f"CUDA runtime call failed with error {rc}")


# --------------------------------------------------------------------------- oracle leg

def oracle_sample(name: str, budget_s: float, nthreads: int):
    """Time the CPU oracle on a bounded sample of the workload: whole calls of the
    step (or rows of them) until about `budget_s` seconds have been spent.
    Returns (tokens or calls processed, seconds, sample description)."""
    import oracle
    if name == "valora_merge":
        c = workloads.make("valora_merge", seed=0)
        t = oracle.Table.from_case(c)
        rows_per = 16
        done = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            rows = np.arange(done, done + rows_per) % c["d_in"]
            oracle.merge(t, c["merge_adapter"], c["W"], +1, nthreads=nthreads, rows=rows)
            done += rows_per
        dt = time.perf_counter() - t0
        # one call = all d_in rows of W
        return done / c["d_in"], dt, f"merge of {done} W rows (of {c['d_in']} per call)"
    if name == "valora_base_fused":
        c = workloads.make("valora_prefill", seed=0)
        W = workloads.make_W(c["d_in"], c["d_out"], seed=0)
        t = oracle.Table.from_case(c)
        done, chunk = 0, 512
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            rows = np.arange(done, done + chunk) % c["n"]
            oracle.base_fused(t, c["ids"], c["x"], W, nthreads=nthreads, rows=rows)
            done += chunk
        dt = time.perf_counter() - t0
        return done, dt, f"{done} rows of the base projection with the adapter term, {chunk}-row chunks"
    if name == "llama7b_decode":
        parts = [workloads.make("llama7b_decode_het", seed=0),
                 workloads.make("llama7b_decode_hom", seed=0)]
    elif name == "lorazor_decode":
        c = workloads.make("lorazor_decode", seed=0)
        parts = [dict(c, ids=workloads.lorazor_ids(c, 0))]
    else:
        parts = [workloads.make(name, seed=0)]
    tables = [oracle.Table.from_case(p) for p in parts]
    done_tok = 0
    t0 = time.perf_counter()
    chunk = 64
    q = 0
    while time.perf_counter() - t0 < budget_s:
        p, t = parts[q % len(parts)], tables[q % len(parts)]
        act = np.flatnonzero(p["ids"] >= 0)
        start = (q // len(parts)) * chunk % max(1, len(act))
        rows = act[start:start + chunk]
        oracle.fused_rows(t, p["ids"], p["x"], p["y"], rows, nthreads=nthreads)
        done_tok += len(rows)
        q += 1
    dt = time.perf_counter() - t0
    return done_tok, dt, f"{done_tok} active rows of the workload's calls, {chunk}-row chunks"


# --------------------------------------------------------------------------- measurement

def _events(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def measure(name, K, W, args, L, torch, ctx, dist, world, local, clocks, cpu_budget,
            extras: bool):
    """Time K steps of one workload (after W warm-up steps) and gather the figures of
    its JSON entry.  extras: repeats, single-call latencies, the LoRazor curve."""
    b = Bench(name, L, torch, ctx, device_ids=args.device_ids)
    stream = torch.cuda.current_stream()
    for i in range(W):
        b.step(i, stream)
    b.learn_paths(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ev0, ev1 = _events(torch)
    n_launch0 = ctx.launch_count()
    t_s0 = time.perf_counter()
    clocks.start()
    t0 = time.perf_counter()
    ev0.record(stream)
    for i in range(K):
        b.step(W + i, stream)
    t_enq = time.perf_counter()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    clocks.pause()
    t_s1 = time.perf_counter()
    n_launched = ctx.launch_count() - n_launch0
    ms = ev0.elapsed_time(ev1)
    calls = K * b.calls_per_step()
    host_enqueue_us = 1e6 * (t_enq - t0) / max(1, calls)
    clk = clocks.summary(t_s0, t_s1)   # the region and the samples at its two edges
    # The per-family split comes from a second pass over the same steps with the
    # profiler on, outside the timed region: a bracketed launch loses its overlap
    # with its neighbours, which would otherwise slow the timed steps themselves.
    ctx.profile_begin(args.profile_every)
    for i in range(K):
        b.step(W + i, stream)
    torch.cuda.synchronize()
    prof = ctx.profile_end()
    tokens_local = sum(b.tokens_per_step(W + i) for i in range(K))
    ms, tokens_all, _ = aggregate_ranks(ms, tokens_local, dist, "cuda")
    pk = peaks()
    # Per kernel family: launches, device time, algorithmic bytes it moves and the
    # rate.  The profiling pass brackets one launch in `profile_every` per family
    # with events; a bracket costs the launch its overlap with its neighbours (they
    # are launched as programmatic dependents), so the bracketed times serve only to
    # split the timed region's device time between the families.  A family's
    # average launch duration is its share of the region divided by its launches
    # (for a one-family workload: region time / launches).  Every kernel of the
    # path is HBM-bound; the roofline line is that of the family with the most time.
    fam_bytes = {}
    for i in range(K):
        for f, v in b.alg_bytes_family(W + i).items():
            fam_bytes[f] = fam_bytes.get(f, 0) + v
    fam_flops = {}
    for i in range(K):
        for f, v in b.flops_family(W + i).items():
            fam_flops[f] = fam_flops.get(f, 0) + v
    sec = ms / 1e3
    # The base projection is a dense contraction: its roofline is the bf16 tensor
    # peak (the sustained figure once the timed region runs for a quarter second or
    # more, the burst figure below that); every other family is bound by HBM.
    tc_peak = pk["bf16_tflops_sustained"] if sec >= 0.25 else pk["bf16_tflops"]
    tc_src = "bf16_tflops_sustained" if sec >= 0.25 else "bf16_tflops"
    bracketed = sum(m for (m, n) in prof.values() if n)
    n_fams = sum(1 for (m, n) in prof.values() if n and m > 0)
    per_family = {}
    for f, (m, n) in prof.items():
        if n and m > 0:
            share_s = sec * (m / bracketed)
            # A launch's duration.  One kernel family: the region over its launches
            # (consecutive launches overlap, and that is the rate they sustain).
            # Several: each launch as timed alone by the events around it.  The
            # families' launches overlap one another by an amount nothing measures, so
            # the region is not divided between them; the bracketed time is the
            # conservative figure (it includes the launch's own ramp, unhidden).
            dur_s = share_s / n if n_fams == 1 else m / 1e3 / n
            gbs = fam_bytes.get(f, 0) / n / dur_s / 1e9
            e = {"kernel": KERNEL_NAMES[f], "launches": n,
                 "us_per_launch": round(1e6 * dur_s, 3),
                 "us_per_launch_bracketed": round(1e3 * m / n, 3),
                 "us_per_launch_share_of_region": round(1e6 * share_s / n, 3),
                 "alg_bytes_per_launch": fam_bytes.get(f, 0) / n,
                 "GB/s": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4), "bound": "hbm",
                 "traffic": None if b.device_ids else measured_traffic(name, f)}
            if f == "proj":
                tf = fam_flops.get(f, 0) / n / dur_s / 1e12
                e.update({"bound": "tensor", "alg_flops_per_launch": fam_flops.get(f, 0) / n,
                          "TFLOP/s": round(tf, 1), "frac": round(tf / tc_peak, 4),
                          "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4)})
            per_family[f] = e
    dominant = max(per_family, key=lambda f: prof[f][0])
    dom = per_family[dominant]
    if dom["bound"] == "tensor":
        achieved, peak, unit_r = dom["TFLOP/s"], tc_peak, "TFLOP/s"
        peak_src = (f"measured (MEASURED_PEAKS.json {tc_src}, cuBLAS bf16 GEMM)"
                    if pk["source"] == "measured" else "fallback 1.9 PFLOP/s bf16")
    else:
        achieved, peak, unit_r = dom["GB/s"], pk["hbm_gbs"], "GB/s"
        peak_src = ("measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
                    if pk["source"] == "measured" else "fallback 6.8 TB/s")
    flops_total = sum(b.flops_step(W + i) for i in range(K))
    bytes_total = sum(fam_bytes.values())
    if b.is_merge:
        value, unit = 2 * K * world / sec, "merge+unmerge calls/s"
    else:
        value, unit = tokens_all / sec, "tokens/s"
    out = {
        "value": value, "unit": unit, "steps": K, "warmup": W, "ms_per_step": ms / K,
        "us_per_call": {"device": 1e6 * sec / max(1, calls),
                        "host_enqueue": round(host_enqueue_us, 3),
                        "per_kernel_launch": {f: v["us_per_launch"] for f, v in per_family.items()}},
        "roofline": {"bound": dom["bound"], "achieved": achieved, "peak": peak, "unit": unit_r,
                     "frac": achieved / peak if achieved else None,
                     "traffic": dom["traffic"],
                     "peak_source": peak_src,
                     "kernel": KERNEL_NAMES[dominant],
                     "bytes_per_launch": per_family[dominant]["alg_bytes_per_launch"],
                     "us_per_launch": per_family[dominant]["us_per_launch"],
                     "per_family": per_family,
                     # the whole call: every family's algorithmic bytes over the region
                     "path": {"bytes_per_step": bytes_total / K,
                              "GB/s": round(bytes_total / sec / 1e9, 1),
                              "frac_of_hbm": round(bytes_total / sec / 1e9 / pk["hbm_gbs"], 4)},
                     "tflops": flops_total / max(1e-12, sec) / 1e12},
        "gpu_launches": n_launched,
        "clocks": clk,
        "l2_sets": b.n_sets,
    }
    if extras:
        out["us_per_call"].update(per_call_stats(b, K, W, torch, ctx, stream))
        if name == "lorazor_decode":
            out["n_act_curve"] = lorazor_curve(b, torch, stream)
    out["e2e"] = end_to_end(b, K, world, torch, stream)
    if cpu_budget > 0 and world == 1 and not args.no_cpu:
        nthreads = args.cpu_threads or os.cpu_count() or 1
        done, dt, desc = oracle_sample(name, cpu_budget, nthreads)
        out["cpu_baseline"] = {"value": done / dt * (2 if b.is_merge else 1), "unit": unit,
                               "cores": nthreads, "kind": "oracle",
                               "sample": desc + f", {dt:.1f} s"}
    b.release()
    return out


def per_call_stats(b, K, W, torch, ctx, stream) -> dict:
    """Median over five repeats of the K-step region (device µs per call), and per
    call of a step: its device time alone after an L2 flush (CUDA events, median of
    20) and its host time (call plus a stream synchronize, inputs already on the
    device, plan and its upload included; median of 20)."""
    reps = []
    for _ in range(5):
        e0, e1 = _events(torch)
        e0.record(stream)
        for i in range(K):
            b.step(W + i, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        reps.append(1e3 * e0.elapsed_time(e1) / (K * b.calls_per_step()))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    single, host = {}, {}
    for key in b.call_keys():
        dev_us, host_us = [], []
        for r in range(20):
            flush.zero_()
            e0, e1 = _events(torch)
            e0.record(stream)
            b.one_call(r, key, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            dev_us.append(1e3 * e0.elapsed_time(e1))
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            b.one_call(r, key, stream)
            stream.synchronize()
            host_us.append(1e6 * (time.perf_counter() - t0))
        single[key] = round(statistics.median(dev_us), 3)
        host[key] = round(statistics.median(host_us), 3)
    del flush
    return {"device_median_of_5_repeats": round(statistics.median(reps), 3),
            "single_call_cold_device": single, "single_call_host": host}


def lorazor_curve(b, torch, stream) -> dict:
    """Device µs of each of the 100 decode steps (20 back-to-back calls of that
    step's ids over the rotating sets, after 3 untimed ones) against its active rows,
    and the least-squares line through them: the time should follow the active rows
    (the grid covers them alone), not the batch size."""
    pts = []
    for t in range(100):
        for r in range(3):
            b.step_on(r, t, stream)
        e0, e1 = _events(torch)
        e0.record(stream)
        for r in range(20):
            b.step_on(3 + r, t, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        n_act = int((np.asarray(b.steps_ids[t][0][1]) >= 0).sum())
        pts.append((n_act, 1e3 * e0.elapsed_time(e1) / 20))
    x = np.array([p[0] for p in pts], np.float64)
    y = np.array([p[1] for p in pts], np.float64)
    slope, icpt = np.polyfit(x, y, 1)
    fit = slope * x + icpt
    r2 = 1.0 - float(np.sum((y - fit) ** 2) / max(1e-30, np.sum((y - y.mean()) ** 2)))
    return {"points_n_act_us": [[int(a), round(float(u), 3)] for a, u in pts],
            "slope_us_per_active_row": float(slope), "intercept_us": float(icpt), "r2": r2,
            "us_at_n_act_128": float(slope * 128 + icpt), "us_at_n_act_29": float(slope * 29 + icpt),
            "batch_rows": 256}


def end_to_end(b, K, world, torch, stream) -> dict:
    b.e2e_setup()
    Ke = min(K, 2000)
    for i in range(3):
        b.e2e_step(i, stream)
    torch.cuda.synchronize()
    e0, e1 = _events(torch)
    e0.record(b.s_in)            # the first thing of the timed region is a copy in
    stream.wait_event(e0)
    b.s_out.wait_event(e0)
    h2d = d2h = 0
    for i in range(Ke):
        h2d, d2h = b.e2e_step(i, stream)
    b.e2e_drain(stream)          # ... and the last is a read back
    e1.record(stream)
    torch.cuda.synchronize()
    es = e0.elapsed_time(e1) / 1e3
    if b.is_merge:
        val, unit = 2 * Ke * world / es, "merge+unmerge calls/s"
    else:
        val, unit = sum(b.tokens_per_step(i) for i in range(Ke)) * world / es, "tokens/s"
    return {"value": val, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": Ke}


def aggregate_ranks(ms: float, tokens: int, dist, device):
    """Replicas only: every rank times its own copy of the workload; the job's time is
    the slowest rank's and its throughput is the sum of all ranks' units over that
    time.  Returns (max ms, total units, world size)."""
    if dist is None or not dist.is_initialized():
        return ms, tokens, 1
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    u = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), int(u.item()), dist.get_world_size()


def default_steps(name):
    return PER_CONFIG_STEPS[name]


def headline_line(name, m, args, world):
    line = {"metric": METRIC, "value": m["value"], "unit": m["unit"], "n_gpus": world,
            "steps": m["steps"], "warmup": m["warmup"], "ms_per_step": m["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": config_for(name, not args.no_early_pages, args.device_ids, not args.no_early_input)}
    for k in ("us_per_call", "roofline", "gpu_launches", "clocks", "e2e", "cpu_baseline",
              "l2_sets", "n_act_curve"):
        if k in m:
            line[k] = m[k]
    return line


def entry(name, m, args):
    e = {"config": config_for(name, not args.no_early_pages, args.device_ids, not args.no_early_input)}
    e.update({k: v for k, v in m.items()})
    return e


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=CONFIGS)
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--no-per-config", action="store_true",
                    help="the headline workload alone (no per_config entries)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for the headline's cpu_baseline")
    ap.add_argument("--cpu-budget-per-config", type=float, default=3.0,
                    help="seconds of oracle time for each per_config cpu_baseline")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads for the oracle (0: every core)")
    ap.add_argument("--no-early-pages", action="store_true",
                    help="keep the adapter-page copies behind the dependency wait")
    ap.add_argument("--no-early-input", action="store_true",
                    help="keep the tensor-core shrink's x loads behind the dependency wait")
    ap.add_argument("--rows-b-over-a", type=int, choices=(-1, 0, 1), default=0,
                    help="LORA_OPT_ROWS_B_OVER_A for the row-gather kernel (0: the library's choice)")
    ap.add_argument("--profile-every", type=int, default=8,
                    help="bracket one kernel launch in N with CUDA events (roofline timing)")
    ap.add_argument("--tiles", default=os.path.join(ROOT, "adapter_sgmv_bgmv_gb300", "tiles.tbl"))
    ap.add_argument("--device-ids", action="store_true",
                    help="decode workloads through lora_fused_device_ids (ids in device memory)")
    ap.add_argument("--probe", choices=PROBES, default=None,
                    help="run one workload's call a few times for a profiler, print nothing")
    args = ap.parse_args()
    if args.probe:
        return run_probe(args.probe)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args)

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import adapter_sgmv_bgmv_gb300 as L
    ctx = L.Context(local, max_rows=1 << 15, max_rank=64)
    if os.path.exists(args.tiles):
        ctx.tiles_load(args.tiles)
    # Every kernel the timed loop launches is this library's, none of which writes
    # the adapter pools or x: the row-gather kernel may copy pages, and the
    # tensor-core shrink load x, before their waits.
    ctx.set_option(L.OPT_EARLY_PAGES, 0 if args.no_early_pages else 1)
    ctx.set_option(L.OPT_EARLY_INPUT, 0 if args.no_early_input else 1)
    ctx.set_option(L.OPT_ROWS_B_OVER_A, args.rows_b_over_a)
    clocks = ClockSampler(torch, local)
    W = max(3, args.warmup)
    if args.all:
        names = [n for n in CONFIGS if not args.device_ids or n in DEVICE_IDS_CONFIGS]
        for name in names:
            K = args.steps if args.steps is not None else default_steps(name)
            m = measure(name, K, W, args, L, torch, ctx, dist, world, local, clocks,
                        args.cpu_budget, extras=True)
            if rank == 0:
                print(json.dumps(headline_line(name, m, args, world)), flush=True)
    else:
        name = args.config
        if args.device_ids and name not in DEVICE_IDS_CONFIGS:
            name = "llama7b_decode"
        K = args.steps if args.steps is not None else default_steps(name)
        m = measure(name, K, W, args, L, torch, ctx, dist, world, local, clocks,
                    args.cpu_budget, extras=True)
        line = headline_line(name, m, args, world)
        if world == 1 and not args.no_per_config:
            per = {}
            others = [n for n in CONFIGS if n != name and
                      (not args.device_ids or n in DEVICE_IDS_CONFIGS)]
            for other in others:
                mo = measure(other, PER_CONFIG_STEPS[other], W, args, L, torch, ctx, None, 1,
                             local, clocks, args.cpu_budget_per_config, extras=True)
                per[other] = entry(other, mo, args)
            line["per_config"] = per
        if rank == 0:
            print(json.dumps(line), flush=True)
    clocks.close()
    ctx.close()
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


PROBES = ("valora", "slora", "llama_het", "llama_hom", "lorazor", "merge_tc", "merge_simt",
          "proj", "page_in", "plan_dev", "device_ids")


def run_probe(name: str) -> int:
    """One workload's library call, a few times, on one set of device buffers (a
    target for a profiler's capture of one kernel: `ncu -k regex:<kernel> -s 1 -c 1
    python bench.py --probe <name>`).  Prints nothing; exits 0 when the calls and the
    status check succeed."""
    import torch
    import adapter_sgmv_bgmv_gb300 as L
    from tests.gpu_util import to_dev, upload_table
    ctx = L.Context(0, max_rows=1 << 15, max_rank=64)
    tiles = os.path.join(ROOT, "adapter_sgmv_bgmv_gb300", "tiles.tbl")
    if os.path.exists(tiles):
        ctx.tiles_load(tiles)
    ctx.set_option(L.OPT_EARLY_PAGES, 1)
    ctx.set_option(L.OPT_EARLY_INPUT, 1)

    def n_sets(step_bytes):
        # copies enough that a pass over them is more than 3 x L2: the call a profiler
        # captures (the second) reads cold HBM, as in the timed loop
        return int(min(16, max(2, math.ceil(3 * L2_BYTES / max(1, step_bytes)))))

    def fused(case, ids):
        sets = [(upload_table(ctx, case), to_dev(case["x"]), to_dev(case["y"]))
                for _ in range(n_sets(alg_bytes_delta(case, ids)))]
        for t, x, y in sets + sets[:1]:
            L.lora_fused(ctx, t, ids, x, y)

    if name in ("valora", "slora"):
        c = workloads.make(f"{name}_prefill", seed=0)
        fused(c, c["ids"])
    elif name in ("llama_het", "llama_hom"):
        c = workloads.make(f"llama7b_decode_{name[6:]}", seed=0)
        fused(c, c["ids"])
    elif name == "lorazor":
        c = workloads.make("lorazor_decode", seed=0)
        fused(c, workloads.lorazor_ids(c, 0))
    elif name in ("merge_tc", "merge_simt"):
        ctx.set_option(L.OPT_MERGE_KERNEL, 0 if name == "merge_tc" else 1)
        c = workloads.make("valora_merge", seed=0)
        sets = [(upload_table(ctx, c), to_dev(c["W"])) for _ in range(n_sets(4 * c["W"].size))]
        for t, W in sets:
            L.lora_merge(ctx, t, c["merge_adapter"], W)
            L.lora_unmerge(ctx, t, c["merge_adapter"], W)
    elif name == "proj":
        c = workloads.make("valora_prefill", seed=0)
        W = to_dev(workloads.make_W(c["d_in"], c["d_out"], seed=0))
        t = upload_table(ctx, c)
        x = to_dev(c["x"])
        y = torch.empty((c["n"], c["d_out"]), dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            L.lora_base_fused(ctx, t, c["ids"], x, W, y)
    elif name == "page_in":
        c = workloads.small(seed=1, n=1, d_in=4096, d_out=4096, n_adapters=32, ranks=[64] * 32,
                            paged=True)
        t = upload_table(ctx, c)
        ha = torch.zeros((64, 4096), dtype=torch.int16).pin_memory()
        hb = torch.zeros((64, 4096), dtype=torch.int16).pin_memory()
        for k in range(8):
            L.lora_page_in(ctx, t, k, ha, hb)
    elif name in ("plan_dev", "device_ids"):
        ctx.set_option(L.OPT_DEVICE_PLAN, 1 if name == "plan_dev" else 0)
        c = workloads.make("lorazor_decode", seed=0)
        ids_h = workloads.lorazor_ids(c, 0)
        ids = torch.from_numpy(np.ascontiguousarray(ids_h, np.int32)).cuda()
        sets = [(upload_table(ctx, c), to_dev(c["x"]), to_dev(c["y"]))
                for _ in range(n_sets(alg_bytes_delta(c, ids_h)))]
        for t, x, y in sets + sets[:1]:
            L.lora_fused_device_ids(ctx, t, ids, x, y)
    torch.cuda.synchronize()
    ctx.sync_status()
    ctx.close()
    return 0


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload, so that the whole run ends within a few minutes."""
    name = args.config
    K = args.steps if args.steps is not None else 20
    W = max(3, args.warmup) if args.warmup is not None else 3
    nthreads = args.cpu_threads or os.cpu_count() or 1
    per_step = max(0.05, min(2.0, 150.0 / max(1, K + W)))
    for _ in range(W):
        oracle_sample(name, per_step / 4, nthreads)
    done = 0.0
    tot = 0.0
    for _ in range(K):
        d, dt, desc = oracle_sample(name, per_step, nthreads)
        done += d
        tot += dt
    is_merge = name == "valora_merge"
    unit = "merge+unmerge calls/s" if is_merge else "tokens/s"
    value = done / tot * (2 if is_merge else 1)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 1,
            "steps": K, "warmup": W, "ms_per_step": 1e3 * tot / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_for(name, not args.no_early_pages, args.device_ids, not args.no_early_input),
            "cpu_baseline": {"value": value, "unit": unit, "cores": nthreads, "kind": "oracle",
                             "sample": f"each step: about {per_step:.2f} s of the oracle on "
                                       f"the workload's rows ({desc.split(',')[0]} in the last)"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
