"""CPU oracle for the heterogeneous multi-LoRA delta -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may import this package.  The library (``adapter_sgmv_bgmv_gb300``)
never does, and this package imports nothing from the library: the two share no
code.  The arithmetic lives in ``oracle.c`` (plain C, double accumulation, one
bf16 round-to-nearest-even per output element); this module only marshals numpy
arrays into it.

Functions and the passages they follow:

* :func:`fused`  -- y_i += s_k (x_i A_k) B_k per row, k = ids[i] >= 0
  (Punica in "BEE-30060 Multi-LoRA serving", Background; S-LoRA page, Batching,
  formula 2).  Pinned by brute force, closed forms and the dense-GEMM reduction.
* :func:`shrink` / :func:`expand` -- the two factors of the same product, v in fp32
  (the split of the delta into x.A and v.B).  Pinned by brute force and by
  shrink-then-expand agreeing with the fused result.
* :func:`merge` -- W +/- s_k A_k B_k in place (VaLoRA blog, section 4.4.1 swift mode
  switch; S-LoRA page, Batching, formula 1).  Pinned by brute force and by
  merged == unmerged inference.
* :func:`base_fused` -- y_i = x_i W + s_k (x_i A_k) B_k rounded once (x_i W alone for a
  released row): the delta fused into the base projection (S-LoRA page, Batching,
  formula 2; VaLoRA blog, C2, unmerged inference; LoRazor page: released rows keep
  the backbone).  x W is a float64 library matmul, the adapter term is oracle_delta
  in double.  Pinned by brute force, W = 0 reducing to :func:`fused`, all rows
  released reducing to the dense product, and merged == unmerged inference.
* :func:`plan` -- active rows and the stable by-adapter grouping (Punica grouping by
  adapter identity; LoRazor page, active-row-aware kernels).  Pinned bit-exactly by
  an independent numpy construction in the tests.
* :func:`bf16_round` -- nearest bf16, ties to even.  Pinned against torch's float32
  conversion and hand-checked bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (plain gcc, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    table = [P, I64, P, I64, P, P, P, P, I]
    lib.oracle_shrink.argtypes = table + [P, I64, P, I64, I, P, I64, I]
    lib.oracle_expand.argtypes = table + [P, I64, P, I64, P, I64, I, I]
    lib.oracle_fused.argtypes = table + [P, I64, P, I64, I, P, I64, I, I]
    lib.oracle_merge.argtypes = table + [I, I, P, I64, I, I, I]
    lib.oracle_delta.argtypes = table + [P, I64, P, I64, I, P, I64, I, I]
    lib.oracle_round_bf16.argtypes = [P, P, I64]
    lib.oracle_plan.argtypes = [P, I64, I, P, P, P, P, P, P]
    lib.oracle_plan.restype = I
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = ctypes.c_double
    for f in (lib.oracle_shrink, lib.oracle_expand, lib.oracle_fused, lib.oracle_merge,
              lib.oracle_delta, lib.oracle_round_bf16):
        f.restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class Table:
    """Host view of an adapter table: pools of bf16 pages (uint16 bit patterns),
    per-adapter rank and scale, and page ids of A's columns and B's rows."""

    def __init__(self, a_pool, b_pool, rank, scale, a_pages, b_pages):
        self.a_pool = _c(a_pool, np.uint16)
        self.b_pool = _c(b_pool, np.uint16)
        self.rank = _c(rank, np.int32)
        self.scale = _c(scale, np.float32)
        self.a_pages = _c(a_pages, np.int32)
        self.b_pages = _c(b_pages, np.int32)
        assert self.a_pool.ndim == 2 and self.b_pool.ndim == 2
        assert self.a_pages.shape == self.b_pages.shape and self.a_pages.ndim == 2
        self.max_rank = int(self.a_pages.shape[1])

    @classmethod
    def from_case(cls, case: dict) -> "Table":
        return cls(case["a_pool"], case["b_pool"], case["rank"], case["scale"],
                   case["a_pages"], case["b_pages"])

    def args(self):
        return (_ptr(self.a_pool), self.a_pool.shape[1], _ptr(self.b_pool),
                self.b_pool.shape[1], _ptr(self.rank), _ptr(self.scale),
                _ptr(self.a_pages), _ptr(self.b_pages), self.max_rank)


def shrink(table: Table, ids, x, nthreads: int = 1) -> np.ndarray:
    """v[i, j] = sum_c x[i, c] A_k[c, j] (fp32 out, NaN where not written)."""
    lib = _load()
    ids = _c(ids, np.int32)
    x = _c(x, np.uint16)
    n, d_in = x.shape
    v = np.full((n, table.max_rank), np.nan, dtype=np.float32)
    lib.oracle_shrink(*table.args(), _ptr(ids), n, _ptr(x), d_in, d_in, _ptr(v),
                      table.max_rank, nthreads)
    return v


def expand(table: Table, ids, v, y_in, nthreads: int = 1) -> np.ndarray:
    """y[i, o] = bf16(y[i, o] + s_k sum_j v[i, j] B_k[j, o]); returns a new array."""
    lib = _load()
    ids = _c(ids, np.int32)
    v = _c(v, np.float32)
    y = np.array(y_in, dtype=np.uint16, copy=True, order="C")
    n, d_out = y.shape
    lib.oracle_expand(*table.args(), _ptr(ids), n, _ptr(v), v.shape[1], _ptr(y),
                      d_out, d_out, nthreads)
    return y


def fused(table: Table, ids, x, y_in, nthreads: int = 1) -> np.ndarray:
    """y_i + s_k (x_i A_k) B_k rounded once to bf16; rows with id -1 copied."""
    lib = _load()
    ids = _c(ids, np.int32)
    x = _c(x, np.uint16)
    y = np.array(y_in, dtype=np.uint16, copy=True, order="C")
    n, d_in = x.shape
    d_out = y.shape[1]
    lib.oracle_fused(*table.args(), _ptr(ids), n, _ptr(x), d_in, d_in, _ptr(y),
                     d_out, d_out, nthreads)
    return y


def fused_rows(table: Table, ids, x, y_in, rows, nthreads: int = 1) -> np.ndarray:
    """The fused result for a subset of rows only (rows are independent)."""
    rows = np.asarray(rows, dtype=np.int64)
    return fused(table, np.asarray(ids)[rows], np.asarray(x)[rows],
                 np.asarray(y_in)[rows], nthreads)


def delta(table: Table, ids, x, d_out: int, nthreads: int = 1) -> np.ndarray:
    """s_k (x_i A_k) B_k per row in double (zeros for released rows), unrounded."""
    lib = _load()
    ids = _c(ids, np.int32)
    x = _c(x, np.uint16)
    n, d_in = x.shape
    out = np.empty((n, d_out), np.float64)
    lib.oracle_delta(*table.args(), _ptr(ids), n, _ptr(x), d_in, d_in, _ptr(out), d_out,
                     d_out, nthreads)
    return out


def round_bf16(v) -> np.ndarray:
    """Nearest bf16 (ties to even) of every element of a float64 array (uint16 bits)."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_round_bf16(_ptr(v), _ptr(out), v.size)
    return out


def base_fused(table: Table, ids, x, W, nthreads: int = 1, rows=None) -> np.ndarray:
    """y_i = bf16(x_i W + s_k (x_i A_k) B_k), y_i = bf16(x_i W) for ids[i] == -1 (the base
    projection with the adapter term, one rounding).  x [n, d_in], W [d_in, d_out] bf16
    bits; rows: optionally a subset of the rows (returns those rows)."""
    x = np.asarray(x, dtype=np.uint16)
    ids = np.asarray(ids, dtype=np.int32)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        x, ids = x[rows], ids[rows]
    W = np.asarray(W, dtype=np.uint16)
    base = bf16_to_f64(x) @ bf16_to_f64(W)          # float64 library matmul
    base += delta(table, ids, x, W.shape[1], nthreads)
    return round_bf16(base)


def merge(table: Table, adapter: int, W, sign: int = +1, nthreads: int = 1,
          rows=None) -> np.ndarray:
    """W + sign * s_k A_k B_k rounded once to bf16 (optionally for a row subset of W,
    given as the row indices of W; returns those rows)."""
    lib = _load()
    W = np.asarray(W, dtype=np.uint16)
    d_out = W.shape[1]
    if rows is None:
        out = np.array(W, copy=True, order="C")
        lib.oracle_merge(*table.args(), int(adapter), int(sign), _ptr(out), d_out,
                         out.shape[0], d_out, nthreads)
        return out
    rows = np.asarray(rows, dtype=np.int64)
    out = np.ascontiguousarray(W[rows])
    # Restricting W to a subset of its rows restricts A_k to the same rows, i.e. each
    # A page to the same positions: a pool whose page p holds a_pool[p, rows].
    sub = Table(np.ascontiguousarray(table.a_pool[:, rows]), table.b_pool, table.rank,
                table.scale, table.a_pages, table.b_pages)
    lib.oracle_merge(*sub.args(), int(adapter), int(sign), _ptr(out), d_out,
                     len(rows), d_out, nthreads)
    return out


def plan(ids, n_adapters: int) -> dict:
    """Active rows, stable by-adapter permutation and segments (int32, bit-exact)."""
    lib = _load()
    ids = _c(ids, np.int32)
    n = ids.shape[0]
    active = np.zeros(max(n, 1), np.int32)
    perm = np.zeros(max(n, 1), np.int32)
    seg_off = np.zeros(n + 1, np.int32)
    seg_ad = np.zeros(max(n, 1), np.int32)
    na = np.zeros(1, np.int64)
    ns = np.zeros(1, np.int64)
    rc = lib.oracle_plan(_ptr(ids), n, int(n_adapters), _ptr(active), _ptr(na),
                         _ptr(perm), _ptr(seg_off), _ptr(seg_ad), _ptr(ns))
    if rc != 0:
        raise ValueError("adapter id out of range")
    na, ns = int(na[0]), int(ns[0])
    return {"active_rows": active[:na].copy(), "perm": perm[:na].copy(),
            "seg_offsets": seg_off[:ns + 1].copy(), "seg_adapter": seg_ad[:ns].copy()}


def bf16_round(v: float) -> int:
    return int(_load().oracle_bf16_round(float(v)))


def bf16_value(h: int) -> float:
    return float(_load().oracle_bf16_value(int(h)))


def bf16_to_f64(a) -> np.ndarray:
    """Exact decode of bf16 bit patterns (uint16) to float64 (bit shift, no math)."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
